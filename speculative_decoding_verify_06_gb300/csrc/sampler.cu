// sampler.cu -- temperature / min-p / top-p sampling distribution of every window position.
//
// "Decode is memory-bound ...", section "Two things the math says to do": the production
// sampler runs at temperature 0.6, top-p 0.95 and min-p 0.05.  The pages fix only the
// constants; this file implements the reading that both filters act on the same
// un-renormalised p = softmax(logits / T) and that the kept set is their intersection:
//   min-p keeps v iff p[v] >= min_p * max p, i.e. e[v] = exp((l[v] - l_max) / T) >= min_p;
//   top-p keeps the shortest prefix of the order (p descending, id ascending) whose mass
//   reaches top_p (the crossing token included).
// Both are prefixes of the same order, so the kept set is described by its last element
// (e_cut, id_cut): v is kept iff e[v] > e_cut or (e[v] == e_cut and v <= id_cut).
//
// One launch per call: a cluster of 16 CTAs per row (8 above 8 rows, or where a cluster of 16
// does not fit), each CTA one slice of the row,
// sharing their partial results through distributed shared memory:
//   1. each CTA's max and argmax (lowest id on ties, NaN skipped); after a cluster barrier
//      every CTA merges the slices' into the row's.  After the lm_head GEMM with its fused
//      epilogue, the CTAs merge the epilogue's per-block maxima and argmaxes instead of
//      scanning the logits (a share of the blocks each), and rank 0 also forms the row's
//      log-normaliser log sum_v exp(l[v] / T) from the blocks' sums;
//   2. e[v] written into the output buffer, mass sums in 2^-36 fixed point (exact integer
//      sums, independent of the split), and the CTA's min-p survivors kept in shared memory;
//   3. rank 0 finds the crossing: if the survivors fit (<= kSortCap) it gathers them from
//      the cluster, bitonic-sorts them and finds the top-p crossing by a prefix scan (one warp
//      in registers for up to 32 survivors, the whole CTA in shared memory above that);
//      otherwise a four-pass radix select over the bit patterns of e (monotone for e >= 0)
//      over the whole row finds the crossing value and a rank scan the crossing id;
//   4. after a cluster barrier every CTA writes probs[v] = kept ? e[v] / S : 0 for its slice,
//      S the kept mass: when the slice's survivors all fit its list, as zeros over the slice
//      and then e / S at the kept survivors (the kept set never reaches below min-p), else by
//      reading e back.
#include <cooperative_groups.h>

#include "svd_common.cuh"

namespace svd {

namespace cg = cooperative_groups;

constexpr int kSmpSlicesFew = 16;                 // CTAs (one cluster) per row, up to 8 rows
constexpr int kSmpSlicesMany = 8;                 // ... above 8 rows (the clusters fit in fewer waves)
constexpr int kSmpFewRows = 8;
constexpr int kSmpThreads = 1024;
constexpr int kSortCap = 2048;                    // survivors sorted in shared memory
constexpr double kFx = 68719476736.0;             // 2^36
constexpr int kSmpBatch = 8;                      // elements a thread loads before using them

__device__ __forceinline__ unsigned long long fx36(float e) {
    return __float2ull_rn(e * 68719476736.0f);  // e in [0, 1]: exact scaling, then rounding
}

// (value, index) max with lowest index on ties; index -1 is "none".
__device__ __forceinline__ void argmax_merge(float &bv, int &bi, float ov, int oi) {
    if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
    }
}

template <int NTHREADS>
__device__ void block_argmax_merge(float &bv, int &bi) {
    __shared__ float sv[NTHREADS / 32];
    __shared__ int si[NTHREADS / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
    if ((threadIdx.x & 31) == 0) {
        sv[threadIdx.x >> 5] = bv;
        si[threadIdx.x >> 5] = bi;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        bv = threadIdx.x < NTHREADS / 32 ? sv[threadIdx.x] : 0.f;
        bi = threadIdx.x < NTHREADS / 32 ? si[threadIdx.x] : -1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
        if (threadIdx.x == 0) {
            sv[0] = bv;
            si[0] = bi;
        }
    }
    __syncthreads();
    bv = sv[0];
    bi = si[0];
    __syncthreads();
}

template <int NTHREADS>
__device__ unsigned long long block_sum_u64(unsigned long long x) {
    __shared__ unsigned long long s[NTHREADS / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = x;
    __syncthreads();
    if (threadIdx.x < 32) {
        x = threadIdx.x < NTHREADS / 32 ? s[threadIdx.x] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (threadIdx.x == 0) s[0] = x;
    }
    __syncthreads();
    x = s[0];
    __syncthreads();
    return x;
}

// Inclusive scan of u64 values over a warp.
__device__ __forceinline__ unsigned long long warp_scan_u64(unsigned long long x) {
    const unsigned lane = threadIdx.x & 31u;
#pragma unroll
    for (unsigned o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// The survivor with the smallest e, the largest id among equals; id -1 is "none".
__device__ __forceinline__ void cmin_merge(float &a, int &ai, float b, int bi) {
    if (bi >= 0 && (ai < 0 || b < a || (b == a && bi > ai))) {
        a = b;
        ai = bi;
    }
}

__device__ __forceinline__ void slice_bounds(int64_t V, int slices, int blk, int64_t *lo, int64_t *hi) {
    const int64_t S = (V + slices - 1) / slices;
    *lo = min(V, S * blk);
    *hi = min(V, *lo + S);
}

// What one CTA of a row's cluster publishes to the others (read through distributed shared
// memory).
struct SmpShared {
    float pmax;              // slice max and argmax
    int pidx;
    unsigned long long z;    // slice mass, 2^-36 fixed point
    unsigned long long zc;   // mass of the slice's min-p survivors
    unsigned cnt;            // survivors of the slice (may exceed the list's capacity)
    float cmin;              // smallest survivor e, largest id among equals
    int cmin_id;
    float e_cut, s_kept;     // rank 0: the row's crossing and kept mass
    int id_cut;
};

// One row per cluster of SL CTAs (grid: SL x rows).
// stats (nullable): the lm_head epilogue's per-block (max, sum of exp2((l - max) * log2e / T),
// argmax bits) for block b of row r at stats[b * rows + r], n_sb blocks; lse (nullable): the
// row's log-normaliser (natural log), written when the sampler is not greedy.
template <int SL>
__global__ void __launch_bounds__(kSmpThreads, 1)
smp_fused_kernel(const float *__restrict__ logits, int64_t V, float T, float top_p, float min_p,
                 int greedy, float *__restrict__ probs, int32_t *__restrict__ argmax_out,
                 const float4 *__restrict__ stats, int n_sb, float *__restrict__ lse) {
    static_assert(SL <= 32, "one warp merges the slices");
    constexpr int kSliceCap = kSortCap / SL;  // survivors kept per CTA
    cg::cluster_group cl = cg::this_cluster();
    const unsigned rank = cl.block_rank();
    const int row = blockIdx.y;
    __shared__ SmpShared sh;
    __shared__ unsigned long long s_list[kSliceCap];
    __shared__ unsigned s_n;
    __shared__ float s_lmax;
    __shared__ int s_am;
    griddep_wait();
    int64_t lo, hi;
    slice_bounds(V, SL, (int)rank, &lo, &hi);
    const float *L = logits + (int64_t)row * V;
    float *P = probs + (int64_t)row * V;

    // ---- 1. max and argmax of the slice, then of the row ------------------------------------
    const int rows = gridDim.y;
    {
        float bv = 0.f;
        int bi = -1;
        if (stats) {
            const int b0 = (int)((int64_t)n_sb * rank / SL), b1 = (int)((int64_t)n_sb * (rank + 1) / SL);
            for (int b = b0 + (int)threadIdx.x; b < b1; b += kSmpThreads) {
                const float4 st = stats[(size_t)b * rows + row];
                argmax_merge(bv, bi, st.x, __float_as_int(st.z));
            }
        } else {
            for (int64_t v0 = lo + threadIdx.x; v0 < hi; v0 += kSmpBatch * kSmpThreads) {
                float f[kSmpBatch];
#pragma unroll
                for (int u = 0; u < kSmpBatch; ++u) {  // the batch's loads first
                    const int64_t v = v0 + (int64_t)u * kSmpThreads;
                    f[u] = v < hi ? L[v] : __int_as_float(0x7fc00000);
                }
#pragma unroll
                for (int u = 0; u < kSmpBatch; ++u)
                    if (f[u] == f[u]) argmax_merge(bv, bi, f[u], (int)(v0 + (int64_t)u * kSmpThreads));
            }
        }
        block_argmax_merge<kSmpThreads>(bv, bi);
        if (threadIdx.x == 0) {
            sh.pmax = bv;
            sh.pidx = bi;
            s_n = 0;
        }
    }
    cl.sync();
    if (threadIdx.x < 32) {
        float bv = 0.f;
        int bi = -1;
        if (threadIdx.x < SL) {
            const SmpShared *r = cl.map_shared_rank(&sh, threadIdx.x);
            bv = r->pmax;
            bi = r->pidx;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
        if (threadIdx.x == 0) {
            s_lmax = bv;
            s_am = bi;
        }
    }
    __syncthreads();
    const float lmax = s_lmax;
    const int am = s_am;
    if (rank == 0 && threadIdx.x == 0 && argmax_out) argmax_out[row] = am;
    if (greedy) {
        for (int64_t v = lo + threadIdx.x; v < hi; v += kSmpThreads) P[v] = (v == am) ? 1.f : 0.f;
        cl.sync();  // the other CTAs have read this one's slice max
        return;
    }

    // ---- 2. e, the fixed-point masses and the slice's min-p survivors -----------------------
    {
        unsigned long long z = 0, zc = 0;
        float cmin = 2.f;
        int cid = -1;
        for (int64_t v0 = lo + threadIdx.x; v0 < hi; v0 += kSmpBatch * kSmpThreads) {
            float lb[kSmpBatch];
#pragma unroll
            for (int ub = 0; ub < kSmpBatch; ++ub) {  // the batch's loads first
                const int64_t vb = v0 + (int64_t)ub * kSmpThreads;
                lb[ub] = vb < hi ? L[vb] : 0.f;
            }
#pragma unroll
            for (int ub = 0; ub < kSmpBatch; ++ub) {
                const int64_t v = v0 + (int64_t)ub * kSmpThreads;
                if (v >= hi) break;
                const float l = lb[ub];
                float e;
                if (l != l) e = 0.f;                       // NaN logits get no mass
                else if (l == lmax) e = 1.f;
                else e = expf((l - lmax) / T);
                P[v] = e;
                const unsigned long long f = fx36(e);
                z += f;
                if (e >= min_p) {
                    zc += f;
                    if (e < cmin || (e == cmin && (int)v > cid)) {
                        cmin = e;
                        cid = (int)v;
                    }
                    const unsigned slot = atomicAdd(&s_n, 1u);
                    if (slot < kSliceCap)
                        s_list[slot] = ((unsigned long long)__float_as_uint(e) << 32) |
                                       (unsigned long long)(0xFFFFFFFFu - (unsigned)v);
                }
            }
        }
        // the CTA's sums and smallest survivor: warp shuffles, then warp 0 over the warps
        __shared__ unsigned long long sz[kSmpThreads / 32], szc[kSmpThreads / 32];
        __shared__ float sv[kSmpThreads / 32];
        __shared__ int si[kSmpThreads / 32];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            z += __shfl_xor_sync(0xffffffffu, z, o);
            zc += __shfl_xor_sync(0xffffffffu, zc, o);
            cmin_merge(cmin, cid, __shfl_xor_sync(0xffffffffu, cmin, o), __shfl_xor_sync(0xffffffffu, cid, o));
        }
        if ((threadIdx.x & 31) == 0) {
            sz[threadIdx.x >> 5] = z;
            szc[threadIdx.x >> 5] = zc;
            sv[threadIdx.x >> 5] = cmin;
            si[threadIdx.x >> 5] = cid;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            static_assert(kSmpThreads / 32 == 32, "warp 0 merges one value per warp");
            z = sz[threadIdx.x];
            zc = szc[threadIdx.x];
            cmin = sv[threadIdx.x];
            cid = si[threadIdx.x];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                z += __shfl_xor_sync(0xffffffffu, z, o);
                zc += __shfl_xor_sync(0xffffffffu, zc, o);
                cmin_merge(cmin, cid, __shfl_xor_sync(0xffffffffu, cmin, o), __shfl_xor_sync(0xffffffffu, cid, o));
            }
            if (threadIdx.x == 0) {
                sh.z = z;
                sh.zc = zc;
                sh.cnt = s_n;
                sh.cmin = cmin;
                sh.cmin_id = cid;
            }
        }
    }
    cl.sync();  // every slice's e (global) and summary (shared) are visible to the cluster

    // ---- 3. rank 0: the crossing (e_cut, id_cut) and the kept mass --------------------------
    if (rank == 0) {
        __shared__ unsigned long long s_key[kSortCap];
        __shared__ unsigned s_off[SL + 1];
        __shared__ unsigned long long s_Z, s_Zc;
        __shared__ float s_cmin;
        __shared__ int s_cid, s_over;
        __shared__ unsigned s_M;
        if (threadIdx.x < 32) {
            const unsigned b = threadIdx.x;
            unsigned long long Z = 0, Zc = 0;
            unsigned c = 0;
            float cmin = 2.f;
            int cid = -1;
            if (b < (unsigned)SL) {
                const SmpShared *r = cl.map_shared_rank(&sh, b);
                Z = r->z;
                Zc = r->zc;
                c = r->cnt;
                if (c > 0) {
                    cmin = r->cmin;
                    cid = r->cmin_id;
                }
            }
            const int over = __any_sync(0xffffffffu, c > (unsigned)kSliceCap);
            // offsets of the slices' kept survivors: an exclusive scan of min(c, kSliceCap)
            const unsigned kept = min(c, (unsigned)kSliceCap);
            unsigned incl = kept;
#pragma unroll
            for (unsigned o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                if (b >= o) incl += y;
            }
            if (b < (unsigned)SL) s_off[b + 1] = incl;
            unsigned M = c;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                Z += __shfl_xor_sync(0xffffffffu, Z, o);
                Zc += __shfl_xor_sync(0xffffffffu, Zc, o);
                M += __shfl_xor_sync(0xffffffffu, M, o);
                cmin_merge(cmin, cid, __shfl_xor_sync(0xffffffffu, cmin, o), __shfl_xor_sync(0xffffffffu, cid, o));
            }
            if (b == 0) {
                s_off[0] = 0;
                s_Z = Z;
                s_Zc = Zc;
                s_M = M;
                s_over = over || (M > (unsigned)kSortCap);
                s_cmin = cmin;
                s_cid = cid;
            }
        }
        __syncthreads();
        const unsigned long long Z = s_Z;
        const double tgt = (double)top_p * (double)Z;
        if (lse) {
            // log sum_v exp(l[v] / T) = lmax / T + log sum_v e[v]: from the epilogue's block sums
            // (each relative to its block's max) when there are any, else from the exact mass
            __shared__ double s_part[kSmpThreads / 32];
            double part = 0.0;
            if (stats) {
                const float k2 = 1.4426950408889634f / T;
                for (int b = threadIdx.x; b < n_sb; b += kSmpThreads) {
                    const float4 st = stats[(size_t)b * rows + row];
                    if (__float_as_int(st.z) >= 0) part += (double)st.y * (double)exp2f((st.x - lmax) * k2);
                }
            } else if (threadIdx.x == 0) {
                part = (double)Z / kFx;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = part;
            __syncthreads();
            if (threadIdx.x < 32) {
                double tot = s_part[threadIdx.x];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
                if (threadIdx.x == 0) lse[row] = (float)((double)lmax / (double)T + log(tot));
            }
        }
        float e_cut;
        int id_cut;
        unsigned long long S;

        if (s_M == 0) {
            // no survivor at all (only possible when every logit is NaN): keep nothing
            e_cut = __int_as_float(0x7f800000);
            id_cut = -1;
            S = 1;
        } else if (top_p >= 1.f) {
            e_cut = s_cmin;
            id_cut = s_cid;
            S = s_Zc;
        } else if (s_M <= 32u) {
            // ---- at most 32 survivors (the usual case): warp 0 gathers them, sorts them with
            // a bitonic network over its lanes (lane i ends with rank i, keys descending), scans
            // their masses and finds the crossing; the keys, sums and decisions are those of the
            // shared-memory path below
            e_cut = 0.f;
            id_cut = -1;
            S = 0;
            if (threadIdx.x < 32) {
                const unsigned M = s_M, i = threadIdx.x;
                unsigned long long key = 0ull;
                if (i < M) {
                    unsigned b = 0;
                    while (i >= s_off[b + 1]) ++b;
                    key = cl.map_shared_rank(s_list, b)[i - s_off[b]];
                }
#pragma unroll
                for (unsigned size = 2; size <= 32; size <<= 1)
#pragma unroll
                    for (unsigned stride = size >> 1; stride > 0; stride >>= 1) {
                        const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, stride);
                        const bool desc = (i & size) == 0, lower = (i & stride) == 0;
                        key = (lower == desc) ? (key > o ? key : o) : (key < o ? key : o);
                    }
                const unsigned long long m = i < M ? fx36(__uint_as_float((unsigned)(key >> 32))) : 0ull;
                const unsigned long long pre = warp_scan_u64(m);
                const unsigned hits = __ballot_sync(0xffffffffu, i < M && (double)pre >= tgt);
                const unsigned rc = hits ? (unsigned)(__ffs(hits) - 1) : M - 1;
                const unsigned long long kc = __shfl_sync(0xffffffffu, key, rc);
                S = __shfl_sync(0xffffffffu, pre, rc);
                e_cut = __uint_as_float((unsigned)(kc >> 32));
                id_cut = (int)(0xFFFFFFFFu - (unsigned)(kc & 0xFFFFFFFFu));
            }
        } else if (!s_over) {
            // ---- fast path: gather the cluster's survivors and sort them ---------------------
            const unsigned M = s_M;
            unsigned Pn = 2;
            while (Pn < M) Pn <<= 1;
            for (unsigned i = threadIdx.x; i < Pn; i += kSmpThreads) {
                unsigned long long key = 0ull;
                if (i < M) {
                    unsigned b = 0;
                    while (i >= s_off[b + 1]) ++b;
                    key = cl.map_shared_rank(s_list, b)[i - s_off[b]];
                }
                s_key[i] = key;
            }
            __syncthreads();
            // bitonic sort, descending
            for (unsigned size = 2; size <= Pn; size <<= 1) {
                for (unsigned stride = size >> 1; stride > 0; stride >>= 1) {
                    for (unsigned i = threadIdx.x; i < Pn / 2; i += kSmpThreads) {
                        const unsigned lo2 = 2 * stride * (i / stride) + (i % stride), hi2 = lo2 + stride;
                        const bool desc = ((lo2 & size) == 0);
                        const unsigned long long a = s_key[lo2], c = s_key[hi2];
                        if ((a < c) == desc) {
                            s_key[lo2] = c;
                            s_key[hi2] = a;
                        }
                    }
                    __syncthreads();
                }
            }
            // prefix sums of the masses in sorted order: each thread a run of ranks
            __shared__ unsigned long long s_run[kSmpThreads];
            __shared__ unsigned s_cross;
            const unsigned per = (M + kSmpThreads - 1) / kSmpThreads;
            const unsigned r0 = threadIdx.x * per, r1 = min(M, r0 + per);
            unsigned long long run = 0;
            for (unsigned r = r0; r < r1; ++r) run += fx36(__uint_as_float((unsigned)(s_key[r] >> 32)));
            if (threadIdx.x == 0) s_cross = 0xFFFFFFFFu;
            // inclusive scan of the runs: each warp's, then warp 0 over the warps' totals
            __shared__ unsigned long long s_wtot[kSmpThreads / 32];
            run = warp_scan_u64(run);
            if ((threadIdx.x & 31) == 31) s_wtot[threadIdx.x >> 5] = run;
            __syncthreads();
            if (threadIdx.x < 32) s_wtot[threadIdx.x] = warp_scan_u64(s_wtot[threadIdx.x]);
            __syncthreads();
            if (threadIdx.x >= 32) run += s_wtot[(threadIdx.x >> 5) - 1];
            s_run[threadIdx.x] = run;
            __syncthreads();
            unsigned long long pre = threadIdx.x ? s_run[threadIdx.x - 1] : 0ull;
            for (unsigned r = r0; r < r1; ++r) {
                pre += fx36(__uint_as_float((unsigned)(s_key[r] >> 32)));
                if ((double)pre >= tgt) {
                    atomicMin(&s_cross, r);
                    break;
                }
            }
            __syncthreads();
            const unsigned rc = s_cross == 0xFFFFFFFFu ? M - 1 : s_cross;
            const unsigned long long key = s_key[rc];
            e_cut = __uint_as_float((unsigned)(key >> 32));
            id_cut = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFu));
            // kept mass = prefix through rank rc, from the thread whose run holds rc
            __shared__ unsigned long long s_S;
            if (r0 <= rc && rc < r1) {
                unsigned long long pk = threadIdx.x ? s_run[threadIdx.x - 1] : 0ull;
                for (unsigned r = r0; r <= rc; ++r) pk += fx36(__uint_as_float((unsigned)(s_key[r] >> 32)));
                s_S = pk;
            }
            __syncthreads();
            S = s_S;
        } else {
            // ---- general path: radix select on the bit patterns of e over the whole row -----
            __shared__ unsigned h_cnt[256];
            __shared__ unsigned long long h_mass[256];
            __shared__ unsigned s_prefix, s_mask, s_ties;
            __shared__ unsigned long long s_above;
            if (threadIdx.x == 0) {
                s_prefix = 0;
                s_mask = 0;
                s_above = 0;
            }
            __syncthreads();
            for (int pass = 0; pass < 4; ++pass) {
                const int shift = 24 - 8 * pass;
                for (int i = threadIdx.x; i < 256; i += kSmpThreads) {
                    h_cnt[i] = 0;
                    h_mass[i] = 0;
                }
                __syncthreads();
                const unsigned pre = s_prefix, msk = s_mask;
                for (int64_t v = threadIdx.x; v < V; v += kSmpThreads) {
                    const float e = P[v];
                    const unsigned bits = __float_as_uint(e);
                    if ((bits & msk) == pre) {
                        const unsigned d = (bits >> shift) & 255u;
                        atomicAdd(&h_cnt[d], 1u);
                        atomicAdd(&h_mass[d], fx36(e));
                    }
                }
                __syncthreads();
                if (threadIdx.x == 0) {
                    unsigned long long above = s_above;
                    int chosen = -1, lastnz = -1;
                    for (int d = 255; d >= 0; --d) {
                        if (h_cnt[d] == 0) continue;
                        lastnz = d;
                        if ((double)(above + h_mass[d]) >= tgt) {
                            chosen = d;
                            break;
                        }
                        above += h_mass[d];
                    }
                    if (chosen < 0) {  // the target exceeds the mass (top_p rounding): keep all
                        chosen = lastnz < 0 ? 0 : lastnz;
                        above -= h_mass[chosen];
                    }
                    s_above = above;
                    s_prefix = pre | ((unsigned)chosen << shift);
                    s_mask = msk | (255u << shift);
                    s_ties = h_cnt[chosen];
                }
                __syncthreads();
            }
            const unsigned tbits = s_prefix;
            const float t = __uint_as_float(tbits);
            const unsigned long long tfx = fx36(t), above = s_above;
            unsigned n = s_ties;
            if (tfx > 0) {
                const double need = ceil((tgt - (double)above) / (double)tfx);
                if (need >= 1.0 && need < (double)n) n = (unsigned)need;
                if (need < 1.0) n = 1;
            }
            // id of the n-th smallest index with e == t
            __shared__ unsigned s_base;
            __shared__ int s_id;
            __shared__ unsigned s_wcnt[kSmpThreads / 32];
            if (threadIdx.x == 0) {
                s_base = 0;
                s_id = -1;
            }
            __syncthreads();
            for (int64_t t0 = 0; t0 < V; t0 += kSmpThreads) {
                const int64_t v = t0 + threadIdx.x;
                const bool tie = v < V && __float_as_uint(P[v]) == tbits;
                const unsigned bal = __ballot_sync(0xffffffffu, tie);
                if ((threadIdx.x & 31) == 0) s_wcnt[threadIdx.x >> 5] = __popc(bal);
                __syncthreads();
                unsigned before = s_base;
                for (int i = 0; i < (int)(threadIdx.x >> 5); ++i) before += s_wcnt[i];
                before += __popc(bal & ((1u << (threadIdx.x & 31)) - 1u));
                if (tie && before + 1 == n) s_id = (int)v;
                __syncthreads();
                if (threadIdx.x == 0) {
                    unsigned tot = 0;
                    for (int i = 0; i < kSmpThreads / 32; ++i) tot += s_wcnt[i];
                    s_base += tot;
                }
                __syncthreads();
                if (s_id >= 0) break;
            }
            if (t >= min_p) {
                e_cut = t;
                id_cut = s_id;
                S = above + (unsigned long long)n * tfx;
            } else {  // the top-p prefix runs past the min-p survivors: keep the survivors
                e_cut = s_cmin;
                id_cut = s_cid;
                S = s_Zc;
            }
        }
        if (threadIdx.x == 0) {
            sh.e_cut = e_cut;
            sh.id_cut = id_cut;
            sh.s_kept = (float)((double)S / kFx);
        }
    }
    cl.sync();

    // ---- 4. the renormalised distribution of the slice --------------------------------------
    __shared__ float s_ec, s_S;
    __shared__ int s_ic;
    if (threadIdx.x == 0) {
        const SmpShared *r0 = cl.map_shared_rank(&sh, 0u);
        s_ec = r0->e_cut;
        s_S = r0->s_kept;
        s_ic = r0->id_cut;
    }
    __syncthreads();
    const float ec = s_ec, S = s_S;
    const int ic = s_ic;
    const unsigned n_list = s_n;
    if (n_list <= (unsigned)kSliceCap) {
        // the kept set lies inside the min-p survivors (the crossing is never below min_p), and
        // this slice's are all in its list: zeros over the slice, then the kept survivors
        for (int64_t v = lo + threadIdx.x; v < hi; v += kSmpThreads) P[v] = 0.f;
        __syncthreads();
        for (unsigned i = threadIdx.x; i < n_list; i += kSmpThreads) {
            const unsigned long long key = s_list[i];
            const float e = __uint_as_float((unsigned)(key >> 32));
            const int v = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFu));
            if ((e > ec) || (e == ec && v <= ic)) P[v] = e / S;
        }
    } else {
        for (int64_t v0 = lo + threadIdx.x; v0 < hi; v0 += kSmpBatch * kSmpThreads) {
            float eb[kSmpBatch];
#pragma unroll
            for (int u = 0; u < kSmpBatch; ++u) {  // the batch's loads first
                const int64_t v = v0 + (int64_t)u * kSmpThreads;
                eb[u] = v < hi ? P[v] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kSmpBatch; ++u) {
                const int64_t v = v0 + (int64_t)u * kSmpThreads;
                if (v >= hi) break;
                const bool kept = (eb[u] > ec) || (eb[u] == ec && v <= ic);
                P[v] = kept ? eb[u] / S : 0.f;
            }
        }
    }
    cl.sync();  // rank 0 keeps its shared memory until every CTA has read the crossing
}

size_t sampler_ws_bytes(int rows, int64_t V) {
    (void)V;
    return (size_t)rows * 256;  // reserved: the fused kernel keeps its scratch in shared memory
}

int sampler_probs(const float *logits, int rows, int64_t V, const svd_sampler *s, float *probs,
                  int32_t *argmax, void *ws, size_t ws_bytes, cudaStream_t stream,
                  const float4 *stats, int n_sb, float *lse) {
    if (!logits || !probs || !s || rows < 1 || rows > SVD_C_MAX || V < 1 || V > (1LL << 24))
        return SVD_ERR_INVALID_ARG;
    if (logits == probs) return SVD_ERR_INVALID_ARG;
    if (!s->greedy && !(s->temperature > 0.f && s->top_p > 0.f && s->top_p <= 1.f &&
                        s->min_p >= 0.f && s->min_p < 1.f))
        return SVD_ERR_INVALID_ARG;
    if (!ws || ws_bytes < sampler_ws_bytes(rows, V)) return SVD_ERR_WORKSPACE;
    // 16 CTAs per row where the rows' clusters of 16 can all be resident at once on this GPU (the
    // count is asked once), else 8
    static int few_max = -1;
    if (few_max < 0) {
        int ok = 0;
        if (cudaFuncSetAttribute(smp_fused_kernel<kSmpSlicesFew>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
            cudaLaunchConfig_t qc = {};
            qc.gridDim = dim3(kSmpSlicesFew, 1);
            qc.blockDim = dim3(kSmpThreads);
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = kSmpSlicesFew;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            qc.attrs = qa;
            qc.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, smp_fused_kernel<kSmpSlicesFew>, &qc) == cudaSuccess)
                ok = n;
        }
        (void)cudaGetLastError();
        few_max = ok;
    }
    const bool few = rows <= kSmpFewRows && rows <= few_max;
    const int slices = few ? kSmpSlicesFew : kSmpSlicesMany;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(slices, rows);
    cfg.blockDim = dim3(kSmpThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = slices;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (few)
        SVD_CUDA_TRY(cudaLaunchKernelEx(&cfg, smp_fused_kernel<kSmpSlicesFew>, logits, V, s->temperature,
                                        s->top_p, s->min_p, s->greedy ? 1 : 0, probs, argmax, stats, n_sb, lse));
    else
        SVD_CUDA_TRY(cudaLaunchKernelEx(&cfg, smp_fused_kernel<kSmpSlicesMany>, logits, V, s->temperature,
                                        s->top_p, s->min_p, s->greedy ? 1 : 0, probs, argmax, stats, n_sb, lse));
    return SVD_OK;
}

}  // namespace svd
