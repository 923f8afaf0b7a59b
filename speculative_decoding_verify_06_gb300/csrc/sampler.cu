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
// Four launches per call, all over rows x 32 slices except the selection:
//   S0 row max and argmax (lowest id on ties, NaN skipped);
//   S1 e[v] written into the output buffer, mass sums in 2^-36 fixed point (exact integer
//      sums, independent of the split), and the min-p survivors compacted per slice;
//   S2 one CTA per row: if the survivors fit (<= 4096) they are bitonic-sorted in shared
//      memory and the top-p crossing is found by a prefix scan; otherwise a four-pass radix
//      select over the bit patterns of e (monotone for e >= 0) finds the crossing value and
//      a rank scan the crossing id;
//   S3 probs[v] = kept ? e[v] / S : 0 with S the kept mass.
#include "svd_common.cuh"

namespace svd {

constexpr int kSmpSlices = 32;      // CTAs per row in S0, S1, S3
constexpr int kSmpThreads = 256;
constexpr int kSelThreads = 1024;   // S2
constexpr int kSliceCap = 256;      // survivors kept per slice
constexpr int kSortCap = 4096;      // survivors sorted in shared memory
constexpr double kFx = 68719476736.0;  // 2^36

struct SmpWs {
    float *pmax;
    int *pidx;
    unsigned long long *z, *zc;
    unsigned *cnt;
    float *cmin;
    int *cmin_id;
    unsigned long long *cand;  // (e bits << 32) | (0xFFFFFFFF - id)
    float *e_cut, *s_kept;
    int *id_cut, *am;
};

static size_t smp_ws_bytes_rows(int rows) {
    const size_t R = (size_t)rows * kSmpSlices;
    size_t b = 0;
    b += align_up(R * 4, 256) * 2;              // pmax, pidx
    b += align_up(R * 8, 256) * 2;              // z, zc
    b += align_up(R * 4, 256) * 3;              // cnt, cmin, cmin_id
    b += align_up(R * kSliceCap * 8, 256);      // cand
    b += align_up((size_t)rows * 4, 256) * 4;   // e_cut, s_kept, id_cut, am
    return b;
}

static SmpWs smp_ws_carve(void *ws, int rows) {
    const size_t R = (size_t)rows * kSmpSlices;
    uint8_t *p = reinterpret_cast<uint8_t *>(ws);
    SmpWs w;
    auto take = [&](size_t bytes) {
        uint8_t *q = p;
        p += align_up(bytes, 256);
        return q;
    };
    w.pmax = reinterpret_cast<float *>(take(R * 4));
    w.pidx = reinterpret_cast<int *>(take(R * 4));
    w.z = reinterpret_cast<unsigned long long *>(take(R * 8));
    w.zc = reinterpret_cast<unsigned long long *>(take(R * 8));
    w.cnt = reinterpret_cast<unsigned *>(take(R * 4));
    w.cmin = reinterpret_cast<float *>(take(R * 4));
    w.cmin_id = reinterpret_cast<int *>(take(R * 4));
    w.cand = reinterpret_cast<unsigned long long *>(take(R * kSliceCap * 8));
    w.e_cut = reinterpret_cast<float *>(take((size_t)rows * 4));
    w.s_kept = reinterpret_cast<float *>(take((size_t)rows * 4));
    w.id_cut = reinterpret_cast<int *>(take((size_t)rows * 4));
    w.am = reinterpret_cast<int *>(take((size_t)rows * 4));
    return w;
}

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

__device__ __forceinline__ void slice_bounds(int64_t V, int blk, int64_t *lo, int64_t *hi) {
    const int64_t S = (V + kSmpSlices - 1) / kSmpSlices;
    *lo = min(V, S * blk);
    *hi = min(V, *lo + S);
}

// S0: max and argmax per (row, slice).
__global__ void __launch_bounds__(kSmpThreads)
smp_rowmax_kernel(const float *__restrict__ logits, int64_t V, float *__restrict__ pmax,
                  int *__restrict__ pidx) {
    griddep_wait();
    const int row = blockIdx.y, blk = blockIdx.x;
    int64_t lo, hi;
    slice_bounds(V, blk, &lo, &hi);
    const float *L = logits + (int64_t)row * V;
    float bv = 0.f;
    int bi = -1;
    for (int64_t v = lo + threadIdx.x; v < hi; v += kSmpThreads) {
        const float f = L[v];
        if (f == f) argmax_merge(bv, bi, f, (int)v);
    }
    block_argmax_merge<kSmpThreads>(bv, bi);
    if (threadIdx.x == 0) {
        pmax[row * kSmpSlices + blk] = bv;
        pidx[row * kSmpSlices + blk] = bi;
    }
}

__device__ void row_argmax(const float *pmax, const int *pidx, int row, float *lmax, int *am) {
    __shared__ float s_l;
    __shared__ int s_a;
    if (threadIdx.x < 32) {
        float bv = pmax[row * kSmpSlices + threadIdx.x];
        int bi = pidx[row * kSmpSlices + threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
        if (threadIdx.x == 0) {
            s_l = bv;
            s_a = bi;
        }
    }
    __syncthreads();
    *lmax = s_l;
    *am = s_a;
    __syncthreads();
}

// S1: e[v] = exp((l[v] - l_max) / T) into `e_out`, fixed-point mass of the slice and of its
// min-p survivors, and the survivors themselves.
__global__ void __launch_bounds__(kSmpThreads)
smp_exp_kernel(const float *__restrict__ logits, int64_t V, float T, float min_p, int greedy,
               SmpWs w, float *__restrict__ e_out) {
    static_assert(kSmpSlices == 32, "row_argmax reduces one warp of slices");
    griddep_wait();
    const int row = blockIdx.y, blk = blockIdx.x;
    float lmax;
    int am;
    row_argmax(w.pmax, w.pidx, row, &lmax, &am);
    if (blk == 0 && threadIdx.x == 0) w.am[row] = am;
    if (greedy) return;
    __shared__ unsigned s_n;
    __shared__ unsigned long long s_list[kSliceCap];
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    int64_t lo, hi;
    slice_bounds(V, blk, &lo, &hi);
    const float *L = logits + (int64_t)row * V;
    float *E = e_out + (int64_t)row * V;
    unsigned long long z = 0, zc = 0;
    float cmin = 2.f;
    int cid = -1;
    for (int64_t v = lo + threadIdx.x; v < hi; v += kSmpThreads) {
        const float l = L[v];
        float e;
        if (l != l) e = 0.f;                       // NaN logits get no mass
        else if (l == lmax) e = 1.f;
        else e = expf((l - lmax) / T);
        E[v] = e;
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
    z = block_sum_u64<kSmpThreads>(z);
    zc = block_sum_u64<kSmpThreads>(zc);
    // smallest survivor e, largest id among equals ("last element of the min-p prefix")
    {
        __shared__ float sv[kSmpThreads / 32];
        __shared__ int si[kSmpThreads / 32];
        auto merge = [](float &a, int &ai, float b, int bi) {
            if (bi >= 0 && (ai < 0 || b < a || (b == a && bi > ai))) {
                a = b;
                ai = bi;
            }
        };
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            merge(cmin, cid, __shfl_xor_sync(0xffffffffu, cmin, o), __shfl_xor_sync(0xffffffffu, cid, o));
        if ((threadIdx.x & 31) == 0) {
            sv[threadIdx.x >> 5] = cmin;
            si[threadIdx.x >> 5] = cid;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int i = 1; i < kSmpThreads / 32; ++i) merge(cmin, cid, sv[i], si[i]);
            const int o = row * kSmpSlices + blk;
            w.z[o] = z;
            w.zc[o] = zc;
            w.cnt[o] = s_n;
            w.cmin[o] = cmin;
            w.cmin_id[o] = cid;
        }
    }
    const unsigned n = min(s_n, (unsigned)kSliceCap);
    unsigned long long *dst = w.cand + ((size_t)row * kSmpSlices + blk) * kSliceCap;
    for (unsigned i = threadIdx.x; i < n; i += kSmpThreads) dst[i] = s_list[i];
}

// S2: the crossing (e_cut, id_cut) and the kept mass of one row.
__global__ void __launch_bounds__(kSelThreads)
smp_select_kernel(int64_t V, float top_p, float min_p, int greedy, SmpWs w,
                  const float *__restrict__ e_all, int32_t *__restrict__ argmax_out) {
    griddep_wait();
    const int row = blockIdx.x;
    if (threadIdx.x == 0 && argmax_out) argmax_out[row] = w.am[row];
    if (greedy) return;

    __shared__ unsigned long long s_key[kSortCap];
    __shared__ unsigned s_off[kSmpSlices + 1];
    __shared__ unsigned long long s_Z, s_Zc;
    __shared__ float s_cmin;
    __shared__ int s_cid, s_over;
    __shared__ unsigned s_M;
    if (threadIdx.x == 0) {
        unsigned long long Z = 0, Zc = 0;
        unsigned M = 0;
        int over = 0;
        float cmin = 2.f;
        int cid = -1;
        s_off[0] = 0;
        for (int b = 0; b < kSmpSlices; ++b) {
            const int o = row * kSmpSlices + b;
            Z += w.z[o];
            Zc += w.zc[o];
            const unsigned c = w.cnt[o];
            if (c > (unsigned)kSliceCap) over = 1;
            M += c;
            s_off[b + 1] = s_off[b] + min(c, (unsigned)kSliceCap);
            if (c > 0) {
                const float cm = w.cmin[o];
                const int ci = w.cmin_id[o];
                if (cid < 0 || cm < cmin || (cm == cmin && ci > cid)) {
                    cmin = cm;
                    cid = ci;
                }
            }
        }
        s_Z = Z;
        s_Zc = Zc;
        s_M = M;
        s_over = over || (M > (unsigned)kSortCap);
        s_cmin = cmin;
        s_cid = cid;
    }
    __syncthreads();
    const unsigned long long Z = s_Z;
    const double tgt = (double)top_p * (double)Z;
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
    } else if (!s_over) {
        // ---- fast path: sort the survivors --------------------------------------------------
        const unsigned M = s_M;
        unsigned P = 2;
        while (P < M) P <<= 1;
        for (unsigned i = threadIdx.x; i < P; i += kSelThreads) {
            unsigned long long key = 0ull;
            if (i < M) {
                int b = 0;
                while (i >= s_off[b + 1]) ++b;
                key = w.cand[((size_t)row * kSmpSlices + b) * kSliceCap + (i - s_off[b])];
            }
            s_key[i] = key;
        }
        __syncthreads();
        // bitonic sort, descending
        for (unsigned size = 2; size <= P; size <<= 1) {
            for (unsigned stride = size >> 1; stride > 0; stride >>= 1) {
                for (unsigned i = threadIdx.x; i < P / 2; i += kSelThreads) {
                    const unsigned lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
                    const bool desc = ((lo & size) == 0);
                    const unsigned long long a = s_key[lo], b = s_key[hi];
                    if ((a < b) == desc) {
                        s_key[lo] = b;
                        s_key[hi] = a;
                    }
                }
                __syncthreads();
            }
        }
        // prefix sums of the masses in sorted order: each thread a run of ranks
        __shared__ unsigned long long s_run[kSelThreads];
        __shared__ unsigned s_cross;
        const unsigned per = (M + kSelThreads - 1) / kSelThreads;
        const unsigned r0 = threadIdx.x * per, r1 = min(M, r0 + per);
        unsigned long long run = 0;
        for (unsigned r = r0; r < r1; ++r) run += fx36(__uint_as_float((unsigned)(s_key[r] >> 32)));
        s_run[threadIdx.x] = run;
        if (threadIdx.x == 0) s_cross = 0xFFFFFFFFu;
        __syncthreads();
        // inclusive scan of s_run (Hillis-Steele over 1024 entries)
        for (unsigned off = 1; off < kSelThreads; off <<= 1) {
            const unsigned long long add = threadIdx.x >= off ? s_run[threadIdx.x - off] : 0ull;
            __syncthreads();
            s_run[threadIdx.x] += add;
            __syncthreads();
        }
        unsigned long long pre = threadIdx.x ? s_run[threadIdx.x - 1] : 0ull;
        for (unsigned r = r0; r < r1; ++r) {
            pre += fx36(__uint_as_float((unsigned)(s_key[r] >> 32)));
            if ((double)pre >= tgt) {
                atomicMin(&s_cross, r);
                break;
            }
        }
        __syncthreads();
        unsigned rc = s_cross == 0xFFFFFFFFu ? M - 1 : s_cross;
        const unsigned long long key = s_key[rc];
        e_cut = __uint_as_float((unsigned)(key >> 32));
        id_cut = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFu));
        // kept mass = prefix through rank rc
        __shared__ unsigned long long s_S;
        if (threadIdx.x == 0) s_S = 0;
        __syncthreads();
        unsigned long long part = 0;
        for (unsigned r = threadIdx.x; r <= rc; r += kSelThreads)
            part += fx36(__uint_as_float((unsigned)(s_key[r] >> 32)));
        atomicAdd(&s_S, part);
        __syncthreads();
        S = s_S;
    } else {
        // ---- general path: radix select on the bit patterns of e ----------------------------
        const float *E = e_all + (int64_t)row * V;
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
            for (int i = threadIdx.x; i < 256; i += kSelThreads) {
                h_cnt[i] = 0;
                h_mass[i] = 0;
            }
            __syncthreads();
            const unsigned pre = s_prefix, msk = s_mask;
            for (int64_t v = threadIdx.x; v < V; v += kSelThreads) {
                const float e = E[v];
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
        __shared__ unsigned s_wcnt[kSelThreads / 32];
        if (threadIdx.x == 0) {
            s_base = 0;
            s_id = -1;
        }
        __syncthreads();
        for (int64_t t0 = 0; t0 < V; t0 += kSelThreads) {
            const int64_t v = t0 + threadIdx.x;
            const bool tie = v < V && __float_as_uint(E[v]) == tbits;
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
                for (int i = 0; i < kSelThreads / 32; ++i) tot += s_wcnt[i];
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
        w.e_cut[row] = e_cut;
        w.id_cut[row] = id_cut;
        w.s_kept[row] = (float)((double)S / kFx);
    }
}

// S3: the renormalised distribution.
__global__ void __launch_bounds__(kSmpThreads)
smp_write_kernel(int64_t V, int greedy, SmpWs w, float *__restrict__ probs) {
    griddep_wait();
    const int row = blockIdx.y, blk = blockIdx.x;
    int64_t lo, hi;
    slice_bounds(V, blk, &lo, &hi);
    float *P = probs + (int64_t)row * V;
    if (greedy) {
        const int am = w.am[row];
        for (int64_t v = lo + threadIdx.x; v < hi; v += kSmpThreads) P[v] = (v == am) ? 1.f : 0.f;
        return;
    }
    const float ec = w.e_cut[row], S = w.s_kept[row];
    const int ic = w.id_cut[row];
    for (int64_t v = lo + threadIdx.x; v < hi; v += kSmpThreads) {
        const float e = P[v];
        const bool kept = (e > ec) || (e == ec && v <= ic);
        P[v] = kept ? e / S : 0.f;
    }
}

size_t sampler_ws_bytes(int rows, int64_t V) {
    (void)V;
    return smp_ws_bytes_rows(rows);
}

int sampler_probs(const float *logits, int rows, int64_t V, const svd_sampler *s, float *probs,
                  int32_t *argmax, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!logits || !probs || !s || rows < 1 || rows > SVD_C_MAX || V < 1 || V > (1LL << 24))
        return SVD_ERR_INVALID_ARG;
    if (logits == probs) return SVD_ERR_INVALID_ARG;
    if (!s->greedy && !(s->temperature > 0.f && s->top_p > 0.f && s->top_p <= 1.f &&
                        s->min_p >= 0.f && s->min_p < 1.f))
        return SVD_ERR_INVALID_ARG;
    if (!ws || ws_bytes < smp_ws_bytes_rows(rows)) return SVD_ERR_WORKSPACE;
    SmpWs w = smp_ws_carve(ws, rows);
    const int greedy = s->greedy ? 1 : 0;
    const dim3 grid(kSmpSlices, rows);
    SVD_CUDA_TRY(launch(smp_rowmax_kernel, grid, dim3(kSmpThreads), 0, stream, false, logits, V,
                        w.pmax, w.pidx));
    SVD_CUDA_TRY(launch(smp_exp_kernel, grid, dim3(kSmpThreads), 0, stream, false, logits, V,
                        s->temperature, s->min_p, greedy, w, probs));
    SVD_CUDA_TRY(launch(smp_select_kernel, dim3(rows), dim3(kSelThreads), 0, stream, false, V,
                        s->top_p, s->min_p, greedy, w, (const float *)probs, argmax));
    SVD_CUDA_TRY(launch(smp_write_kernel, grid, dim3(kSmpThreads), 0, stream, false, V, greedy, w,
                        probs));
    return SVD_OK;
}

}  // namespace svd
