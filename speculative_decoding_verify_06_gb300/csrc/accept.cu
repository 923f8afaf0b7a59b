// accept.cu -- the lossless acceptance rule of speculative decoding, one CTA per verify window.
//
// "100 tokens per second from a 27B model on a 24 GB AMD card", section "How speculative
// decoding gets past a per-token wall", and "Decode is memory-bound ...", section
// "Speculative decoding": a drafter proposes x_1..x_k, the target scores them in one pass, a
// token-by-token rule keeps a prefix and the target's own next token caps the window.
//  * greedy: accept x_i while it equals the target's argmax (the HN thread's "D E F" example);
//  * sampled (Leviathan et al. 2023, Chen et al. 2023): accept x_i with probability
//    min(1, p(x_i)/q(x_i)); at the first rejection resample from the normalised (p - q)+; if
//    every draft is accepted, draw the capping token from p_{k+1}.
//
// The accept test u*q < p is taken in double precision, where the product of a 24-bit uniform
// and an fp32 probability is exact, so it never depends on rounding.  The draw over the
// vocabulary uses weights rounded to 2^-62 fixed point and 128-bit integer sums: the running
// sum is exactly associative, so the token chosen does not depend on how the sum is split
// over threads.  The search for the crossing is hierarchical: the CTA sums eight slices,
// keeps the slice that contains u' * R, and repeats on it until 32 elements are left; only the
// first level streams the whole row from HBM, the deeper levels re-read a shrinking slice that
// is still cached.
//
// Two kernels share that logic.  accept_kernel gives every window one CTA of 256 threads, which
// suits many windows at once.  accept_cluster_kernel gives a window a cluster of eight CTAs of
// 1024 threads on eight SMs: the first level of the draw is split over the cluster's 256 warps
// (each warp's slice sum is one dependent 128-bit chain, so the width shortens it), the CTAs
// exchange their slice sums through distributed shared memory, and the CTA whose slice holds the
// crossing finishes the search alone.  The host picks the cluster
// kernel when there are fewer sampled windows than SMs, the case of one verify pass.
#include <cooperative_groups.h>

#include "svd_common.cuh"

namespace svd {

int sm_count();

constexpr int kAccThreads = 256;
constexpr int kAccWarps = kAccThreads / 32;
// The cluster kernel (one window on eight SMs) runs wider CTAs: its first level of the draw is
// one 128-bit sum chain per warp, so more warps shorten it.
constexpr int kAccCThreads = 1024;
constexpr int kAccCWarps = kAccCThreads / 32;
constexpr int kAccMaxWarps = kAccCWarps > kAccWarps ? kAccCWarps : kAccWarps;
typedef unsigned __int128 u128;

// round(f * 2^62) for f in [0, 1] (round half up); NaN, infinities, negatives and values
// above one set SVD_ST_BAD_PROB and are clamped into [0, 1].
__device__ __forceinline__ uint64_t prob_fx(float f, int &st) {
    if (!(f >= 0.f && f <= 1.f)) {
        st |= SVD_ST_BAD_PROB;
        return (f > 1.f) ? (1ull << 62) : 0ull;
    }
    const uint32_t bits = __float_as_uint(f) & 0x7FFFFFFFu;
    const int E = (int)(bits >> 23);
    if (E == 0) return 0ull;  // below 2^-126: under half a unit of 2^-62
    const uint64_t m = (uint64_t)((bits & 0x7FFFFFu) | 0x800000u);
    if (E >= 88) return m << (E - 88);  // value * 2^62 = m * 2^(E - 88)
    const int sh = 88 - E;
    if (sh >= 25) return 0ull;
    return (m + (1ull << (sh - 1))) >> sh;
}

__device__ __forceinline__ double prob_clamped(float f, int &st) {
    if (!(f >= 0.f && f <= 1.f)) {
        st |= SVD_ST_BAD_PROB;
        return (f > 1.f) ? 1.0 : 0.0;
    }
    return (double)f;
}

// A q value's status alone (where p is zero the residual is zero whatever q is).
__device__ __forceinline__ void q_status(float f, int &st) {
    if (!(f >= 0.f && f <= 1.f)) st |= SVD_ST_BAD_PROB;
}

// kSkipZero: rows from the sampler, where all but the kept tokens are zero (the one-window
// cluster kernel); dense rows take the plain path, which the test would only slow down.
template <bool kSkipZero = false>
__device__ __forceinline__ uint64_t weight_fx(const float *rp, const float *rq, int64_t v, int &st) {
    const float fp = __ldg(rp + v);
    if (kSkipZero && fp == 0.f) {  // a filtered-out token: no weight, no conversion
        if (rq) q_status(__ldg(rq + v), st);
        return 0ull;
    }
    const uint64_t a = prob_fx(fp, st);
    if (rq) {
        const uint64_t b = prob_fx(__ldg(rq + v), st);
        return a > b ? a - b : 0ull;
    }
    return a;
}

__device__ __forceinline__ u128 warp_sum_u128(u128 x) {
    uint64_t lo = (uint64_t)x, hi = (uint64_t)(x >> 64);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t olo = __shfl_xor_sync(0xffffffffu, lo, o);
        const uint64_t ohi = __shfl_xor_sync(0xffffffffu, hi, o);
        const uint64_t nlo = lo + olo;
        hi = hi + ohi + (nlo < lo ? 1ull : 0ull);
        lo = nlo;
    }
    return ((u128)hi << 64) | lo;
}

// Sum of the weights of [lo, hi) for this warp's slice; float4 loads when allowed.
template <bool kSkipZero = false>
__device__ u128 slice_sum(const float *rp, const float *rq, int64_t lo, int64_t hi, bool vec,
                          int &st) {
    const int lane = threadIdx.x & 31;
    u128 acc = 0;
    int64_t v = lo;
    if (vec && ((lo & 3) == 0)) {
        const int64_t nvec = (hi - lo) >> 2;
        const float4 *p4 = reinterpret_cast<const float4 *>(rp + lo);
        const float4 *q4 = rq ? reinterpret_cast<const float4 *>(rq + lo) : nullptr;
        int64_t t = lane;
        for (; t + 96 < nvec; t += 128) {
            float4 a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] = __ldg(p4 + t + 32 * u);
            if (q4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) b[u] = __ldg(q4 + t + 32 * u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float av[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
                const float bv[4] = {q4 ? b[u].x : 0.f, q4 ? b[u].y : 0.f, q4 ? b[u].z : 0.f,
                                     q4 ? b[u].w : 0.f};
                if (kSkipZero && av[0] == 0.f && av[1] == 0.f && av[2] == 0.f && av[3] == 0.f) {
                    // four filtered-out tokens: no weight; q still reports a bad value
                    if (q4) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) q_status(bv[e], st);
                    }
                    continue;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint64_t x = prob_fx(av[e], st);
                    uint64_t r = x;
                    if (q4) {
                        const uint64_t y = prob_fx(bv[e], st);
                        r = x > y ? x - y : 0ull;
                    }
                    acc += r;
                }
            }
        }
        for (; t < nvec; t += 32) {
            const float4 a = __ldg(p4 + t);
            const float4 b = q4 ? __ldg(q4 + t) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
            if (kSkipZero && av[0] == 0.f && av[1] == 0.f && av[2] == 0.f && av[3] == 0.f) {
                if (q4) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) q_status(bv[e], st);
                }
                continue;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint64_t x = prob_fx(av[e], st);
                uint64_t r = x;
                if (q4) {
                    const uint64_t y = prob_fx(bv[e], st);
                    r = x > y ? x - y : 0ull;
                }
                acc += r;
            }
        }
        v = lo + (nvec << 2);
    }
    for (int64_t x = v + lane; x < hi; x += 32) acc += weight_fx<kSkipZero>(rp, rq, x, st);
    return warp_sum_u128(acc);
}

struct AcceptShared {
    u128 part[kAccMaxWarps];
    u128 base, target, total;
    int64_t lo, hi;
    int st_or[kAccMaxWarps];
    int j;             // first rejected position (k when all accepted)
    uint32_t m2;       // resampling uniform as a 24-bit integer
    int64_t amax;      // greedy: argmax of the current row
    int found;
};

// CTA-wide argmax of a row (lowest index on ties, NaN skipped; -1 when every value is NaN).
__device__ int64_t block_argmax(const float *row, int64_t V, int &st, AcceptShared &sh) {
    __shared__ float s_val[kAccWarps];
    __shared__ int64_t s_idx[kAccWarps];
    float best = 0.f;
    int64_t bi = -1;
    for (int64_t v = threadIdx.x; v < V; v += kAccThreads) {
        const float f = __ldg(row + v);
        if (f != f) {
            st |= SVD_ST_BAD_PROB;
            continue;
        }
        if (bi < 0 || f > best) {
            best = f;
            bi = v;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int64_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi >= 0 && (bi < 0 || ov > best || (ov == best && oi < bi))) {
            best = ov;
            bi = oi;
        }
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        s_val[warp] = best;
        s_idx[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.f;
        int64_t i = -1;
        for (int w = 0; w < kAccWarps; ++w)
            if (s_idx[w] >= 0 && (i < 0 || s_val[w] > b || (s_val[w] == b && s_idx[w] < i))) {
                b = s_val[w];
                i = s_idx[w];
            }
        sh.amax = i;
    }
    __syncthreads();
    const int64_t r = sh.amax;
    __syncthreads();
    return r;
}

// The accept tests of window w, one lane of the calling warp per drafted position: the first
// rejected position j (k when every draft is accepted) and the resampling uniform of the draw
// that follows go to sh.j and sh.m2, the status bits of positions up to j to sh.st_or[0];
// the accepted drafts are written to tok when write_tok.
__device__ void accept_tests(const float *__restrict__ p, const int64_t *__restrict__ p_rows,
                             const float *__restrict__ q, const int64_t *__restrict__ q_rows,
                             const int32_t *__restrict__ draft, int k, int64_t V, uint64_t seed,
                             uint64_t woff, const float *__restrict__ uniforms, int64_t w,
                             int32_t *tok, AcceptShared &sh, bool write_tok = true) {
    const int lane = threadIdx.x & 31;
    auto prow = [&](int i) -> const float * {
        const int64_t r = p_rows ? p_rows[w * (k + 1) + i] : w * (k + 1) + i;
        return p + r * V;
    };
    auto qrow = [&](int i) -> const float * {
        const int64_t r = q_rows ? q_rows[w * k + i] : w * k + i;
        return q + r * V;
    };
    const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
    const uint64_t widx = woff + (uint64_t)w;
    int st = 0;
    bool acc = false;
    uint32_t m2 = 0;
    if (lane < k) {
        double u;
        if (uniforms) {
            u = (double)uniforms[(w * (k + 1) + lane) * 2];
            const float u2 = uniforms[(w * (k + 1) + lane) * 2 + 1];
            m2 = (uint32_t)fminf(fmaxf(floorf(u2 * 16777216.f), 0.f), 16777215.f);
        } else {
            const Philox4 r = philox4x32_10((uint32_t)widx, (uint32_t)(widx >> 32),
                                            (uint32_t)lane, 0u, key0, key1);
            u = (double)(r.v[0] >> 8) * (1.0 / 16777216.0);
            m2 = r.v[1] >> 8;
        }
        const int32_t x = draft[w * k + lane];
        if (x < 0 || x >= V) {
            st |= SVD_ST_BAD_TOKEN;
        } else {
            const double pv = prob_clamped(__ldg(prow(lane) + x), st);
            const double qv = prob_clamped(__ldg(qrow(lane) + x), st);
            if (qv == 0.0) st |= SVD_ST_Q_ZERO;
            acc = u * qv < pv;
        }
    }
    const uint32_t kmask = (k >= 32) ? 0xffffffffu : ((1u << k) - 1u);
    const uint32_t amask = __ballot_sync(0xffffffffu, acc) & kmask;
    const uint32_t rej = (~amask) & kmask;
    const int j = rej ? (__ffs(rej) - 1) : k;
    const int st_all = __reduce_or_sync(0xffffffffu, lane <= j ? st : 0);
    const uint32_t m2j = __shfl_sync(0xffffffffu, m2, j < 32 ? j : 0);
    if (write_tok && lane < j) tok[lane] = draft[w * k + lane];
    if (lane == 0) {
        sh.j = j;
        sh.st_or[0] = st_all;
        if (j < k) {
            sh.m2 = m2j;
        } else if (uniforms) {
            const float u2 = uniforms[(w * (k + 1) + k) * 2 + 1];
            sh.m2 = (uint32_t)fminf(fmaxf(floorf(u2 * 16777216.f), 0.f), 16777215.f);
        } else {
            const Philox4 r = philox4x32_10((uint32_t)widx, (uint32_t)(widx >> 32),
                                            (uint32_t)k, 0u, key0, key1);
            sh.m2 = r.v[1] >> 8;
        }
    }
}

__global__ void __launch_bounds__(kAccThreads)
accept_kernel(const float *__restrict__ p, const int64_t *__restrict__ p_rows,
              const float *__restrict__ q, const int64_t *__restrict__ q_rows,
              const int32_t *__restrict__ tgt_am, const int32_t *__restrict__ draft, int k,
              int64_t V, uint64_t seed, uint64_t woff, const float *__restrict__ uniforms,
              int32_t *__restrict__ out_tokens, int32_t *__restrict__ n_emitted,
              int32_t *__restrict__ status, int vec_ok) {
    __shared__ AcceptShared sh;
    griddep_wait();
    const int64_t w = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t *tok = out_tokens + w * (k + 1);
    auto prow = [&](int i) -> const float * {
        const int64_t r = p_rows ? p_rows[w * (k + 1) + i] : w * (k + 1) + i;
        return p + r * V;
    };
    auto qrow = [&](int i) -> const float * {
        const int64_t r = q_rows ? q_rows[w * k + i] : w * k + i;
        return q + r * V;
    };
    for (int i = threadIdx.x; i <= k; i += kAccThreads) tok[i] = -1;

    if (q == nullptr) {
        // ---- greedy -----------------------------------------------------------------------
        int st = 0, ne = 0;
        for (int i = 0; i <= k; ++i) {
            int64_t a;
            if (tgt_am) {
                a = tgt_am[w * (k + 1) + i];
            } else {
                a = block_argmax(prow(i), V, st, sh);
            }
            if (a < 0 || a >= V) {
                st |= SVD_ST_EMPTY;
                break;
            }
            const int32_t x = (i < k) ? draft[w * k + i] : -1;
            if (i < k && x == a) {
                if (threadIdx.x == 0) tok[ne] = (int32_t)a;
                ++ne;
                continue;
            }
            if (i < k && (x < 0 || x >= V)) st |= SVD_ST_BAD_TOKEN;
            if (threadIdx.x == 0) tok[ne] = (int32_t)a;
            ++ne;
            break;
        }
        // st differs per thread only through the argmax scans: OR it over the CTA
        st = __reduce_or_sync(0xffffffffu, st);
        if (lane == 0) sh.st_or[warp] = st;
        __syncthreads();
        if (threadIdx.x == 0) {
            int s = 0;
            for (int i = 0; i < kAccWarps; ++i) s |= sh.st_or[i];
            n_emitted[w] = ne;
            status[w] = s;
        }
        return;
    }

    // ---- sampled: the accept tests, one lane per drafted position --------------------------
    if (warp == 0) accept_tests(p, p_rows, q, q_rows, draft, k, V, seed, woff, uniforms, w, tok, sh);
    __syncthreads();
    const int j = sh.j;
    const uint32_t m2 = sh.m2;
    const float *rp = prow(j);
    int st = 0;
    if (threadIdx.x == 0) st = sh.st_or[0];

    // ---- the draw: level 1 streams the whole row and yields the total R ---------------------
    // Each level sums eight slices of [lo, hi) and keeps the one holding the crossing, the
    // smallest v with (sum of weights up to v) * 2^24 > m2 * R; at most 32 elements remain.
    const bool vec = vec_ok != 0;
    const float *rq = (j < k) ? qrow(j) : nullptr;
    int64_t lo = 0, hi = V;
    u128 base = 0, total = 0, target = 0;
    bool known = false;  // total known from level 1
    for (int attempt = 0; attempt < 2; ++attempt) {
        lo = 0;
        hi = V;
        base = 0;
        known = false;
        bool level1 = true;
        while (hi - lo > 32) {
            int64_t part = (hi - lo + kAccWarps - 1) / kAccWarps;
            if (level1 && vec) part = (part + 3) & ~int64_t(3);
            const int64_t a = min(hi, lo + part * warp), bnd = min(hi, a + part);
            const u128 s = (a < bnd) ? slice_sum(rp, rq, a, bnd, vec && level1, st) : (u128)0;
            if (lane == 0) sh.part[warp] = s;
            __syncthreads();
            if (threadIdx.x == 0) {
                if (level1) {
                    u128 R = 0;
                    for (int i = 0; i < kAccWarps; ++i) R += sh.part[i];
                    sh.total = R;
                    sh.target = (u128)m2 * R;
                    sh.base = 0;
                }
                int chosen = -1;
                u128 b = sh.base;
                if (sh.total != 0) {
                    for (int i = 0; i < kAccWarps; ++i) {
                        if (((b + sh.part[i]) << 24) > sh.target) {
                            chosen = i;
                            break;
                        }
                        b += sh.part[i];
                    }
                }
                sh.found = chosen;
                if (chosen >= 0) {
                    sh.base = b;
                    sh.lo = min(hi, lo + part * chosen);
                    sh.hi = min(hi, sh.lo + part);
                }
            }
            __syncthreads();
            total = sh.total;
            target = sh.target;
            known = true;
            if (sh.found < 0) break;  // zero mass (the only way no slice holds the crossing)
            lo = sh.lo;
            hi = sh.hi;
            base = sh.base;
            level1 = false;
        }
        if (known && total == 0 && rq != nullptr) {
            if (threadIdx.x == 0) st |= SVD_ST_ZERO_RESIDUAL;
            rq = nullptr;  // READING: an empty residual falls back to p_j
            __syncthreads();
            continue;
        }
        break;
    }

    // ---- final scan of at most 32 elements by warp 0 ------------------------------------------
    int64_t token = -1;
    if (warp == 0 && !(known && total == 0)) {
        const int64_t v = lo + lane;
        u128 r = (v < hi) ? (u128)weight_fx(rp, rq, v, st) : (u128)0;
        if (!known) {  // V <= 32: this scan is the whole row
            total = warp_sum_u128(r);
            if (total == 0 && rq != nullptr) {
                if (lane == 0) st |= SVD_ST_ZERO_RESIDUAL;
                rq = nullptr;
                r = (v < hi) ? (u128)weight_fx(rp, rq, v, st) : (u128)0;
                total = warp_sum_u128(r);
            }
            target = (u128)m2 * total;
        }
        uint64_t plo = (uint64_t)r, phi = (uint64_t)(r >> 64);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t olo = __shfl_up_sync(0xffffffffu, plo, o);
            const uint64_t ohi = __shfl_up_sync(0xffffffffu, phi, o);
            if (lane >= o) {
                const uint64_t nlo = plo + olo;
                phi = phi + ohi + (nlo < plo ? 1ull : 0ull);
                plo = nlo;
            }
        }
        const u128 incl = ((u128)phi << 64) | plo;
        const bool hit = (v < hi) && (total != 0) && (((base + incl) << 24) > target);
        const uint32_t hm = __ballot_sync(0xffffffffu, hit);
        if (total != 0) {
            if (hm) {
                token = lo + (__ffs(hm) - 1);
            } else {  // unreachable for consistent sums: last element with weight
                const uint32_t nz = __ballot_sync(0xffffffffu, (v < hi) && r != 0);
                token = nz ? lo + (31 - __clz(nz)) : -1;
            }
        }
    }
    // status: OR over the CTA
    st = __reduce_or_sync(0xffffffffu, st);
    __syncthreads();
    if (lane == 0) sh.st_or[warp] = st;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int i = 0; i < kAccWarps; ++i) s |= sh.st_or[i];
        if (token < 0) s |= SVD_ST_EMPTY;
        else tok[j] = (int32_t)token;
        n_emitted[w] = j + (token >= 0 ? 1 : 0);
        status[w] = s;
    }
}

// ---- one window per cluster of eight CTAs --------------------------------------------------
constexpr int kAccCluster = 8;

// Inclusive scan of u128 values over a warp.
__device__ __forceinline__ u128 warp_scan_u128(u128 x) {
    const int lane = threadIdx.x & 31;
    uint64_t lo = (uint64_t)x, hi = (uint64_t)(x >> 64);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t olo = __shfl_up_sync(0xffffffffu, lo, o);
        const uint64_t ohi = __shfl_up_sync(0xffffffffu, hi, o);
        if (lane >= o) {
            const uint64_t nlo = lo + olo;
            hi = hi + ohi + (nlo < lo ? 1ull : 0ull);
            lo = nlo;
        }
    }
    return ((u128)hi << 64) | lo;
}

__global__ void __cluster_dims__(kAccCluster, 1, 1) __launch_bounds__(kAccCThreads, 1)
accept_cluster_kernel(const float *__restrict__ p, const int64_t *__restrict__ p_rows,
                      const float *__restrict__ q, const int64_t *__restrict__ q_rows,
                      const int32_t *__restrict__ draft, int k, int64_t V, uint64_t seed,
                      uint64_t woff, const float *__restrict__ uniforms,
                      int32_t *__restrict__ out_tokens, int32_t *__restrict__ n_emitted,
                      int32_t *__restrict__ status, int vec_ok) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ AcceptShared sh;
    __shared__ u128 s_wsum[2][kAccCWarps];  // this CTA's slice sums, per attempt
    __shared__ int s_cst[2];               // status bits of this CTA's slices, per attempt
    const int crank = (int)cluster.block_rank();
    const int64_t w = blockIdx.x / kAccCluster;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t *tok = out_tokens + w * (k + 1);
    griddep_wait();
    if (warp == 0)
        accept_tests(p, p_rows, q, q_rows, draft, k, V, seed, woff, uniforms, w, tok, sh, false);
    if (threadIdx.x < 2) s_cst[threadIdx.x] = 0;
    __syncthreads();
    const int j = sh.j;
    const uint32_t m2 = sh.m2;
    int st_win = sh.st_or[0];  // the accept tests' bits, the same in every CTA
    const float *rp = p + (p_rows ? p_rows[w * (k + 1) + j] : w * (k + 1) + j) * V;
    const float *rq = (j < k) ? q + (q_rows ? q_rows[w * k + j] : w * k + j) * V : nullptr;
    const bool vec = vec_ok != 0;

    // Level 1 over the cluster: CTA c takes piece c of the row, its warp i one eighth of that,
    // so slice 8 c + i in cluster order is slice i of CTA c.
    int64_t piece = (V + kAccCluster - 1) / kAccCluster;
    if (vec) piece = (piece + 3) & ~int64_t(3);
    auto slice_of = [&](int c, int i, int64_t *lo, int64_t *hi) {
        const int64_t c_lo = min(V, (int64_t)c * piece), c_hi = min(V, c_lo + piece);
        int64_t part = (c_hi - c_lo + kAccCWarps - 1) / kAccCWarps;
        if (vec) part = (part + 3) & ~int64_t(3);
        *lo = min(c_hi, c_lo + part * i);
        *hi = min(c_hi, *lo + part);
    };
    int64_t lo, hi;
    slice_of(crank, warp, &lo, &hi);
    int found = -1;
    u128 base = 0, total = 0, target = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        int st = 0;
        const u128 sum = (lo < hi) ? slice_sum<true>(rp, rq, lo, hi, vec, st) : (u128)0;
        st = __reduce_or_sync(0xffffffffu, st);
        if (lane == 0) {
            s_wsum[attempt][warp] = sum;
            if (st) atomicOr(&s_cst[attempt], st);
        }
        cluster.sync();
        if (warp == 0) {
            // lane t holds the cluster's slices kPer t .. kPer t + kPer - 1 (in row order)
            constexpr int kPer = kAccCluster * kAccCWarps / 32;
            u128 xs[kPer], lt = 0;
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int i = kPer * lane + e;
                xs[e] = *cluster.map_shared_rank(&s_wsum[attempt][i % kAccCWarps], i / kAccCWarps);
                lt += xs[e];
            }
            int sts = lane < kAccCluster ? *cluster.map_shared_rank(&s_cst[attempt], lane) : 0;
            sts = __reduce_or_sync(0xffffffffu, sts);
            const u128 incl = warp_scan_u128(lt);
            const u128 excl = incl - lt;
            const uint64_t tlo = __shfl_sync(0xffffffffu, (uint64_t)incl, 31);
            const uint64_t thi = __shfl_sync(0xffffffffu, (uint64_t)(incl >> 64), 31);
            const u128 R = ((u128)thi << 64) | tlo;
            const u128 tgt = (u128)m2 * R;
            const uint32_t hm = __ballot_sync(0xffffffffu, R != 0 && (incl << 24) > tgt);
            if (lane == 0) {
                sh.total = R;
                sh.target = tgt;
                sh.st_or[1] = sts;
                sh.found = -1;
            }
            if (hm && lane == __ffs(hm) - 1) {
                u128 run = excl;
                int e = 0;
                while (e < kPer - 1 && ((run + xs[e]) << 24) <= tgt) run += xs[e++];
                sh.found = kPer * lane + e;
                sh.base = run;
            }
        }
        cluster.sync();  // every read of another CTA's shared memory is done
        total = sh.total;
        target = sh.target;
        found = sh.found;
        base = sh.base;
        st_win |= sh.st_or[1];
        if (total == 0 && rq != nullptr) {
            st_win |= SVD_ST_ZERO_RESIDUAL;
            rq = nullptr;  // READING: an empty residual falls back to p_j
            continue;
        }
        break;
    }
    const int finisher = found >= 0 ? found / kAccCWarps : 0;
    if (crank != finisher) return;

    // ---- the CTA holding the crossing narrows its slice down to 32 elements ------------------
    int st = 0;
    if (found >= 0) {
        slice_of(finisher, found % kAccCWarps, &lo, &hi);
        while (hi - lo > 32) {
            const int64_t part = (hi - lo + kAccCWarps - 1) / kAccCWarps;
            const int64_t a = min(hi, lo + part * warp), bnd = min(hi, a + part);
            const u128 sum = (a < bnd) ? slice_sum<true>(rp, rq, a, bnd, false, st) : (u128)0;
            if (lane == 0) sh.part[warp] = sum;
            __syncthreads();
            if (threadIdx.x == 0) {
                int chosen = -1;
                u128 b = sh.base;
                for (int i = 0; i < kAccCWarps; ++i) {
                    if (((b + sh.part[i]) << 24) > target) {
                        chosen = i;
                        break;
                    }
                    b += sh.part[i];
                }
                sh.found = chosen;
                if (chosen >= 0) {
                    sh.base = b;
                    sh.lo = min(hi, lo + part * chosen);
                    sh.hi = min(hi, sh.lo + part);
                }
            }
            __syncthreads();
            if (sh.found < 0) break;  // unreachable for consistent sums
            lo = sh.lo;
            hi = sh.hi;
            base = sh.base;
            __syncthreads();
        }
    }
    // ---- final scan of at most 32 elements by warp 0 ------------------------------------------
    int64_t token = -1;
    if (warp == 0 && found >= 0) {
        const int64_t v = lo + lane;
        const u128 r = (v < hi) ? (u128)weight_fx<true>(rp, rq, v, st) : (u128)0;
        const u128 incl = warp_scan_u128(r);
        const bool hit = (v < hi) && (((base + incl) << 24) > target);
        const uint32_t hm = __ballot_sync(0xffffffffu, hit);
        if (hm) {
            token = lo + (__ffs(hm) - 1);
        } else {  // unreachable for consistent sums: last element with weight
            const uint32_t nz = __ballot_sync(0xffffffffu, (v < hi) && r != 0);
            token = nz ? lo + (31 - __clz(nz)) : -1;
        }
    }
    st = __reduce_or_sync(0xffffffffu, st);
    if (lane == 0) sh.st_or[warp] = st;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s2 = st_win;
        for (int i = 0; i < kAccCWarps; ++i) s2 |= sh.st_or[i];
        for (int i = 0; i < j; ++i) tok[i] = draft[w * k + i];
        for (int i = j; i <= k; ++i) tok[i] = -1;
        if (token < 0) s2 |= SVD_ST_EMPTY;
        else tok[j] = (int32_t)token;
        n_emitted[w] = j + (token >= 0 ? 1 : 0);
        status[w] = s2;
    }
}

int accept(const float *p, const int64_t *p_rows, const float *q, const int64_t *q_rows,
           const int32_t *tgt_am, const int32_t *draft, int64_t n, int k, int64_t V,
           uint64_t seed, uint64_t woff, const float *uniforms, int32_t *out_tokens,
           int32_t *n_emitted, int32_t *status, cudaStream_t stream) {
    if (n < 0 || k < 1 || k > SVD_K_MAX || V < 1 || V > 2147483647LL) return SVD_ERR_INVALID_ARG;
    if (n == 0) return SVD_OK;
    if (!p || !draft || !out_tokens || !n_emitted || !status) return SVD_ERR_INVALID_ARG;
    if (n > 2147483647LL) return SVD_ERR_UNSUPPORTED;
    const int vec_ok = (aligned16(p) && (!q || aligned16(q)) && (V % 4 == 0)) ? 1 : 0;
    // sampled windows fewer than the SMs (one verify pass): a cluster of eight CTAs each
    if (q && n * kAccCluster <= (int64_t)kAccCluster * sm_count() && V > 32 * kAccCluster) {
        SVD_CUDA_TRY(launch(accept_cluster_kernel, dim3((unsigned)(n * kAccCluster)),
                            dim3(kAccCThreads), 0, stream, false, p, p_rows, q, q_rows, draft, k,
                            V, seed, woff, uniforms, out_tokens, n_emitted, status, vec_ok));
        return SVD_OK;
    }
    SVD_CUDA_TRY(launch(accept_kernel, dim3((unsigned)n), dim3(kAccThreads), 0, stream, false,
                        p, p_rows, q, q_rows, tgt_am, draft, k, V, seed, woff, uniforms,
                        out_tokens, n_emitted, status, vec_ok));
    return SVD_OK;
}

}  // namespace svd
