// kv_attention.cu -- attention of the K+1 window queries over a quantised KV cache.
//
// "Decode is memory-bound ..." ("The ceiling"): at long context attention reads the whole KV
// cache on every pass, a second bandwidth stream beside the weights.  "100 tokens per second
// ..." ("The wall"; "The last mile"): the target's cache holds q8_0 keys and q4_0 values at a
// 32K context.
//
// Operation, for window position c (0..C-1) and query head h, kv head g = h / (Hq / Hkv):
//   s_j = scale * <q, k_j>   for the cache positions j = 0 .. n_past + c
//   o   = sum_j softmax(s)_j v_j
// Keys: int8 code q with value d * q; values: 4-bit code c with value d * (c - 8); one fp16 d
// per 32 dimensions of a position.  The head dimension is 128.
//
// Native cache layout.  A "unit" is 16 consecutive positions of one kv head, 3328 bytes (the
// q8_0 + q4_0 size of 16 positions):
//   [   0, 2048)  key codes biased by +128, in the A-fragment order of mma.m16n8k16 with rows =
//                 positions and k = dimensions: lane l owns the four 16-byte pieces at
//                 512 i + 16 l; piece i is the dimension block i (k-steps 2i, 2i+1), each
//                 k-step two words (a0, a1) and (a2, a3) of two codes per register;
//   [2048, 3072)  value codes in the A-fragment order of the transposed product (rows =
//                 dimensions, k = positions): lane l's word for m-tile mt sits at
//                 512 (mt / 4) + 16 l + 4 (mt % 4), register p's two codes at bits 4p, 16 + 4p;
//   [3072, 3200)  key scales, 16 bytes per row group r = 0..7: blocks 0..3 of position r, then
//                 of position r + 8;
//   [3200, 3328)  value scales in the same order.
// A layer's cache is [Hkv][units_cap][3328]; svd_kv_repack writes it from the canonical
// arrays.
//
// Kernel.  CTA (split, g, row group) covers a contiguous run of the head's units; each of its 8
// warps streams its own sub-run through a private ring of 4 slots (one bulk copy per unit,
// completing on an mbarrier) and keeps a flash-decoding state for up to 24 query rows
// (row = c * G + head-in-group):
//   S^T = K Q^T on f16 tensor cores: codes and bf16 queries are exact in f16, so each product
//     is exact; one fresh fp32 accumulator per 32-dimension block, scaled by d_k in fp32;
//   online softmax in base 2 with a lazy running max: the state is rescaled only when a score
//     exceeds the max by more than 8 (p <= 256 in between);
//   O^T += V^T P'^T on bf16 tensor cores with P' = p * d_v per value block: the value scale
//     varies along the contraction (positions), so it is folded into P, and P' is moved from
//     the accumulator layout into the B-fragment layout with movmatrix.
// The warps of a CTA merge in shared memory and write one partial (max, sum, O) per row; a
// second kernel, launched as a programmatic dependent, merges the splits of every row.
#include <algorithm>

#include "svd_common.cuh"

namespace svd {
namespace {

constexpr int kD = 128;
constexpr int kUnitPos = 16;
constexpr int kUnitBytes = 3328;
constexpr int kOffV = 2048, kOffKS = 3072, kOffVS = 3200;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kRing = 4;
constexpr int kRowsPerGroup = 24;
constexpr int kPitch = 132;  // floats per row of the merge buffer (conflict-free writes)
constexpr float kLazy = 8.0f;
constexpr int kRingBytes = kWarps * kRing * kUnitBytes;
constexpr int kMbarBytes = kWarps * kRing * 8;
constexpr int kSmemBytes = kRingBytes + kMbarBytes + 2 * kWarps * kRowsPerGroup * 4;
constexpr size_t kHeaderBytes = 256;
constexpr size_t kPartialBytes = (size_t)kRowsPerGroup * kD * 4 + (size_t)kRowsPerGroup * 8;
static_assert(kWarps * kRowsPerGroup * kPitch * 4 <= kRingBytes, "merge buffer fits the ring");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

struct KvaParams {
    const uint16_t *q;            // bf16 [C][Hq][128]
    const unsigned char *cache;   // native [Hkv][units_cap][3328]
    float *out;                   // [C][Hq][128]
    float *part_o;                // [cta][24][128]
    float2 *part_ml;              // [cta][24]: (max, sum) in base-2 units
    unsigned *flags;              // bit 0: a ring wait gave up
    int Hq, Hkv, G, C, n_past, units_cap, n_units, splits, n_rg, rows;
    float scale_log2;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
// Two f16 registers (1024 + u) from four biased key bytes, then minus 1152: the codes q exactly.
__device__ __forceinline__ void key_regs(uint32_t w, uint32_t &lo, uint32_t &hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(w), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(w), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}
// Four bf16 registers (128 + c) - 136 = c - 8 exactly, from one value word.
__device__ __forceinline__ void value_regs(uint32_t w, uint32_t a[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t v;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(w >> (4 * p)), "r"(0x000F000Fu),
            "r"(0x43004300u));
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(a[p]) : "r"(v), "r"(0x43084308u));
    }
}
__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) kv_attention_kernel(const KvaParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const int split = blockIdx.x, g = blockIdx.y, rg = blockIdx.z;
    const int cta = (rg * P.Hkv + g) * P.splits + split;
    float *wm = reinterpret_cast<float *>(smem + kRingBytes + kMbarBytes);
    float *wl = wm + kWarps * kRowsPerGroup;

    griddep_launch_dependents();  // the merge kernel may become resident and wait
    griddep_wait();               // queries and cache written by the kernels before this one

    // This warp's run of units.
    const int cb = (int)((long long)split * P.n_units / P.splits);
    const int ce = (int)((long long)(split + 1) * P.n_units / P.splits);
    const int wb = cb + (int)((long long)warp * (ce - cb) / kWarps);
    const int we = cb + (int)((long long)(warp + 1) * (ce - cb) / kWarps);
    const unsigned char *head = P.cache + (size_t)g * P.units_cap * kUnitBytes;
    const uint32_t ring = smem_u32(smem) + warp * kRing * kUnitBytes;
    const uint32_t mb0 = smem_u32(smem + kRingBytes) + warp * kRing * 8;
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRing; ++r) mbar_init(mb0 + 8 * r, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
#pragma unroll
        for (int r = 0; r < kRing; ++r)
            if (wb + r < we) {
                mbar_expect_tx(mb0 + 8 * r, kUnitBytes);
                bulk_g2s(ring + r * kUnitBytes, head + (size_t)(wb + r) * kUnitBytes, kUnitBytes,
                         mb0 + 8 * r);
            }
    }
    __syncwarp();

    // Query B fragments (f16): k-step ks, n-tile nt -> rows 8 nt + gid, dims 16 ks + 2 tig (+8).
    uint32_t qf[8][NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int row = rg * kRowsPerGroup + 8 * nt + gid;
        const bool ok = row < P.rows;
        const int c = ok ? row / P.G : 0, h = g * P.G + (ok ? row % P.G : 0);
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(P.q + ((size_t)c * P.Hq + h) * kD);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t bits = ok ? __ldg(qrow + 8 * ks + tig + 4 * j) : 0u;
                qf[ks][nt][j] = pack_f16(__uint_as_float(bits << 16),
                                         __uint_as_float(bits & 0xFFFF0000u));
            }
    }

    float o[8][NT][4];
    float m[NT][2], l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            m[nt][e] = -INFINITY;
            l[nt][e] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
    }
    const int L = P.n_past + P.C;
    bool failed = false;
    int it_f = 0;

    for (int u = wb, it = 0; u < we; ++u, ++it) {
        const int slot = it % kRing;
        const bool ok = mbar_wait_ok(mb0 + 8 * slot, (uint32_t)(it / kRing) & 1u);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            failed = true;
            it_f = it;
            break;
        }
        const uint32_t su = ring + slot * kUnitBytes;
        const uint4 ksr = lds128(su + kOffKS + 16 * gid);
        const float scl = P.scale_log2;
        const float2 kA01 = half2_bits_to_float2(ksr.x), kA23 = half2_bits_to_float2(ksr.y);
        const float2 kB01 = half2_bits_to_float2(ksr.z), kB23 = half2_bits_to_float2(ksr.w);
        const float kA[4] = {kA01.x * scl, kA01.y * scl, kA23.x * scl, kA23.y * scl};
        const float kB[4] = {kB01.x * scl, kB01.y * scl, kB23.x * scl, kB23.y * scl};

        // S^T = K Q^T, one fresh accumulator per 32-dimension block.
        float s[NT][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint4 kw = lds128(su + 512 * b + 16 * lane);
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
            uint32_t a[4];
            key_regs(kw.x, a[0], a[1]);
            key_regs(kw.y, a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], a, qf[2 * b][nt][0], qf[2 * b][nt][1]);
            key_regs(kw.z, a[0], a[1]);
            key_regs(kw.w, a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_f16(acc[nt], a, qf[2 * b + 1][nt][0], qf[2 * b + 1][nt][1]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (b == 0) {
                    s[nt][0] = kA[0] * acc[nt][0];
                    s[nt][1] = kA[0] * acc[nt][1];
                    s[nt][2] = kB[0] * acc[nt][2];
                    s[nt][3] = kB[0] * acc[nt][3];
                } else {
                    s[nt][0] = fmaf(kA[b], acc[nt][0], s[nt][0]);
                    s[nt][1] = fmaf(kA[b], acc[nt][1], s[nt][1]);
                    s[nt][2] = fmaf(kB[b], acc[nt][2], s[nt][2]);
                    s[nt][3] = fmaf(kB[b], acc[nt][3], s[nt][3]);
                }
            }
        }

        const uint4 vsr = lds128(su + kOffVS + 16 * gid);
        float2 vA01 = half2_bits_to_float2(vsr.x), vA23 = half2_bits_to_float2(vsr.y);
        float2 vB01 = half2_bits_to_float2(vsr.z), vB23 = half2_bits_to_float2(vsr.w);
        const int pA = u * kUnitPos + gid, pB = pA + 8;
        if (u * kUnitPos + kUnitPos - 1 > P.n_past) {
            // The unit reaches into the window: mask what each row may not see, and make the
            // positions past the cache's end contribute exact zeros whatever their bytes hold.
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = rg * kRowsPerGroup + 8 * nt + 2 * tig + e;
                    const int lim = P.n_past + min(row / P.G, P.C - 1);
                    if (pA > lim) s[nt][e] = -INFINITY;
                    if (pB > lim) s[nt][e + 2] = -INFINITY;
                }
            if (pA >= L) vA01 = vA23 = make_float2(0.f, 0.f);
            if (pB >= L) vB01 = vB23 = make_float2(0.f, 0.f);
        }

        // Online softmax with a lazy running max.
        bool need = false;
        float mloc[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mloc[nt][e] = fmaxf(s[nt][e], s[nt][e + 2]);
                need |= mloc[nt][e] > m[nt][e] + kLazy;
            }
        if (__any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float mx = mloc[nt][e];
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
                    const float mn = fmaxf(m[nt][e], mx);
                    const float f = m[nt][e] == -INFINITY ? 0.f : ex2(m[nt][e] - mn);
                    m[nt][e] = mn;
                    l[nt][e] *= f;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        o[mt][nt][e] *= f;
                        o[mt][nt][e + 2] *= f;
                    }
                }
        }
        float p[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float ms = m[nt][e] == -INFINITY ? 0.f : m[nt][e];
                p[nt][e] = ex2(s[nt][e] - ms);
                p[nt][e + 2] = ex2(s[nt][e + 2] - ms);
                l[nt][e] += p[nt][e] + p[nt][e + 2];
            }

        // O^T += V^T P'^T, P' = p * d_v of the value block.
        const uint4 vw0 = lds128(su + kOffV + 16 * lane);
        const uint4 vw1 = lds128(su + kOffV + 512 + 16 * lane);
        const uint32_t vw[8] = {vw0.x, vw0.y, vw0.z, vw0.w, vw1.x, vw1.y, vw1.z, vw1.w};
        __syncwarp();
        if (lane == 0 && u + kRing < we) {
            mbar_expect_tx(mb0 + 8 * slot, kUnitBytes);
            bulk_g2s(su, head + (size_t)(u + kRing) * kUnitBytes, kUnitBytes, mb0 + 8 * slot);
        }
        const float vA[4] = {vA01.x, vA01.y, vA23.x, vA23.y};
        const float vB[4] = {vB01.x, vB01.y, vB23.x, vB23.y};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t b0[NT], b1[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                b0[nt] = transpose8x8(pack_bf16(p[nt][0] * vA[b], p[nt][1] * vA[b]));
                b1[nt] = transpose8x8(pack_bf16(p[nt][2] * vB[b], p[nt][3] * vB[b]));
            }
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
                uint32_t a[4];
                value_regs(vw[2 * b + mm], a);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16(o[2 * b + mm][nt], a, b0[nt], b1[nt]);
            }
        }
    }

    if (failed) {
        // A ring wait gave up at iteration it_f: record it, then wait (bounded) for the copies
        // still in flight -- units wb + it_f .. wb + it_f + kRing - 1 -- before the shared memory
        // is reused.
        if (lane == 0) {
            atomicOr(P.flags, 1u);
            for (int j = it_f; j < it_f + kRing && wb + j < we; ++j)
                (void)mbar_wait_ok(mb0 + 8 * (j % kRing), (uint32_t)(j / kRing) & 1u);
        }
        __syncwarp();
    }

    // Row sums over the 8 position lanes; m is already uniform across them.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float v = l[nt][e];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
            l[nt][e] = v;
        }
    if (gid == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                wm[warp * kRowsPerGroup + 8 * nt + 2 * tig + e] = m[nt][e];
                wl[warp * kRowsPerGroup + 8 * nt + 2 * tig + e] = l[nt][e];
            }
    }
    __syncthreads();  // every warp is done with its ring: the ring becomes the merge buffer

    float *buf = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = 8 * nt + 2 * tig + e;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kRowsPerGroup + row]);
            const float mine = wm[warp * kRowsPerGroup + row];
            const float f = mine == -INFINITY ? 0.f : ex2(mine - M);
            float *dst = buf + (warp * kRowsPerGroup + row) * kPitch;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                dst[16 * mt + gid] = o[mt][nt][e] * f;
                dst[16 * mt + gid + 8] = o[mt][nt][e + 2] * f;
            }
        }
    __syncthreads();

    for (int idx = threadIdx.x; idx < 8 * NT * 32; idx += kThreads) {
        const int row = idx >> 5, d4 = idx & 31;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float4 v =
                *reinterpret_cast<const float4 *>(buf + (w * kRowsPerGroup + row) * kPitch + 4 * d4);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        *reinterpret_cast<float4 *>(P.part_o + ((size_t)cta * kRowsPerGroup + row) * kD + 4 * d4) = acc;
    }
    if (threadIdx.x < 8 * NT) {
        const int row = threadIdx.x;
        float M = -INFINITY, S = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kRowsPerGroup + row]);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = wm[w * kRowsPerGroup + row];
            S += mw == -INFINITY ? 0.f : ex2(mw - M) * wl[w * kRowsPerGroup + row];
        }
        P.part_ml[(size_t)cta * kRowsPerGroup + row] = make_float2(M, S);
    }
}

// One warp per (row group, kv head, row): merges the splits' partials and writes o = O / l.
__global__ void __launch_bounds__(128) kv_attention_merge_kernel(const KvaParams P) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int wgl = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int row = wgl % kRowsPerGroup, gg = wgl / kRowsPerGroup;
    const int g = gg % P.Hkv, rg = gg / P.Hkv;
    if (rg >= P.n_rg) return;
    const int grow = rg * kRowsPerGroup + row;
    if (grow >= P.rows) return;
    const int c = grow / P.G, h = g * P.G + grow % P.G;
    const size_t base = (size_t)(rg * P.Hkv + g) * P.splits;
    float M = -INFINITY;
    for (int s = lane; s < P.splits; s += 32) M = fmaxf(M, P.part_ml[(base + s) * kRowsPerGroup + row].x);
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 1));
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 2));
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 4));
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 8));
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 16));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float S = 0.f;
#pragma unroll 4
    for (int s = 0; s < P.splits; ++s) {
        const float2 ml = P.part_ml[(base + s) * kRowsPerGroup + row];
        const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
        const float4 v =
            *reinterpret_cast<const float4 *>(P.part_o + ((base + s) * kRowsPerGroup + row) * kD + 4 * lane);
        S += w * ml.y;
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    }
    const float inv = 1.f / S;
    *reinterpret_cast<float4 *>(P.out + ((size_t)c * P.Hq + h) * kD + 4 * lane) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// ---- native layout: byte offsets inside a unit ----------------------------------------------
__device__ __forceinline__ int key_code_offset(int r, int i) {
    const int ks = i >> 4, ii = i & 15, lane = (r & 7) * 4 + ((ii & 7) >> 1);
    return 512 * (ks >> 1) + 16 * lane + 8 * (ks & 1) + 4 * (ii >> 3) + 2 * (r >> 3) + (ii & 1);
}
// Byte holding the value codes of dimensions 16 mt + gid (low nibble) and 16 mt + gid + 8 (high
// nibble) at position r of the unit.
__device__ __forceinline__ int value_byte_offset(int r, int mt, int gid) {
    const int lane = gid * 4 + ((r & 7) >> 1);
    return kOffV + 512 * (mt >> 2) + 16 * lane + 4 * (mt & 3) + (r >> 3) + 2 * (r & 1);
}
__device__ __forceinline__ int scale_offset(int r, int b) { return 16 * (r & 7) + 2 * (4 * (r >> 3) + b); }

// One thread per (kv head, position): canonical row -> native unit bytes.
__global__ void kv_repack_kernel(const int8_t *kc, const uint16_t *ks, const uint8_t *vc,
                                 const uint16_t *vs, int Hkv, int ld, int p0, int p1,
                                 unsigned char *cache, int units_cap) {
    const long long n = (long long)(p1 - p0) * Hkv;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    const int g = (int)(idx / (p1 - p0)), pos = p0 + (int)(idx % (p1 - p0)), r = pos & 15;
    unsigned char *unit = cache + ((size_t)g * units_cap + (pos >> 4)) * kUnitBytes;
    const size_t row = (size_t)g * ld + pos;
    const int8_t *krow = kc + row * kD;
    for (int i = 0; i < kD; ++i) unit[key_code_offset(r, i)] = (unsigned char)((int)krow[i] + 128);
    const uint8_t *vrow = vc + row * (kD / 2);
    for (int mt = 0; mt < 8; ++mt)
        for (int gi = 0; gi < 8; ++gi) {
            const int d0 = 16 * mt + gi, d1 = d0 + 8;
            const int c0 = (vrow[d0 >> 1] >> (4 * (d0 & 1))) & 15;
            const int c1 = (vrow[d1 >> 1] >> (4 * (d1 & 1))) & 15;
            unit[value_byte_offset(r, mt, gi)] = (unsigned char)(c0 | (c1 << 4));
        }
    for (int b = 0; b < 4; ++b) {
        *reinterpret_cast<uint16_t *>(unit + kOffKS + scale_offset(r, b)) = ks[row * 4 + b];
        *reinterpret_cast<uint16_t *>(unit + kOffVS + scale_offset(r, b)) = vs[row * 4 + b];
    }
}

// The inverse: native unit bytes -> canonical row.
__global__ void kv_unpack_kernel(const unsigned char *cache, int units_cap, int Hkv, int p0,
                                 int p1, int8_t *kc, uint16_t *ks, uint8_t *vc, uint16_t *vs,
                                 int ld) {
    const long long n = (long long)(p1 - p0) * Hkv;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    const int g = (int)(idx / (p1 - p0)), pos = p0 + (int)(idx % (p1 - p0)), r = pos & 15;
    const unsigned char *unit = cache + ((size_t)g * units_cap + (pos >> 4)) * kUnitBytes;
    const size_t row = (size_t)g * ld + pos;
    for (int i = 0; i < kD; ++i) kc[row * kD + i] = (int8_t)((int)unit[key_code_offset(r, i)] - 128);
    uint8_t bytes[kD / 2];
    for (int t = 0; t < kD / 2; ++t) bytes[t] = 0;
    for (int mt = 0; mt < 8; ++mt)
        for (int gi = 0; gi < 8; ++gi) {
            const int d0 = 16 * mt + gi, d1 = d0 + 8;
            const int v = unit[value_byte_offset(r, mt, gi)];
            bytes[d0 >> 1] |= (uint8_t)((v & 15) << (4 * (d0 & 1)));
            bytes[d1 >> 1] |= (uint8_t)((v >> 4) << (4 * (d1 & 1)));
        }
    for (int t = 0; t < kD / 2; ++t) vc[row * (kD / 2) + t] = bytes[t];
    for (int b = 0; b < 4; ++b) {
        ks[row * 4 + b] = *reinterpret_cast<const uint16_t *>(unit + kOffKS + scale_offset(r, b));
        vs[row * 4 + b] = *reinterpret_cast<const uint16_t *>(unit + kOffVS + scale_offset(r, b));
    }
}

int units_for(int positions) { return (positions + kUnitPos - 1) / kUnitPos; }

struct KvaGeom {
    int G, rows, n_rg, nt, splits, n_units;
    size_t ctas;
};

bool kva_geom(int Hq, int Hkv, int n_past, int C, KvaGeom &k) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || C <= 0 || n_past < 0) return false;
    k.G = Hq / Hkv;
    const long long rows = (long long)C * k.G;
    if (rows > (1 << 20) || (long long)C * Hq * kD > (1ll << 31) - 1) return false;
    k.rows = (int)rows;
    k.n_rg = (k.rows + kRowsPerGroup - 1) / kRowsPerGroup;
    k.nt = (std::min(k.rows, kRowsPerGroup) + 7) / 8;
    k.n_units = units_for(n_past + C);
    const int heads = Hkv * k.n_rg;
    int splits = std::max(1, sm_count() / heads);
    splits = std::min(splits, std::max(1, k.n_units / (2 * kWarps)));
    k.splits = splits;
    k.ctas = (size_t)splits * heads;
    return true;
}

size_t kva_workspace(int Hq, int Hkv, int C) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || C <= 0) return 0;
    const long long rows = (long long)C * (Hq / Hkv);
    const long long heads = (long long)Hkv * ((rows + kRowsPerGroup - 1) / kRowsPerGroup);
    const long long ctas = std::max<long long>(heads, sm_count());
    return kHeaderBytes + (size_t)ctas * kPartialBytes;
}

template <int NT>
cudaError_t launch_kva(const KvaParams &P, dim3 grid, cudaStream_t stream) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kv_attention_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    e = launch(kv_attention_kernel<NT>, grid, dim3(kThreads), kSmemBytes, stream, false, P);
    if (e != cudaSuccess) return e;
    const int warps = P.n_rg * P.Hkv * kRowsPerGroup;
    return launch(kv_attention_merge_kernel, dim3((warps + 3) / 4), dim3(128), 0, stream, true, P);
}

}  // namespace
}  // namespace svd

using namespace svd;

extern "C" size_t svd_kv_cache_bytes(int n_kv_heads, int capacity) {
    if (n_kv_heads <= 0 || capacity <= 0) return 0;
    return (size_t)n_kv_heads * units_for(capacity) * kUnitBytes;
}

extern "C" int svd_kv_repack(const int8_t *k_codes, const uint16_t *k_scales,
                             const uint8_t *v_codes, const uint16_t *v_scales, int n_kv_heads,
                             int ld, int pos_begin, int pos_end, void *cache, int capacity,
                             svd_stream_t stream) {
    if (!k_codes || !k_scales || !v_codes || !v_scales || !cache || n_kv_heads <= 0 ||
        capacity <= 0 || pos_begin < 0 || pos_end < pos_begin || pos_end > capacity || pos_end > ld)
        return SVD_ERR_INVALID_ARG;
    if (!aligned16(cache)) return SVD_ERR_INVALID_ARG;
    if (pos_end == pos_begin) return SVD_OK;
    const long long n = (long long)(pos_end - pos_begin) * n_kv_heads;
    kv_repack_kernel<<<(unsigned)((n + 127) / 128), 128, 0, (cudaStream_t)stream>>>(
        k_codes, k_scales, v_codes, v_scales, n_kv_heads, ld, pos_begin, pos_end,
        (unsigned char *)cache, units_for(capacity));
    SVD_CUDA_TRY(cudaGetLastError());
    return SVD_OK;
}

extern "C" int svd_kv_unpack(const void *cache, int capacity, int n_kv_heads, int pos_begin,
                             int pos_end, int8_t *k_codes, uint16_t *k_scales, uint8_t *v_codes,
                             uint16_t *v_scales, int ld, svd_stream_t stream) {
    if (!k_codes || !k_scales || !v_codes || !v_scales || !cache || n_kv_heads <= 0 ||
        capacity <= 0 || pos_begin < 0 || pos_end < pos_begin || pos_end > capacity || pos_end > ld)
        return SVD_ERR_INVALID_ARG;
    if (!aligned16(cache)) return SVD_ERR_INVALID_ARG;
    if (pos_end == pos_begin) return SVD_OK;
    const long long n = (long long)(pos_end - pos_begin) * n_kv_heads;
    kv_unpack_kernel<<<(unsigned)((n + 127) / 128), 128, 0, (cudaStream_t)stream>>>(
        (const unsigned char *)cache, units_for(capacity), n_kv_heads, pos_begin, pos_end, k_codes,
        k_scales, v_codes, v_scales, ld);
    SVD_CUDA_TRY(cudaGetLastError());
    return SVD_OK;
}

extern "C" size_t svd_kv_attention_workspace_bytes(int n_q_heads, int n_kv_heads, int C) {
    return kva_workspace(n_q_heads, n_kv_heads, C);
}

extern "C" int svd_kv_attention(const uint16_t *q, const void *cache, int capacity, int n_q_heads,
                                int n_kv_heads, int n_past, int C, float scale, float *out,
                                void *workspace, size_t workspace_bytes, svd_stream_t stream) {
    KvaGeom k;
    if (!q || !cache || !out || capacity <= 0 || !kva_geom(n_q_heads, n_kv_heads, n_past, C, k) ||
        (long long)n_past + C > capacity || !(scale > 0.f) || !(scale < INFINITY))
        return SVD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(cache) || !aligned16(out)) return SVD_ERR_INVALID_ARG;
    const size_t need = kva_workspace(n_q_heads, n_kv_heads, C);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return SVD_ERR_WORKSPACE;
    KvaParams P;
    P.q = q;
    P.cache = (const unsigned char *)cache;
    P.out = out;
    P.flags = (unsigned *)workspace;
    P.part_ml = (float2 *)((unsigned char *)workspace + kHeaderBytes);
    P.part_o = (float *)((unsigned char *)workspace + kHeaderBytes + k.ctas * kRowsPerGroup * 8);
    P.Hq = n_q_heads;
    P.Hkv = n_kv_heads;
    P.G = k.G;
    P.C = C;
    P.n_past = n_past;
    P.units_cap = units_for(capacity);
    P.n_units = k.n_units;
    P.splits = k.splits;
    P.n_rg = k.n_rg;
    P.rows = k.rows;
    P.scale_log2 = scale * 1.4426950408889634f;
    const dim3 grid(k.splits, n_kv_heads, k.n_rg);
    cudaError_t e;
    switch (k.nt) {
        case 1: e = launch_kva<1>(P, grid, (cudaStream_t)stream); break;
        case 2: e = launch_kva<2>(P, grid, (cudaStream_t)stream); break;
        default: e = launch_kva<3>(P, grid, (cudaStream_t)stream); break;
    }
    SVD_CUDA_TRY(e);
    return SVD_OK;
}
