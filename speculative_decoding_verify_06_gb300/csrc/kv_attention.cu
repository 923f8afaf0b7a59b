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
constexpr int kQPitch = 272;  // bytes per f16 query row in shared memory (conflict-free ldmatrix)
constexpr int kRingBytes = kWarps * kRing * kUnitBytes;
constexpr int kMbarBytes = kWarps * kRing * 8;
constexpr int kQBytes = kRowsPerGroup * kQPitch;
constexpr int kCorrBytes = kRowsPerGroup * 4 * 4;
constexpr int kSmemBytes = kRingBytes + kMbarBytes + kQBytes + kCorrBytes + 2 * kWarps * kRowsPerGroup * 4;
constexpr int kMaxSplitRounds = 5;  // splits per row merged by one warp: up to 32 per round
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
    const float *k_new, *v_new;   // the window's fp32 keys / values to append first, or null
    int ld_new;                   // floats between window positions of k_new / v_new
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
// Two f16 registers (1024 + u) = q + 1152 from four biased key bytes u = q + 128 (exact); the
// 1152 * sum(q) offset of each 32-dimension block is removed through the accumulator's initial
// value.
__device__ __forceinline__ void key_regs(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(w), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(w), "r"(0x64646464u));
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
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// Two fp32 values in one 64-bit register pair, for the paired fp32 instructions of sm_100+.
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t f2(float lo, float hi) {
    f2_t r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unf2(f2_t v, float &lo, float &hi) {
    asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t mul2(f2_t a, f2_t b) {
    f2_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t fma2(f2_t a, f2_t b, f2_t c) {
    f2_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f2_t add2(f2_t a, f2_t b) {
    f2_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// First product of a block's accumulator: C = (c0, c1, c0, c1), the per-row offset removal.
__device__ __forceinline__ void mma_f16_init(float d[4], const uint32_t a[4], uint32_t b0,
                                             uint32_t b1, float c0, float c1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%10,%11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
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

// One warp quantises one cache position of one kv head -- its 128 key values to q8_0 and 128
// value values to q4_0, block by block of 32 (lane l holds dimension 32 b + l), in the fp32 steps
// of the formats' definitions (llama.cpp's block types of the same names):
//   q8_0: d = max|x| / 127, q = round-half-away(x * (1/d)), 0 when d = 0;
//   q4_0: m = the value of largest magnitude (the lowest dimension on ties), d = m / -8,
//         c = min(15, trunc(x * (1/d) + 8.5)), 8 when d = 0;
// and writes the codes and fp16 scales (round to nearest even) into the position's native unit.
__device__ __forceinline__ void append_position(const float *kr, const float *vr,
                                                unsigned char *unit, int r, int lane) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int dim = 32 * b + lane;
        const float x = kr[dim];
        float amax = fabsf(x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float d = __fdiv_rn(amax, 127.0f);
        const float id = d != 0.f ? __fdiv_rn(1.0f, d) : 0.f;
        const int q = (int)roundf(__fmul_rn(x, id));
        unit[key_code_offset(r, dim)] = (unsigned char)(q + 128);
        if (lane == 0)
            *reinterpret_cast<uint16_t *>(unit + kOffKS + scale_offset(r, b)) =
                __half_as_ushort(__float2half_rn(d));

        const float y = vr[dim];
        float ay = fabsf(y);
        int at = lane;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oa = __shfl_xor_sync(0xFFFFFFFFu, ay, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, at, o);
            if (oa > ay || (oa == ay && oi < at)) {
                ay = oa;
                at = oi;
            }
        }
        const float m = __shfl_sync(0xFFFFFFFFu, y, at);
        const float dv = __fdiv_rn(m, -8.0f);
        const float idv = dv != 0.f ? __fdiv_rn(1.0f, dv) : 0.f;
        const int cq = min(15, (int)__fadd_rn(__fmul_rn(y, idv), 8.5f));
        // Dimensions 16 mt + j and 16 mt + j + 8 share a byte: lane l (l & 8 == 0) takes the code
        // of lane l + 8 for the high nibble.
        const int hi = __shfl_down_sync(0xFFFFFFFFu, cq, 8);
        if ((lane & 8) == 0)
            unit[value_byte_offset(r, dim >> 4, dim & 7)] = (unsigned char)(cq | (hi << 4));
        if (lane == 0)
            *reinterpret_cast<uint16_t *>(unit + kOffVS + scale_offset(r, b)) =
                __half_as_ushort(__float2half_rn(dv));
    }
}

// One warp per (window position c, kv head g): appends position n_past + c (append_position).
__global__ void kv_append_kernel(const float *k, const float *v, int ld, int C, int Hkv,
                                 int n_past, unsigned char *cache, int units_cap) {
    griddep_launch_dependents();  // the attention that reads these positions may become resident
    griddep_wait();               // k and v come from the kernel before this one
    const int w = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (w >= C * Hkv) return;
    const int c = w / Hkv, g = w % Hkv, pos = n_past + c;
    append_position(k + (size_t)c * ld + (size_t)g * kD, v + (size_t)c * ld + (size_t)g * kD,
                    cache + ((size_t)g * units_cap + (pos >> 4)) * kUnitBytes, pos & 15, lane);
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) kv_attention_kernel(const KvaParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const int split = blockIdx.x, g = blockIdx.y, rg = blockIdx.z;
    const int cta = (rg * P.Hkv + g) * P.splits + split;
    float *corr_s = reinterpret_cast<float *>(smem + kRingBytes + kMbarBytes + kQBytes);
    float *wm = corr_s + kRowsPerGroup * 4;
    float *wl = wm + kWarps * kRowsPerGroup;
    const uint32_t qs = smem_u32(smem + kRingBytes + kMbarBytes);

    griddep_launch_dependents();  // the merge kernel may become resident and wait

    // This CTA's and this warp's runs of units.  In append mode the last split, which holds the
    // window and quantises it first, gets about two units per warp fewer.
    const int shift = P.k_new ? min(2 * kWarps, P.n_units / (2 * P.splits)) : 0;
    const int cb = min(P.n_units, (int)((long long)split * (P.n_units + shift) / P.splits));
    const int ce = min(P.n_units, (int)((long long)(split + 1) * (P.n_units + shift) / P.splits));
    const int wb = cb + (int)((long long)warp * (ce - cb) / kWarps);
    const int we = cb + (int)((long long)(warp + 1) * (ce - cb) / kWarps);
    const unsigned char *head = P.cache + (size_t)g * P.units_cap * kUnitBytes;
    const uint32_t ring = smem_u32(smem) + warp * kRing * kUnitBytes;
    const uint32_t mb0 = smem_u32(smem + kRingBytes) + warp * kRing * 8;
    // Units wholly before the window's first position hold only positions written by earlier
    // passes (an append before this kernel writes from n_past on), so this warp's first copies of
    // them go out before the dependency wait.
    const int early_end = min(we, P.n_past / kUnitPos);
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRing; ++r) mbar_init(mb0 + 8 * r, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
#pragma unroll
        for (int r = 0; r < kRing; ++r)
            if (wb + r < early_end) {
                mbar_expect_tx(mb0 + 8 * r, kUnitBytes);
                bulk_g2s(ring + r * kUnitBytes, head + (size_t)(wb + r) * kUnitBytes, kUnitBytes,
                         mb0 + 8 * r);
            }
    }
    griddep_wait();  // queries and cache written by the kernels before this one
    // polls after which a ring wait gives up: word 1 of the workspace minus one when it is set
    // (a test hook; 1 makes every ring wait give up at once)
    const unsigned poll_set = *(reinterpret_cast<volatile const unsigned *>(P.flags) + 1);
    const uint32_t poll_limit = poll_set ? poll_set - 1u : kDefaultPolls;
    // The window's positions inside this CTA's units (append mode) are quantised into the cache
    // by this CTA (no other CTA reads them) and made visible to the bulk copies that read them
    // back.  When no warp's first kRing units hold one, the prologue copies go first and the
    // append overlaps their latency (ordered by the barrier after the query staging); otherwise
    // it comes before the prologue.
    const int p_lo = max(P.n_past, cb * kUnitPos), p_hi = min(P.n_past + P.C, ce * kUnitPos);
    const bool do_append = P.k_new != nullptr && p_lo < p_hi;
    bool late_ok = do_append;
    if (do_append) {
        for (int u = p_lo / kUnitPos; u <= (p_hi - 1) / kUnitPos; ++u)
            for (int w = 0; w < kWarps; ++w) {
                const int b0 = cb + (int)((long long)w * (ce - cb) / kWarps);
                const int b1 = cb + (int)((long long)(w + 1) * (ce - cb) / kWarps);
                if (u >= b0 && u < b1 && u < b0 + kRing) late_ok = false;
            }
    }
    auto append_window = [&]() {
        for (int pos = p_lo + warp; pos < p_hi; pos += kWarps) {
            const int c = pos - P.n_past;
            append_position(P.k_new + (size_t)c * P.ld_new + (size_t)g * kD,
                            P.v_new + (size_t)c * P.ld_new + (size_t)g * kD,
                            const_cast<unsigned char *>(head) + (size_t)(pos >> 4) * kUnitBytes,
                            pos & 15, lane);
        }
        __threadfence();
    };
    if (do_append && !late_ok) {
        append_window();
        __syncthreads();
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRing; ++r)
            if (wb + r < we && wb + r >= early_end) {
                mbar_expect_tx(mb0 + 8 * r, kUnitBytes);
                bulk_g2s(ring + r * kUnitBytes, head + (size_t)(wb + r) * kUnitBytes, kUnitBytes,
                         mb0 + 8 * r);
            }
    }

    // The CTA's query rows (row = c * G + head in group) as f16 in shared memory, zero past the
    // last row; each warp reads them as B fragments with ldmatrix.
    for (int idx = threadIdx.x; idx < kRowsPerGroup * (kD / 2); idx += kThreads) {
        const int r = idx / (kD / 2), pr = idx % (kD / 2);
        const int row = rg * kRowsPerGroup + r;
        uint32_t bits = 0u;
        if (row < P.rows) {
            const int c = row / P.G, h = g * P.G + row % P.G;
            bits = __ldg(reinterpret_cast<const uint32_t *>(P.q + ((size_t)c * P.Hq + h) * kD) + pr);
        }
        const uint32_t v = pack_f16(__uint_as_float(bits << 16), __uint_as_float(bits & 0xFFFF0000u));
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(qs + r * kQPitch + 4 * pr), "r"(v));
    }
    if (do_append && late_ok) append_window();
    __syncthreads();
    if (do_append && late_ok) asm volatile("fence.proxy.async.global;" ::: "memory");
    // -1152 * (sum of the f16 query values of each row and 32-dimension block), in fp32.
    if (threadIdx.x < kRowsPerGroup * 4) {
        const int r = threadIdx.x >> 2, b = threadIdx.x & 3;
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = lds128(qs + r * kQPitch + 64 * b + 16 * i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = half2_bits_to_float2(w[j]);
                acc += f.x + f.y;
            }
        }
        corr_s[r * 4 + b] = -1152.f * acc;
    }
    __syncthreads();
    float corr[4][NT][2];
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) corr[b][nt][e] = corr_s[(8 * nt + 2 * tig + e) * 4 + b];
    // ldmatrix row address of this lane: matrix i = lane / 8 covers k-step 2b + i / 2, dims
    // +8 (i % 2); row 8 nt + lane % 8.
    const uint32_t qlane = qs + (lane & 7) * kQPitch + 2 * (16 * (lane >> 4) + 8 * ((lane >> 3) & 1));

    float o[8][NT][4];
    float m[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) m[nt][e] = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
    }
    const int L = P.n_past + P.C;
    const float scl = P.scale_log2;
    const f2_t scl2 = f2(scl, scl);
    const float lazy = kLazy / scl;  // the rescale threshold in code units
    f2_t nm[NT], lsum[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        nm[nt] = f2(0.f, 0.f);
        lsum[nt] = f2(0.f, 0.f);
    }
    bool failed = false;
    int it_f = 0;

    for (int u = wb, it = 0; u < we; ++u, ++it) {
        const int slot = it % kRing;
        const bool ok = mbar_wait_ok(mb0 + 8 * slot, (uint32_t)(it / kRing) & 1u, poll_limit);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            failed = true;
            it_f = it;
            break;
        }
        const uint32_t su = ring + slot * kUnitBytes;
        const uint4 ksr = lds128(su + kOffKS + 16 * gid);
        const float2 kA01 = half2_bits_to_float2(ksr.x), kA23 = half2_bits_to_float2(ksr.y);
        const float2 kB01 = half2_bits_to_float2(ksr.z), kB23 = half2_bits_to_float2(ksr.w);
        const f2_t kA[4] = {f2(kA01.x, kA01.x), f2(kA01.y, kA01.y), f2(kA23.x, kA23.x),
                            f2(kA23.y, kA23.y)};
        const f2_t kB[4] = {f2(kB01.x, kB01.x), f2(kB01.y, kB01.y), f2(kB23.x, kB23.x),
                            f2(kB23.y, kB23.y)};

        // S^T = K Q^T in code units, one fresh accumulator per 32-dimension block scaled by its
        // key scale: sA = the row pair of position gid, sB = of position gid + 8.
        f2_t sA[NT], sB[NT];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint4 kw = lds128(su + 512 * b + 16 * lane);
            float acc[NT][4];
            uint32_t qb[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) ldsm_x4(qlane + 8 * nt * kQPitch + 64 * b, qb[nt]);
            uint32_t a[4];
            key_regs(kw.x, a[0], a[1]);
            key_regs(kw.y, a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_f16_init(acc[nt], a, qb[nt][0], qb[nt][1], corr[b][nt][0], corr[b][nt][1]);
            key_regs(kw.z, a[0], a[1]);
            key_regs(kw.w, a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], a, qb[nt][2], qb[nt][3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const f2_t x = f2(acc[nt][0], acc[nt][1]), y = f2(acc[nt][2], acc[nt][3]);
                sA[nt] = b == 0 ? mul2(x, kA[0]) : fma2(x, kA[b], sA[nt]);
                sB[nt] = b == 0 ? mul2(y, kB[0]) : fma2(y, kB[b], sB[nt]);
            }
        }
        float s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            unf2(sA[nt], s[nt][0], s[nt][1]);
            unf2(sB[nt], s[nt][2], s[nt][3]);
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

        // Online softmax in base 2 with a lazy running max.  m is kept in code units (the scale
        // is positive), with nm = -m * scale for the exponent's fused multiply-add.
        bool need = false;
        float mloc[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mloc[nt][e] = fmaxf(s[nt][e], s[nt][e + 2]);
                need |= mloc[nt][e] > m[nt][e] + lazy;
            }
        if (__any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float nmv[2], fv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float mx = mloc[nt][e];
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
                    const float mn = fmaxf(m[nt][e], mx);
                    const float f = m[nt][e] == -INFINITY ? 0.f : ex2((m[nt][e] - mn) * scl);
                    m[nt][e] = mn;
                    nmv[e] = mn == -INFINITY ? 0.f : -mn * scl;
                    fv[e] = f;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        o[mt][nt][e] *= f;
                        o[mt][nt][e + 2] *= f;
                    }
                }
                nm[nt] = f2(nmv[0], nmv[1]);
                lsum[nt] = mul2(lsum[nt], f2(fv[0], fv[1]));
            }
        }
        // p = 2^(s * scale - m * scale); masked scores give exactly 0.
        float p[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float t[4];
            unf2(fma2(f2(s[nt][0], s[nt][1]), scl2, nm[nt]), t[0], t[1]);
            unf2(fma2(f2(s[nt][2], s[nt][3]), scl2, nm[nt]), t[2], t[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) p[nt][i] = ex2(t[i]);
            lsum[nt] = add2(lsum[nt], add2(f2(p[nt][0], p[nt][1]), f2(p[nt][2], p[nt][3])));
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
        const f2_t vA[4] = {f2(vA01.x, vA01.x), f2(vA01.y, vA01.y), f2(vA23.x, vA23.x),
                            f2(vA23.y, vA23.y)};
        const f2_t vB[4] = {f2(vB01.x, vB01.x), f2(vB01.y, vB01.y), f2(vB23.x, vB23.x),
                            f2(vB23.y, vB23.y)};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t b0[NT], b1[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float x0, x1, y0, y1;
                unf2(mul2(f2(p[nt][0], p[nt][1]), vA[b]), x0, x1);
                unf2(mul2(f2(p[nt][2], p[nt][3]), vB[b]), y0, y1);
                b0[nt] = transpose8x8(pack_bf16(x0, x1));
                b1[nt] = transpose8x8(pack_bf16(y0, y1));
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

    // Row sums over the 8 position lanes; m is already uniform across them.  From here on m is
    // in base-2 units (m * scale), as the merge expects.
    float l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        unf2(lsum[nt], l[nt][0], l[nt][1]);
#pragma unroll
        for (int e = 0; e < 2; ++e) m[nt][e] = m[nt][e] * scl;
    }
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
    const int rows_here = min(kRowsPerGroup, P.rows - rg * kRowsPerGroup);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = 8 * nt + 2 * tig + e;
            if (row >= rows_here) continue;
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

    for (int idx = threadIdx.x; idx < rows_here * 32; idx += kThreads) {
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
    if (threadIdx.x < rows_here) {
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

// One warp per (row group, kv head, row): merges the splits' partials and writes o = O / l.  All
// loads of a round of 32 splits are issued before any is used (one L2 round trip per round).
__global__ void __launch_bounds__(128) kv_attention_merge_kernel(const KvaParams P) {
    griddep_launch_dependents();  // the next layer's split pass may become resident and wait
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
    const float4 *po = reinterpret_cast<const float4 *>(P.part_o) + row * (kD / 4) + lane;
    constexpr size_t kStride4 = (size_t)kRowsPerGroup * kD / 4;  // float4s per partial

    float2 ml[kMaxSplitRounds];
    float4 v[32];
#pragma unroll
    for (int k = 0; k < kMaxSplitRounds; ++k) {
        const int s = lane + 32 * k;
        ml[k] = s < P.splits ? P.part_ml[(base + s) * kRowsPerGroup + row] : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (i < P.splits) v[i] = po[(base + i) * kStride4];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxSplitRounds; ++k) M = fmaxf(M, ml[k].x);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    float wr[kMaxSplitRounds], S = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxSplitRounds; ++k) {
        wr[k] = ml[k].x == -INFINITY ? 0.f : ex2(ml[k].x - M);
        S += wr[k] * ml[k].y;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float w = __shfl_sync(0xFFFFFFFFu, wr[0], i);
        if (i < P.splits) {
            acc.x += w * v[i].x;
            acc.y += w * v[i].y;
            acc.z += w * v[i].z;
            acc.w += w * v[i].w;
        }
    }
#pragma unroll
    for (int k = 1; k < kMaxSplitRounds; ++k) {
        if (32 * k >= P.splits) break;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (32 * k + i < P.splits) v[i] = po[(base + 32 * k + i) * kStride4];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float w = __shfl_sync(0xFFFFFFFFu, wr[k], i);
            if (32 * k + i < P.splits) {
                acc.x += w * v[i].x;
                acc.y += w * v[i].y;
                acc.z += w * v[i].z;
                acc.w += w * v[i].w;
            }
        }
    }
    const float inv = 1.f / S;
    *reinterpret_cast<float4 *>(P.out + ((size_t)c * P.Hq + h) * kD + 4 * lane) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

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
    splits = std::min(splits, 32 * kMaxSplitRounds);
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
    e = launch(kv_attention_kernel<NT>, grid, dim3(kThreads), kSmemBytes, stream, true, P);
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

static int kv_attention_launch(const uint16_t *q, const float *k_new, const float *v_new, int ld,
                               const void *cache, int capacity, int n_q_heads, int n_kv_heads,
                               int n_past, int C, float scale, float *out, void *workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
    KvaGeom k;
    if (!q || !cache || !out || capacity <= 0 || !kva_geom(n_q_heads, n_kv_heads, n_past, C, k) ||
        (long long)n_past + C > capacity || !(scale > 0.f) || !(scale < INFINITY))
        return SVD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(cache) || !aligned16(out)) return SVD_ERR_INVALID_ARG;
    if (k_new && (!v_new || ld < n_kv_heads * kD)) return SVD_ERR_INVALID_ARG;
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
    P.k_new = P.v_new = nullptr;
    P.ld_new = 0;
    if (k_new) {
        if (k.n_rg == 1) {
            // One CTA reads each unit: the CTAs holding the window's positions append them.
            P.k_new = k_new;
            P.v_new = v_new;
            P.ld_new = ld;
        } else {
            // Several row groups read the same units: append first, in a kernel of its own.
            const long long warps = (long long)C * n_kv_heads;
            SVD_CUDA_TRY(launch(kv_append_kernel, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0,
                                stream, true, k_new, v_new, ld, C, n_kv_heads, n_past,
                                (unsigned char *)const_cast<void *>(cache), units_for(capacity)));
        }
    }
    const dim3 grid(k.splits, n_kv_heads, k.n_rg);
    cudaError_t e;
    switch (k.nt) {
        case 1: e = launch_kva<1>(P, grid, stream); break;
        case 2: e = launch_kva<2>(P, grid, stream); break;
        default: e = launch_kva<3>(P, grid, stream); break;
    }
    SVD_CUDA_TRY(e);
    return SVD_OK;
}

extern "C" int svd_kv_attention(const uint16_t *q, const void *cache, int capacity, int n_q_heads,
                                int n_kv_heads, int n_past, int C, float scale, float *out,
                                void *workspace, size_t workspace_bytes, svd_stream_t stream) {
    return kv_attention_launch(q, nullptr, nullptr, 0, cache, capacity, n_q_heads, n_kv_heads,
                               n_past, C, scale, out, workspace, workspace_bytes,
                               (cudaStream_t)stream);
}

extern "C" int svd_kv_attention_append(const uint16_t *q, const float *k, const float *v, int ld,
                                       void *cache, int capacity, int n_q_heads, int n_kv_heads,
                                       int n_past, int C, float scale, float *out,
                                       void *workspace, size_t workspace_bytes,
                                       svd_stream_t stream) {
    if (!k || !v) return SVD_ERR_INVALID_ARG;
    return kv_attention_launch(q, k, v, ld, cache, capacity, n_q_heads, n_kv_heads, n_past, C,
                               scale, out, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" int svd_kv_append(const float *k, const float *v, int ld, int C, int n_kv_heads,
                             int n_past, void *cache, int capacity, svd_stream_t stream) {
    if (!k || !v || !cache || C <= 0 || n_kv_heads <= 0 || n_past < 0 || capacity <= 0 ||
        (long long)n_past + C > capacity || ld < n_kv_heads * kD)
        return SVD_ERR_INVALID_ARG;
    if (!aligned16(cache)) return SVD_ERR_INVALID_ARG;
    const long long warps = (long long)C * n_kv_heads;
    SVD_CUDA_TRY(launch(kv_append_kernel, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0,
                        (cudaStream_t)stream, true, k, v, ld, C, n_kv_heads, n_past,
                        (unsigned char *)cache, units_for(capacity)));
    return SVD_OK;
}
