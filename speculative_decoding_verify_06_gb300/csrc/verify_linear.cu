// verify_linear.cu -- the weight-streaming dequant GEMM of the verify pass.
//
// "100 tokens per second from a 27B model on a 24 GB AMD card", section "How speculative
// decoding gets past a per-token wall": the target scores K drafts in one forward pass because
// every weight matrix is read once and applied to a K-wide batch of activations; the HN thread
// on speculative decoding makes the same point layer by layer.  So the kernel here streams each
// 4-bit matrix from HBM exactly once and multiplies it against the C = K+1 columns of a window:
//
//     Y[c][j] = sum_b s[j][b] * sum_{i in block b} (code[j][i] - 8) * X[c][i]
//
// Three kernels:
//  * vl_stream_kernel (NATIVE layout, C <= 16; C <= 32 on request) -- a persistent stream-K
//    kernel over (64-row block, 64-input chunk) units.  Every warp is a stream-K worker with
//    its own ring of bulk-copy slots (the codes and scales of two consecutive units, completing
//    on the slot's mbarrier) that its lane 0 refills as soon as the warp has read a slot, so no
//    warp waits for another while it computes.  Each warp dequantises nibbles straight into
//    bf16 A fragments with one lop3 and one bf16x2 subtract per pair (value 128 + c built from
//    the exponent pattern 0x4300, then minus 136 gives c - 8 exactly) and runs mma.sync
//    m16n8k16 (bf16 in, fp32 accumulate) against the activations as the B operand.  Every
//    32-input block gets a fresh accumulator that is scaled by its fp16 scale in fp32, so the
//    only rounding is fp32 accumulation.  A row block split between CTAs is finished by the
//    CTA holding its first unit, from tagged partials the others store without waiting
//    (summed in CTA order: deterministic).  A chain of matrices runs in one cooperative launch
//    with a grid barrier between matrices; the weights of the next matrix keep streaming
//    through it.
//  * vl_tc_kernel (NATIVE layout, 17 <= C <= 32; verify_linear_tc.cuh) -- the same stream-K
//    decomposition over 128-row units on the tcgen05 tensor cores: fp16 A operands with the
//    block scale folded in, staged in shared memory, fp32 accumulators in tensor memory.
//  * vl_simt_kernel (CANONICAL layout) -- the plain CUDA-core version: one warp per output
//    row, each lane one 32-input block at a time, fp32 FMAs, warp-shuffle reduction.
//
// The stream-K kernel also serves two extensions:
//  * Q4_K super-blocks (SVD_LAYOUT_Q4K_NATIVE, C <= 16): units of 64 rows x 256 inputs with
//    the super-blocks' headers; the codes enter the MMA as bf16 (128 + q), each sub-block's sum
//    is rescaled by its 6-bit scale in fp32, and the mins and the 128 offset leave through MMAs
//    against the sub-block sums of the activations (the layout is described below);
//  * the lm_head epilogue (single-op launches, C <= 8): per 64-row block and column the max,
//    the sum of exp((y - max) / T) and the argmax, which the sampler merges instead of scanning
//    the logits.
// The Q4_K bytes as stored run on a CUDA-core kernel of their own (kquant.cu).
#include <cooperative_groups.h>

#include <memory>
#include <mutex>

#include "svd_common.cuh"

namespace svd {

// ---- native layout geometry ------------------------------------------------------------
#ifndef SVD_TILES
#define SVD_TILES 4
#endif
constexpr int kTiles = SVD_TILES;                  // MMA tiles of 16 rows per unit
constexpr int kRowsPerBlock = 16 * kTiles;
constexpr int kChunk = 64;              // inputs per unit (2 scale blocks, 4 k16 steps)
constexpr int kUnitCodeBytes = 512 * kTiles;   // rows x 64 inputs x 4 bit
constexpr int kUnitScaleBytes = 64 * kTiles;   // rows x 2 blocks x fp16

struct NativeGeom {
    int64_t n_rb, n_kc, n_units;
};
static NativeGeom native_geom(int64_t in_f, int64_t out_f) {
    NativeGeom g;
    g.n_rb = (out_f + kRowsPerBlock - 1) / kRowsPerBlock;
    g.n_kc = (in_f + kChunk - 1) / kChunk;
    g.n_units = g.n_rb * g.n_kc;
    return g;
}

// Q4_K native layout (SVD_LAYOUT_Q4K_NATIVE): units of 64 rows x 256 inputs (one super-block
// column of a 64-row block), row-block-major like the native units.  A unit is 8192 bytes of
// codes -- four 64-input sub-chunks, each laid out exactly like a native unit's codes, the
// nibble holding the super-block's code q -- in the codes array, and the 64 rows' 16-byte
// super-block headers (fp16 d, fp16 dmin, 12 packed scale bytes) in row order in the header
// array: 144 bytes per 256 weights of a row, the format's own size.
constexpr int kKqIn = 256;                              // inputs per Q4_K unit
constexpr int kKqSub = kKqIn / kChunk;                  // 64-input sub-chunks per unit
constexpr int kKqUnitCodeBytes = kKqSub * kUnitCodeBytes;
constexpr int kKqUnitHdrBytes = kRowsPerBlock * 16;
constexpr int kKqBlockBytes = 144;                      // one super-block of the raw format
static NativeGeom kq_geom(int64_t in_f, int64_t out_f) {
    NativeGeom g;
    g.n_rb = (out_f + kRowsPerBlock - 1) / kRowsPerBlock;
    g.n_kc = in_f / kKqIn;
    g.n_units = g.n_rb * g.n_kc;
    return g;
}

// Inside a unit, lane l = 4*g + t of a warp owns, for tile r and k16 step s (s = 0..3), one
// 32-bit word whose nibble at bit 4p + 16h feeds A-fragment register p, half h:
//   row   = 16 r + g + 8 (p & 1)
//   input = 32 (s >> 1) + 8 t + 4 (s & 1) + 2 (p >> 1) + h        (relative to the chunk)
// Steps 0,1 cover scale block 0 and steps 2,3 block 1; lane l's inputs of a block are the 8
// consecutive ones at 32 b + 8 t, so its B fragments are one 16-byte load of X.
__host__ __device__ inline void native_word_coords(int s, int p, int h, int g, int t,
                                                   int *row_in_tile, int *input_in_chunk) {
    *row_in_tile = g + 8 * (p & 1);
    *input_in_chunk = 32 * (s >> 1) + 8 * t + 4 * (s & 1) + 2 * (p >> 1) + h;
}

__global__ void repack_codes_kernel(const uint8_t *__restrict__ src, uint32_t *__restrict__ dst,
                                    int64_t in_f, int64_t out_f, int64_t n_kc, int64_t n_words) {
    const int64_t wid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (wid >= n_words) return;
    const int s = (int)(wid & 3), lane = (int)((wid >> 2) & 31), r = (int)((wid >> 7) % kTiles);
    const int64_t unit = wid / (128 * kTiles), rb = unit / n_kc, kc = unit % n_kc;
    const int g = lane >> 2, t = lane & 3;
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            int rt, ic;
            native_word_coords(s, p, h, g, t, &rt, &ic);
            const int64_t row = rb * kRowsPerBlock + 16 * r + rt, i = kc * kChunk + ic;
            uint32_t nib = 8;  // code 8 is the value 0
            if (row < out_f && i < in_f) {
                const uint8_t byte = src[row * (in_f / 2) + i / 2];
                nib = (i & 1) ? (byte >> 4) : (byte & 15);
            }
            word |= nib << (4 * p + 16 * h);
        }
    dst[wid] = word;
}

// Scales of a unit: tile r, group g: 8 bytes = fp16 s(g, blk0), s(g, blk1), s(g+8, blk0),
// s(g+8, blk1), so lane 4g+t reads its four scales with one 8-byte load.
__global__ void repack_scales_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                     int64_t in_f, int64_t out_f, int64_t n_kc, int64_t n_halves) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_halves) return;
    const int q = (int)(idx & 3), g = (int)((idx >> 2) & 7), r = (int)((idx >> 5) % kTiles);
    const int64_t unit = idx / (32 * kTiles), rb = unit / n_kc, kc = unit % n_kc;
    const int64_t row = rb * kRowsPerBlock + 16 * r + g + 8 * (q >> 1), blk = 2 * kc + (q & 1);
    const int64_t nblk = in_f / 32;
    dst[idx] = (row < out_f && blk < nblk) ? src[row * nblk + blk] : (uint16_t)0;
}

__global__ void unpack_codes_kernel(const uint32_t *__restrict__ src, uint8_t *__restrict__ dst,
                                    int64_t in_f, int64_t out_f, int64_t n_kc) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t half_in = in_f / 2;
    if (idx >= out_f * half_in) return;
    const int64_t row = idx / half_in, byte = idx % half_in;
    uint8_t outb = 0;
    for (int h2 = 0; h2 < 2; ++h2) {
        const int64_t i = 2 * byte + h2;
        const int64_t rb = row / kRowsPerBlock, rr = row % kRowsPerBlock;
        const int r = (int)(rr / 16), rt = (int)(rr % 16), g = rt % 8, prow = rt / 8;
        const int64_t kc = i / kChunk;
        const int ii = (int)(i % kChunk), sblk = ii / 32, iw = ii % 32, t = iw / 8;
        const int slo = (iw % 8) / 4, e = iw % 4;
        const int s = 2 * sblk + slo, p = 2 * (e >> 1) + prow, h = e & 1;
        const int64_t wid = (((rb * n_kc + kc) * kTiles + r) * 32 + (4 * g + t)) * 4 + s;
        const uint32_t nib = (src[wid] >> (4 * p + 16 * h)) & 15u;
        outb |= (uint8_t)(nib << (4 * h2));
    }
    dst[idx] = outb;
}

__global__ void unpack_scales_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                     int64_t in_f, int64_t out_f, int64_t n_kc) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nblk = in_f / 32;
    if (idx >= out_f * nblk) return;
    const int64_t row = idx / nblk, blk = idx % nblk;
    const int64_t rb = row / kRowsPerBlock, rr = row % kRowsPerBlock;
    const int r = (int)(rr / 16), rt = (int)(rr % 16), g = rt % 8, prow = rt / 8;
    const int64_t kc = blk / 2;
    const int q = 2 * prow + (int)(blk & 1);
    dst[idx] = src[(((rb * n_kc + kc) * kTiles + r) * 8 + g) * 4 + q];
}

// Q4_K -> Q4_K native.  Word wid of the codes: unit wid / 2048, sub-chunk (wid >> 9) & 3, tile
// (wid >> 7) & 3, lane (wid >> 2) & 31, k16 step wid & 3; input 256 kc + 64 sub + (native
// input of the word's nibble), whose code sits in byte 16 + 32 (j / 2) + (i mod 32) of its
// super-block, low nibble for even sub-block j.  Padding rows get code 0 and a zero header
// (d = dmin = 0: every weight 0).
static_assert(kTiles == 4, "the Q4_K unit layout assumes four 16-row tiles per row block");
__global__ void kq_repack_codes_kernel(const uint8_t *__restrict__ src, uint32_t *__restrict__ dst,
                                       int64_t in_f, int64_t out_f, int64_t n_kc, int64_t n_words) {
    const int64_t wid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (wid >= n_words) return;
    const int s = (int)(wid & 3), lane = (int)((wid >> 2) & 31), r = (int)((wid >> 7) & 3);
    const int sub = (int)((wid >> 9) & 3);
    const int64_t unit = wid >> 11, rb = unit / n_kc, kc = unit % n_kc;
    const int g = lane >> 2, t = lane & 3;
    const int64_t row_bytes = in_f / kKqIn * kKqBlockBytes;
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            int rt, ic;
            native_word_coords(s, p, h, g, t, &rt, &ic);
            const int64_t row = rb * kRowsPerBlock + 16 * r + rt;
            const int i = kChunk * sub + ic;  // input within the super-block
            uint32_t nib = 0;
            if (row < out_f) {
                const int j = i >> 5;
                const uint8_t byte = src[row * row_bytes + kc * kKqBlockBytes + 16 + 32 * (j >> 1) + (i & 31)];
                nib = (j & 1) ? (byte >> 4) : (byte & 15);
            }
            word |= nib << (4 * p + 16 * h);
        }
    dst[wid] = word;
}

__global__ void kq_repack_hdr_kernel(const uint8_t *__restrict__ src, uint4 *__restrict__ dst,
                                     int64_t in_f, int64_t out_f, int64_t n_kc, int64_t n_rows) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_rows) return;
    const int64_t unit = idx / kRowsPerBlock, rb = unit / n_kc, kc = unit % n_kc;
    const int64_t row = rb * kRowsPerBlock + idx % kRowsPerBlock;
    const int64_t row_bytes = in_f / kKqIn * kKqBlockBytes;
    dst[idx] = row < out_f ? *reinterpret_cast<const uint4 *>(src + row * row_bytes + kc * kKqBlockBytes)
                           : make_uint4(0u, 0u, 0u, 0u);
}

// Q4_K native -> Q4_K: one thread per byte of the raw matrix.
__global__ void kq_unpack_kernel(const uint32_t *__restrict__ codes, const uint8_t *__restrict__ hdr,
                                 uint8_t *__restrict__ dst, int64_t in_f, int64_t out_f, int64_t n_kc) {
    const int64_t row_bytes = in_f / kKqIn * kKqBlockBytes;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= out_f * row_bytes) return;
    const int64_t row = idx / row_bytes, b = idx % row_bytes, kc = b / kKqBlockBytes;
    const int off = (int)(b % kKqBlockBytes);
    const int64_t rb = row / kRowsPerBlock, rr = row % kRowsPerBlock, unit = rb * n_kc + kc;
    if (off < 16) {
        dst[idx] = hdr[(unit * kRowsPerBlock + rr) * 16 + off];
        return;
    }
    const int r = (int)(rr / 16), rt = (int)(rr % 16), g = rt % 8, prow = rt / 8;
    uint8_t outb = 0;
    for (int hi = 0; hi < 2; ++hi) {
        const int j = 2 * ((off - 16) / 32) + hi, i = 32 * j + (off - 16) % 32;  // input in block
        const int sub = i / kChunk, ic = i % kChunk, sblk = ic / 32, iw = ic % 32, t = iw / 8;
        const int slo = (iw % 8) / 4, e = iw % 4;
        const int s = 2 * sblk + slo, p = 2 * (e >> 1) + prow, h = e & 1;
        const int64_t wid = ((((unit * kKqSub + sub) * kTiles + r) * 32) + (4 * g + t)) * 4 + s;
        outb |= (uint8_t)(((codes[wid] >> (4 * p + 16 * h)) & 15u) << (4 * hi));
    }
    dst[idx] = outb;
}

// ---- device building blocks -----------------------------------------------------------
// Loads from the ring by their 32-bit shared-memory address: ~1 % faster than the same loads
// through generic pointers in the stream kernel's one-n-tile, two-slot instances (measured; not
// in the others, nor in the Q4_K or tcgen05 unit bodies).
__device__ __forceinline__ uint4 lds_v4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}
__device__ __forceinline__ uint2 lds_v2(const void *p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
    return v;
}

// Activations read through L2 only: in a chain, op i+1 may read what op i wrote in the same
// kernel, so the non-coherent path must not be used there.
__device__ __forceinline__ uint4 ldg_cg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// Four bf16x2 A registers from one native word: (bits >> 4p) & 0x000F000F | 0x43004300 is the
// pair (128 + c_lo, 128 + c_hi) exactly; subtracting (136, 136) leaves (c - 8) exactly.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t a[4]) {
    const uint32_t magic = 0x43004300u, bias = 0x43084308u;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t v;
        const uint32_t sh = w >> (4 * p);
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(sh), "r"(0x000F000Fu), "r"(magic));
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(a[p]) : "r"(v), "r"(bias));
    }
}

// The pairs (128 + q_lo, 128 + q_hi) alone, without the subtraction: the Q4_K path takes the
// 128 x (sum of the activations) out afterwards, once per tile and unit.
__device__ __forceinline__ void dequant_word_b128(uint32_t w, uint32_t a[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t sh = w >> (4 * p);
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[p]) : "r"(sh), "r"(0x000F000Fu), "r"(0x43004300u));
    }
}

__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One verify-linear launch in the native layout (a link of a chain).
struct VlOp {
    const uint8_t *codes;
    const uint8_t *scales;
    const __nv_bfloat16 *X;
    float *Y;
    int64_t in_f, out_f;
    uint32_t n_kc, n_units;  // n_units * (CTAs + 1) < 2^32 (checked on the host)
};

template <int MAXOPS>
struct VlOps {
    int n;
    int C;
    // lm_head epilogue (single-op launches with C <= 8 only, else null): per 64-row block rb and
    // column c,
    // stats[rb * C + c] = (max of the block's outputs, sum of exp2((y - max) * stat_k) over
    // them, argmax as int bits, 0); NaN outputs and padding rows take no part.
    float4 *stats = nullptr;
    float stat_k = 0.f;  // log2(e) / T
    VlOp op[MAXOPS];
};

// (value, index) max with the lowest index on ties; index -1 is "none".
__device__ __forceinline__ void stat_argmax(float &bv, int &bi, float ov, int oi) {
    if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
    }
}

// ---- the tensor-core stream-K kernel ---------------------------------------------------
// Every warp is an independent stream-K worker.  The units of an op (64-row block x 64-input
// chunk, row-block-major) are split into W_op = min(G * NW, n_units) contiguous ranges, one
// per worker (warp w of CTA b is worker b * NW + w), so the shares differ by one unit at
// most.  Each warp streams its own units through its own ring of R slots in shared memory:
// its lane 0 issues the two bulk copies of a unit (codes, scales) R units ahead, completing
// on the slot's mbarrier, and refills a slot as soon as the warp has read it, so no warp
// waits for another while it computes.  A warp's unit sequence runs across op boundaries:
// the weights of op i+1 are in flight while op i finishes.
//
// A 64-row block the warp covers whole goes straight to Y.  The partial blocks at the two
// ends of its range are parked in shared memory, and when all warps of the CTA are done
// with the op they are added block by block in worker order.  A block whose first unit lies
// in this CTA is finished here (the CTA is its OWNER; if the block runs on into later CTAs,
// their partials are added in CTA order); otherwise the CTA stores its partial -- each value
// paired with a tag naming the launch and the op in one 64-bit store -- and moves on, and
// the owner waits for the tags.  No tickets, no fences and a fixed summation order: the
// result is deterministic.  Ops of a chain are separated by a barrier among all CTAs
// (cooperative launch); op 0 waits for the preceding kernel with griddepcontrol.wait before
// touching activations or the workspace.
constexpr int kPartialMax = 32 * kTiles * 4 * 4;  // entries of the largest partial (NT = 4)

template <int NT, int NW, int TW, int R, int U, int MAXOPS, int KQ>
struct VlCfg {
    static constexpr int kThreads = NW * 32;
    static constexpr int kWG = kTiles / TW;           // warps sharing a unit (one per TW tiles)
    static constexpr int kNG = NW / kWG;              // worker groups per CTA
    static constexpr int kAcc = kTiles * NT * 4;      // fp32 accumulators of a unit per lane
    static constexpr int kAccW = TW * NT * 4;         // ... of the tiles one warp works on
    static constexpr int kPartial = 32 * kAcc;        // entries of a row block's partial
    static constexpr int kPer = (kPartial + kThreads - 1) / kThreads;
    static constexpr int kUC = KQ ? kKqUnitCodeBytes : kUnitCodeBytes;  // codes of a unit
    static constexpr int kUS = KQ ? kKqUnitHdrBytes : kUnitScaleBytes;   // its scales / headers
    static constexpr int kSlotBytes = U * (kUC + kUS);  // codes of U units, then their scales
    static constexpr size_t kRing = (size_t)kNG * R * kSlotBytes;
    static constexpr size_t kPark = (size_t)NW * 2 * 32 * kAccW * sizeof(float);
    // Q4_K: each warp's decoded headers of its rows of the current unit (floats): sub-block
    // scales [TW][8 j][8 g][2]; per row the pairs (m[2t], m[2t+1]) then (sc[2t], sc[2t+1]) as
    // bf16x2 [TW * 16 rows][8]; (d, dmin) [TW * 16 rows]
    static constexpr int kKqScrW = TW * 288;
    static constexpr size_t kScratch = KQ ? (size_t)NW * kKqScrW * sizeof(float) : 0;
    static constexpr size_t kSmem = kRing + kPark + kScratch + (size_t)MAXOPS * sizeof(VlOp);
    static_assert(!KQ || NT <= 2, "Q4_K units take up to 16 columns");
    static_assert(kTiles % TW == 0 && NW % kWG == 0 && (kWG == 1 || kNG <= 15), "worker groups");
    static_assert(kPartial <= kPartialMax, "partial slot size");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

// Tagged partial entries: the value's bits in the low word, the tag in the high word.  The
// 64-bit store and load are single-copy atomic, so a matching tag guarantees the value.
__device__ __forceinline__ void st_tagged(unsigned long long *p, float v, uint32_t tag) {
    const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long *p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
// Failure detection.  Every spin-wait of the kernel is bounded: kPollLimit polls, or fewer when
// the workspace asks for a stall injection (a test hook, below).  A wait that runs out sets a
// bit of the workspace's status word (read by svd_verify_status) and the CTA's stop flag; from
// then on every wait of the CTA returns at once, a ring slot is refilled only if the wait for
// its previous copy succeeded, the kernel runs to its end without waiting (its output is
// undefined) and, before exiting, waits a bounded time for the copies it may have in flight.
// The stall injection makes the kernel issue no weight copy at all, as if the copy engine had
// stopped, so that a ring wait really runs out.
constexpr uint32_t kPollLimit = kDefaultPolls;
constexpr uint32_t kDrainLimit = 1u << 16;  // non-blocking polls: a few milliseconds at most
// Workspace words after the partial slots: [0] grid-barrier counter, [1] exit counter, both
// returned to zero by the last CTA out; [2] status bits; [3] stall injection (0 = none, else
// one more than the number of polls after which a wait gives up); [63] launch epoch, advanced
// by the last CTA out.
constexpr int kBarCount = 0, kBarExit = 1, kBarStatus = 2, kBarPoll = 3, kBarEpoch = 63;
constexpr unsigned kStCopy = 1u, kStPartial = 2u, kStOrder = 4u;  // status bits

// The CTA's wait state in shared memory: the poll limit, the stop flag, the status word.
struct WaitCtl {
    uint32_t limit;
    uint32_t stop;
    unsigned *status;
};
__device__ __forceinline__ bool wait_stopped(const WaitCtl *wc) {
    return *reinterpret_cast<const volatile uint32_t *>(&wc->stop) != 0u;
}
__device__ __forceinline__ void wait_fail(WaitCtl *wc, unsigned bit) {
    if (!wait_stopped(wc)) {
        *reinterpret_cast<volatile uint32_t *>(&wc->stop) = 1u;
        atomicOr(wc->status, bit);
    }
}

// Waits for an entry carrying `tag` and returns its value.
__device__ __forceinline__ float wait_tagged(const unsigned long long *p, uint32_t tag, WaitCtl *wc) {
    unsigned long long w = ld_tagged(p);
    for (uint32_t it = 0; (uint32_t)(w >> 32) != tag; ++it) {
        if (it >= wc->limit || wait_stopped(wc)) {
            wait_fail(wc, kStPartial);
            break;
        }
        if (it > 64) __nanosleep(64);
        w = ld_tagged(p);
    }
    return __uint_as_float((uint32_t)w);
}

// The gi-th barrier of a launch among all G CTAs: one release-add per CTA (after a CTA
// barrier, so that it carries every warp's writes) on a counter in the workspace, then
// acquire polling until the counter reaches gi * G.
__device__ __forceinline__ void grid_barrier(unsigned *count, unsigned target, WaitCtl *wc) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
    for (uint32_t it = 0;; ++it) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
        if (v >= target) return;
        if (it >= wc->limit || wait_stopped(wc)) {
            wait_fail(wc, kStOrder);
            return;
        }
        if (it > 512) __nanosleep(32);
    }
}
// Waits for phase `parity` of a ring slot's barrier with try_wait (which may suspend the thread
// until the phase completes); every 256 polls it checks the stop flag and the limit.  Returns
// whether the phase completed.
__device__ __forceinline__ bool slot_wait(uint32_t mbar, uint32_t parity, WaitCtl *wc) {
    for (uint32_t it = 0;; ++it) {
        if (mbar_poll(mbar, parity, true)) return true;
        if ((it & 255u) == 255u) {
            if (wait_stopped(wc)) return false;
            if (it >= wc->limit) break;
        }
    }
    wait_fail(wc, kStCopy);
    return false;
}
__device__ __forceinline__ unsigned atom_add_acqrel_gpu(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Partial tags: (e24 << 8) | op, where e24 = 1 + launch epoch mod (2^24 - 1) is never 0, so a
// zero-filled slot never matches; when e24 comes back to 1 the last CTA out of the launch
// before clears every partial slot, so a tag left from an earlier cycle never matches either.
__host__ __device__ inline uint32_t partial_epoch24(uint32_t epoch) { return epoch % 0xFFFFFFu + 1u; }

#ifndef SVD_PROBE
#define SVD_PROBE(gi, what)  // timing hook for instrumented builds; nothing by default
#endif

template <int NT, int NW, int TW, int R, int U, int MAXOPS, int KQ>
__global__ void __launch_bounds__(NW * 32, 1)
vl_stream_kernel(const __grid_constant__ VlOps<MAXOPS> P, unsigned long long *__restrict__ part,
                 uint32_t part_entries, unsigned *__restrict__ gbar) {
    using Cfg = VlCfg<NT, NW, TW, R, U, MAXOPS, KQ>;
    constexpr int kSlotBytes = Cfg::kSlotBytes, kWG = Cfg::kWG, kNG = Cfg::kNG;
    constexpr int kUC = Cfg::kUC, kUS = Cfg::kUS;
    constexpr int kAcc = Cfg::kAcc, kAccW = Cfg::kAccW, kPartial = Cfg::kPartial, kPer = Cfg::kPer;
    constexpr int kThreads = Cfg::kThreads;
    constexpr int kParkW = 32 * kAccW;  // floats of one parked partial
    // With few columns the next unit's activations are loaded while this unit computes; with
    // many the registers go to the accumulators and each unit loads its own.
    constexpr bool kPrefetchX = NT <= 2;
    constexpr uint32_t kNone = 0xFFFFFFFFu;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_full[kNG * R];
    __shared__ uint32_t s_park_rb[NW * 2];    // row block of a parked partial, kNone if none
    __shared__ uint32_t s_park_head[NW * 2];  // 1 if that partial starts at its block's start
    __shared__ uint32_t s_epoch, s_last;
    __shared__ WaitCtl s_wc;
    __shared__ uint32_t s_own[2 * NW], s_nown;  // lm_head epilogue: blocks finished from partials
    float *park = reinterpret_cast<float *>(smem + Cfg::kRing);
    // The op descriptors live in shared memory: read from the parameter space with a
    // run-time index they would go through the small constant cache on every access.
    VlOp *ops = reinterpret_cast<VlOp *>(smem + Cfg::kRing + Cfg::kPark + Cfg::kScratch);
    const int n_ops = P.n;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *const kq_scr = reinterpret_cast<float *>(smem + Cfg::kRing + Cfg::kPark) + warp * Cfg::kKqScrW;
    const int grp = warp / kWG, sub = warp % kWG;  // worker group, and this warp's tiles in it
    const uint32_t G = gridDim.x, b = blockIdx.x;
    const uint32_t Wtot = G * kNG, gw = b * kNG + grp;
    const uint32_t full0 = smem_u32(&s_full[grp * R]);
    uint8_t *const ring = smem + (size_t)grp * R * kSlotBytes;
    const uint32_t ring0 = smem_u32(ring);

    // This worker's unit range of an op: [lo, hi), empty when the op has fewer units than
    // there are workers and this one is not needed.
    auto range = [&](const VlOp &o, uint32_t *lo, uint32_t *hi) {
        const uint32_t Wop = min(Wtot, o.n_units);
        if (gw < Wop) {
            *lo = gw * o.n_units / Wop;
            *hi = (gw + 1) * o.n_units / Wop;
        } else {
            *lo = *hi = 0u;
        }
    };
    // The CTA whose workers hold unit n of an op.
    auto cta_of = [&](const VlOp &o, uint32_t n) {
        const uint32_t Wop = min(Wtot, o.n_units);
        return (((n + 1) * Wop - 1) / o.n_units) / kNG;
    };
    // The warps of a group have all read a slot.
    auto group_sync = [&]() {
        if constexpr (kWG == 1) {
            __syncwarp();
        } else {
            asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(kWG * 32) : "memory");
        }
    };

    {
        static_assert(sizeof(VlOp) % 8 == 0, "op descriptor copied in 8-byte words");
        const uint64_t *src = reinterpret_cast<const uint64_t *>(&P.op[0]);
        uint64_t *dst = reinterpret_cast<uint64_t *>(ops);
        for (int i = threadIdx.x; i < n_ops * (int)(sizeof(VlOp) / 8); i += kThreads) dst[i] = src[i];
    }
    if (sub == 0 && lane == 0) {
        for (int i = 0; i < R; ++i) mbar_init(full0 + 8 * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x == 0) s_wc.stop = 0u;
    __syncthreads();

    // Issue cursor of this group (uniform across its warps; the first warp's lane 0 issues):
    // the next unit to load is unit c_u of op c_op, c_hi ends that op's range, c_codes /
    // c_scales point at that unit's bytes; c_issued counts filled slots.  A slot takes the
    // next U units of the range (fewer at its end; never units of two ops).
    int c_op = -1;
    uint32_t c_u = 0, c_hi = 0, c_issued = 0;

    const uint8_t *c_codes = nullptr, *c_scales = nullptr;
    auto issue = [&]() {
        while (c_u >= c_hi) {
            if (++c_op >= n_ops) return;
            range(ops[c_op], &c_u, &c_hi);
            c_codes = ops[c_op].codes + (size_t)c_u * kUC;
            c_scales = ops[c_op].scales + (size_t)c_u * kUS;
        }
        const uint32_t slot = c_issued % R, n = min((uint32_t)U, c_hi - c_u);
        if (sub == 0 && lane == 0) {
            const uint32_t bar = full0 + 8 * slot, dst = ring0 + slot * kSlotBytes;
            mbar_expect_tx(bar, n * (kUC + kUS));
            bulk_g2s(dst, c_codes, n * kUC, bar);
            bulk_g2s(dst + U * kUC, c_scales, n * kUS, bar);
        }
        c_u += n;
        ++c_issued;
        c_codes += n * kUC;
        c_scales += n * kUS;
    };
    // The stall injection (workspace word kBarPoll, written only by the test hook, never by an
    // earlier kernel of the stream, so it may be read before the dependency wait): no copy.
    if (*reinterpret_cast<volatile unsigned *>(gbar + kBarPoll) != 0u) c_op = n_ops;
    // weights never depend on earlier kernels: start streaming before waiting for them
    for (int i = 0; i < R; ++i) issue();

    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        s_epoch = *reinterpret_cast<volatile unsigned *>(gbar + kBarEpoch);
        const unsigned lim = *reinterpret_cast<volatile unsigned *>(gbar + kBarPoll);
        s_wc.limit = lim ? lim - 1u : kPollLimit;
        s_wc.status = gbar + kBarStatus;
    }
    __syncthreads();
    const uint32_t epoch = s_epoch;

    const int g4 = lane >> 2, t4 = lane & 3;
    const int C = P.C;
    float acc[TW][NT][4];
#pragma unroll
    for (int r = 0; r < TW; ++r)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[r][nt][q] = 0.f;

    uint32_t c_used = 0;  // slots this group has consumed (its ring position)
    for (int gi = 0; gi < n_ops; ++gi) {
        const VlOp &o = ops[gi];
        if (gi > 0) {
            __syncthreads();
            if (threadIdx.x == 0) grid_barrier(gbar + kBarCount, (unsigned)gi * G, &s_wc);
            __syncthreads();
        }
        SVD_PROBE(gi, 0);
        const uint32_t n_kc = o.n_kc;
        const int64_t in_f = o.in_f, out_f = o.out_f;
        const uint32_t tag = (partial_epoch24(epoch) << 8) | (uint32_t)(gi & 255);
        // (row, column) of accumulator q of n-tile nt of tile rt (0..kTiles-1) of lane lsrc
        auto coords = [&](int lsrc, int rt, int nt, int q, uint32_t rb, int64_t *row, int *col) {
            *row = (int64_t)rb * kRowsPerBlock + 16 * rt + (lsrc >> 2) + ((q >> 1) ? 8 : 0);
            *col = nt * 8 + (lsrc & 3) * 2 + (q & 1);
        };
        // Parked partial k (0: the range's first segment, 1: its last) of warp `sub` of group
        // `grp` goes to place (2 grp + k) kWG + sub, so that places in order hold nondecreasing
        // row blocks (worker order) with the warps of a group side by side.
        auto park_at = [&](int k) { return (2 * grp + k) * kWG + sub; };
        if (lane < 2) {
            s_park_rb[park_at(lane)] = kNone;
            s_park_head[park_at(lane)] = 0u;
        }
        if (threadIdx.x == 0) s_nown = 0u;

        uint32_t lo, hi;
        range(o, &lo, &hi);
        if (lo < hi) {
            const __nv_bfloat16 *xrow[NT];
            bool xok[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = nt * 8 + g4;
                xok[nt] = col < C;
                xrow[nt] = o.X + (int64_t)(xok[nt] ? col : 0) * in_f + t4 * 8;
            }
            const bool tail32 = (in_f & 63) != 0;  // the last chunk holds one 32-input block
            auto load_x = [&](uint32_t kc, uint4 (&xr)[NT][2]) {
                const bool lastc = tail32 && (kc == n_kc - 1);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const __nv_bfloat16 *src = xrow[nt] + (size_t)kc * kChunk;
                    if constexpr (MAXOPS > 1) {
                        xr[nt][0] = xok[nt] ? ldg_cg_v4(src) : make_uint4(0u, 0u, 0u, 0u);
                        xr[nt][1] = (xok[nt] && !lastc) ? ldg_cg_v4(src + 32) : make_uint4(0u, 0u, 0u, 0u);
                    } else {
                        xr[nt][0] = xok[nt] ? ldg_nc_v4(src) : make_uint4(0u, 0u, 0u, 0u);
                        xr[nt][1] = (xok[nt] && !lastc) ? ldg_nc_v4(src + 32) : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            };

            uint32_t rb = lo / n_kc, kc = lo - rb * n_kc, seg_lo = lo;
            uint4 xr[NT][2], xr2[NT][2];  // the next unit's (Q4_K: the next two sub-chunks') activations
            if constexpr (kPrefetchX) load_x(KQ ? kKqSub * kc : kc, xr);
            if constexpr (kPrefetchX && KQ && NT == 1) load_x(kKqSub * kc + 1, xr2);
            for (uint32_t u = lo; u < hi; ++u) {
                const uint32_t slot = c_used % R, in_slot = (u - lo) % U;
                const uint32_t kn = (kc + 1 == n_kc) ? 0u : kc + 1;
                if constexpr (KQ) {
                    // ---- a Q4_K unit: 64 rows x 256 inputs; this warp's TW tiles of it
                    if (in_slot == 0u && !slot_wait(full0 + 8 * slot, (c_used / R) & 1u, &s_wc)) c_op = n_ops;
                    const uint8_t *cbase = ring + slot * kSlotBytes + in_slot * kUC + lane * 16;
                    const uint8_t *hbase = ring + slot * kSlotBytes + U * kUC + in_slot * kUS;
                    float *sc_s = kq_scr;
                    uint32_t *m_s = reinterpret_cast<uint32_t *>(kq_scr + TW * 128);
                    float2 *d_s = reinterpret_cast<float2 *>(kq_scr + TW * 256);
                    // decode the headers of this warp's rows: lane l takes local rows l, l + 32, ...
                    for (int lr = lane; lr < TW * 16; lr += 32) {
                        const uint4 hd = *reinterpret_cast<const uint4 *>(hbase + (sub * TW * 16 + lr) * 16);
                        uint32_t scv[8], mv[8];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            scv[j] = (hd.y >> (8 * j)) & 63u;
                            mv[j] = (hd.z >> (8 * j)) & 63u;
                            const uint32_t lo4 = (hd.w >> (8 * j)) & 255u;
                            scv[j + 4] = (lo4 & 15u) | (((hd.y >> (8 * j + 6)) & 3u) << 4);
                            mv[j + 4] = (lo4 >> 4) | (((hd.z >> (8 * j + 6)) & 3u) << 4);
                        }
                        const int r = lr >> 4, rt = lr & 15, g = rt & 7, hh = rt >> 3;
#pragma unroll
                        for (int j = 0; j < 8; ++j) sc_s[((r * 8 + j) * 8 + g) * 2 + hh] = (float)scv[j];
                        uint32_t mw[8];  // (m[2t], m[2t+1]), (sc[2t], sc[2t+1]) as bf16 pairs, exact (< 64)
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            mw[t] = (__float_as_uint((float)mv[2 * t]) >> 16) |
                                    (__float_as_uint((float)mv[2 * t + 1]) & 0xFFFF0000u);
                            mw[4 + t] = (__float_as_uint((float)scv[2 * t]) >> 16) |
                                        (__float_as_uint((float)scv[2 * t + 1]) & 0xFFFF0000u);
                        }
                        *reinterpret_cast<uint4 *>(m_s + lr * 8) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
                        *reinterpret_cast<uint4 *>(m_s + lr * 8 + 4) = make_uint4(mw[4], mw[5], mw[6], mw[7]);
                        d_s[lr] = make_float2(__half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu))),
                                              __half2float(__ushort_as_half((unsigned short)(hd.x >> 16))));
                    }
                    __syncwarp();
                    // per tile T = sum_j sc_j (sum_{i in j} (128 + q_i) x_i); and the sub-block sums
                    // of x as an MMA of X (rows = columns) against an indicator: D[col][j] = sum_{i in j} x
                    float T[TW][NT][4], xsd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int r = 0; r < TW; ++r)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int q = 0; q < 4; ++q) T[r][nt][q] = 0.f;
#pragma unroll
                    for (int s4 = 0; s4 < kKqSub; ++s4) {
                        uint4 xq[NT][2];
                        if constexpr (kPrefetchX && NT == 1) {
                            // two sub-chunks ahead (into the next unit of the range at the end)
                            xq[0][0] = xr[0][0];
                            xq[0][1] = xr[0][1];
                            xr[0][0] = xr2[0][0];
                            xr[0][1] = xr2[0][1];
                            if (s4 + 2 < kKqSub) load_x(kKqSub * kc + s4 + 2, xr2);
                            else if (u + 1 < hi) load_x(kKqSub * kn + s4 + 2 - kKqSub, xr2);
                        } else if constexpr (kPrefetchX) {
                            // two n-tiles: one sub-chunk ahead (the registers go to the accumulators)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                xq[nt][0] = xr[nt][0];
                                xq[nt][1] = xr[nt][1];
                            }
                            if (s4 + 1 < kKqSub) load_x(kKqSub * kc + s4 + 1, xr);
                            else if (u + 1 < hi) load_x(kKqSub * kn, xr);
                        } else {
                            load_x(kKqSub * kc + s4, xq);
                        }
#pragma unroll
                        for (int r = 0; r < TW; ++r) {
                            const uint4 cw = *reinterpret_cast<const uint4 *>(cbase + s4 * kUnitCodeBytes + (sub * TW + r) * 512);
#pragma unroll
                            for (int blk = 0; blk < 2; ++blk) {
                                uint32_t a0[4], a1[4];
                                dequant_word_b128(blk ? cw.z : cw.x, a0);
                                dequant_word_b128(blk ? cw.w : cw.y, a1);
                                const float2 sc2 = *reinterpret_cast<const float2 *>(sc_s + ((r * 8 + 2 * s4 + blk) * 8 + g4) * 2);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    float d4[4] = {0.f, 0.f, 0.f, 0.f};
                                    mma_bf16_16816(d4, a0, xq[nt][blk].x, xq[nt][blk].y);
                                    mma_bf16_16816(d4, a1, xq[nt][blk].z, xq[nt][blk].w);
                                    T[r][nt][0] = fmaf(sc2.x, d4[0], T[r][nt][0]);
                                    T[r][nt][1] = fmaf(sc2.x, d4[1], T[r][nt][1]);
                                    T[r][nt][2] = fmaf(sc2.y, d4[2], T[r][nt][2]);
                                    T[r][nt][3] = fmaf(sc2.y, d4[3], T[r][nt][3]);
                                }
                            }
                        }
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk) {
                            const uint32_t ind = (g4 == 2 * s4 + blk) ? 0x3F803F80u : 0u;  // bf16 (1, 1)
                            // A rows 0-7: columns 0-7; rows 8-15: columns 8-15 (the second n-tile)
                            const uint32_t ax0[4] = {xq[0][blk].x, NT > 1 ? xq[NT - 1][blk].x : 0u, xq[0][blk].y,
                                                     NT > 1 ? xq[NT - 1][blk].y : 0u};
                            const uint32_t ax1[4] = {xq[0][blk].z, NT > 1 ? xq[NT - 1][blk].z : 0u, xq[0][blk].w,
                                                     NT > 1 ? xq[NT - 1][blk].w : 0u};
                            mma_bf16_16816(xsd, ax0, ind, ind);
                            mma_bf16_16816(xsd, ax1, ind, ind);
                        }
                    }
                    // lane (g, t) holds the sums of sub-blocks 2t, 2t+1 for column g (and g + 8):
                    // exactly the B fragment of the products sum_j m_j xs_j (the mins) and
                    // sum_j sc_j xs_j (the 128 offset of the codes), with xs split into bf16 hi + lo
                    uint32_t bh[NT], bl[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(xsd[2 * nt], xsd[2 * nt + 1]);
                        const float2 hif = __bfloat1622float2(hi2);
                        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(xsd[2 * nt] - hif.x, xsd[2 * nt + 1] - hif.y);
                        bh[nt] = *reinterpret_cast<const uint32_t *>(&hi2);
                        bl[nt] = *reinterpret_cast<const uint32_t *>(&lo2);
                    }
#pragma unroll
                    for (int r = 0; r < TW; ++r) {
                        const uint32_t *p0 = m_s + (16 * r + g4) * 8 + t4, *p1 = m_s + (16 * r + g4 + 8) * 8 + t4;
                        const uint32_t am[4] = {p0[0], p1[0], p0[0], p1[0]};
                        const uint32_t as[4] = {p0[4], p1[4], p0[4], p1[4]};
                        const float2 e0 = d_s[16 * r + g4], e1 = d_s[16 * r + g4 + 8];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            float dm[4] = {0.f, 0.f, 0.f, 0.f}, ds[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_bf16_16816(dm, am, bh[nt], bl[nt]);
                            mma_bf16_16816(ds, as, bh[nt], bl[nt]);
                            acc[r][nt][0] = fmaf(e0.x, fmaf(-128.f, ds[0], T[r][nt][0]), fmaf(-e0.y, dm[0], acc[r][nt][0]));
                            acc[r][nt][1] = fmaf(e0.x, fmaf(-128.f, ds[1], T[r][nt][1]), fmaf(-e0.y, dm[1], acc[r][nt][1]));
                            acc[r][nt][2] = fmaf(e1.x, fmaf(-128.f, ds[2], T[r][nt][2]), fmaf(-e1.y, dm[2], acc[r][nt][2]));
                            acc[r][nt][3] = fmaf(e1.x, fmaf(-128.f, ds[3], T[r][nt][3]), fmaf(-e1.y, dm[3], acc[r][nt][3]));
                        }
                    }
                    __syncwarp();  // the scratch is rewritten for the next unit
                } else {
                uint4 xc[NT][2];
                if constexpr (kPrefetchX) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        xc[nt][0] = xr[nt][0];
                        xc[nt][1] = xr[nt][1];
                    }
                    if (u + 1 < hi) load_x(kn, xr);
                } else {
                    load_x(kc, xc);
                }
                // a wait that gave up ends this warp's copies: its slot may still be filling, so it
                // is never refilled (the issue cursor is exhausted)
                if (in_slot == 0u && !slot_wait(full0 + 8 * slot, (c_used / R) & 1u, &s_wc)) c_op = n_ops;
                const uint8_t *cbase = ring + slot * kSlotBytes + in_slot * kUnitCodeBytes;
                const uint8_t *sbase = ring + slot * kSlotBytes + U * kUnitCodeBytes + in_slot * kUnitScaleBytes;
#pragma unroll
                for (int r = 0; r < TW; ++r) {
                    const int rt = sub * TW + r;
                    uint4 cw;
                    uint2 scw;
                    if constexpr (NT == 1 && R == 2) {  // (the other instances measure or spill worse)
                        cw = lds_v4(cbase + rt * 512 + lane * 16);
                        scw = lds_v2(sbase + rt * 64 + g4 * 8);
                    } else {
                        cw = *reinterpret_cast<const uint4 *>(cbase + rt * 512 + lane * 16);
                        scw = *reinterpret_cast<const uint2 *>(sbase + rt * 64 + g4 * 8);
                    }
                    const float2 s_lo = __half22float2(*reinterpret_cast<const __half2 *>(&scw.x));
                    const float2 s_hi = __half22float2(*reinterpret_cast<const __half2 *>(&scw.y));
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        uint32_t a0[4], a1[4];
                        dequant_word(blk ? cw.z : cw.x, a0);
                        dequant_word(blk ? cw.w : cw.y, a1);
                        const float sg = blk ? s_lo.y : s_lo.x, sh = blk ? s_hi.y : s_hi.x;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_bf16_16816(d, a0, xc[nt][blk].x, xc[nt][blk].y);
                            mma_bf16_16816(d, a1, xc[nt][blk].z, xc[nt][blk].w);
                            acc[r][nt][0] = fmaf(sg, d[0], acc[r][nt][0]);
                            acc[r][nt][1] = fmaf(sg, d[1], acc[r][nt][1]);
                            acc[r][nt][2] = fmaf(sh, d[2], acc[r][nt][2]);
                            acc[r][nt][3] = fmaf(sh, d[3], acc[r][nt][3]);
                        }
                    }
                }
                }  // native unit
                // Once the group has read the slot, refill it with the units R slots further
                // on.  Every value a warp loaded from the slot has been consumed by the
                // instructions above (issued in order), so the bulk copy cannot overwrite a
                // pending read.
                if (in_slot == U - 1u || u + 1 == hi) {
                    group_sync();
                    issue();
                    ++c_used;
                }

                // end of a segment (a row block's end, or the range's): a whole block goes
                // to Y, a partial one is parked
                const bool rb_end = kc + 1 == n_kc;
                if (rb_end || u + 1 == hi) {
                    const bool head = seg_lo == rb * n_kc;
                    if (head && rb_end) {
#pragma unroll
                        for (int r = 0; r < TW; ++r)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    int64_t row;
                                    int col;
                                    coords(lane, sub * TW + r, nt, q, rb, &row, &col);
                                    if (row < out_f && col < C) o.Y[(int64_t)col * out_f + row] = acc[r][nt][q];
                                }
                        if constexpr (NT == 1 && TW == kTiles && MAXOPS == 1) {
                            // the lm_head epilogue from the registers: lane (g, t) holds rows
                            // 16 r + g (+ 8) of every tile for columns 2 t and 2 t + 1
                            if (P.stats != nullptr) {
#pragma unroll
                                for (int qc = 0; qc < 2; ++qc) {
                                    float bv = 0.f;
                                    int bi = -1;
#pragma unroll
                                    for (int r = 0; r < TW; ++r)
#pragma unroll
                                        for (int hh = 0; hh < 2; ++hh) {
                                            const int64_t row = (int64_t)rb * kRowsPerBlock + 16 * r + g4 + 8 * hh;
                                            const float v = acc[r][0][qc + 2 * hh];
                                            if (row < out_f && v == v) stat_argmax(bv, bi, v, (int)row);
                                        }
#pragma unroll
                                    for (int m = 4; m < 32; m <<= 1)
                                        stat_argmax(bv, bi, __shfl_xor_sync(0xFFFFFFFFu, bv, m), __shfl_xor_sync(0xFFFFFFFFu, bi, m));
                                    float sum = 0.f;
#pragma unroll
                                    for (int r = 0; r < TW; ++r)
#pragma unroll
                                        for (int hh = 0; hh < 2; ++hh) {
                                            const int64_t row = (int64_t)rb * kRowsPerBlock + 16 * r + g4 + 8 * hh;
                                            const float v = acc[r][0][qc + 2 * hh];
                                            if (row < out_f && v == v) sum += exp2f((v - bv) * P.stat_k);
                                        }
#pragma unroll
                                    for (int m = 4; m < 32; m <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, m);
                                    const int col = 2 * t4 + qc;
                                    if (g4 == 0 && col < C)
                                        P.stats[(size_t)rb * C + col] =
                                            make_float4(bi >= 0 ? bv : -INFINITY, sum, __int_as_float(bi), 0.f);
                                }
                            }
                        }
                    } else {
                        const int k = seg_lo == lo ? 0 : 1;
                        float4 *dst = reinterpret_cast<float4 *>(park + park_at(k) * kParkW + lane * kAccW);
#pragma unroll
                        for (int r = 0; r < TW; ++r)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                dst[r * NT + nt] = make_float4(acc[r][nt][0], acc[r][nt][1],
                                                               acc[r][nt][2], acc[r][nt][3]);
                        if (lane == 0) {
                            s_park_rb[park_at(k)] = rb;
                            s_park_head[park_at(k)] = head ? 1u : 0u;
                        }
                    }
#pragma unroll
                    for (int r = 0; r < TW; ++r)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[r][nt][q] = 0.f;
                    seg_lo = u + 1;
                    rb += rb_end ? 1u : 0u;
                }
                kc = kn;
            }
        }
        SVD_PROBE(gi, 1);

        // ---- all warps are done with the op: add the parked partials block by block, in
        // worker order (first segment before last within a group).  Parked partial i (i < 2 NW) is
        // looked at by lane i of every warp; runs of equal row blocks are found with ballots.
        // Entry e of a block's partial is accumulator e % kAcc of lane e / kAcc of the whole
        // unit; a parked partial holds the tiles of the warp that parked it.
        __syncthreads();
        {
            static_assert(2 * NW <= 32, "one lane per parked partial");
            const uint32_t my_rb = lane < 2 * NW ? s_park_rb[lane] : kNone;
            const bool my_head = lane < 2 * NW && s_park_head[lane] != 0u;
            const uint32_t valid = __ballot_sync(0xFFFFFFFFu, my_rb != kNone);
            // previous parked partial in worker order, and whether this one starts a run
            const uint32_t below = valid & ((1u << lane) - 1u);
            const int prev = below ? 31 - __clz(below) : -1;
            const uint32_t prev_rb = __shfl_sync(0xFFFFFFFFu, my_rb, prev < 0 ? lane : prev);
            const uint32_t starts =
                __ballot_sync(0xFFFFFFFFu, my_rb != kNone && (prev < 0 || prev_rb != my_rb));
            // parked partials of the warps working on tile group h: places congruent to h
            uint32_t sub_mask[kWG];
#pragma unroll
            for (int h = 0; h < kWG; ++h) {
                uint32_t m = 0u;
                for (int i = h; i < 2 * NW; i += kWG) m |= 1u << i;
                sub_mask[h] = m;
            }
            for (uint32_t rest = starts; rest != 0u;) {
                const int p = __ffs(rest) - 1;
                rest &= rest - 1u;
                const uint32_t next = rest ? (uint32_t)(__ffs(rest) - 1) : 32u;
                const uint32_t members = valid & ~((1u << p) - 1u) & (next < 32u ? (1u << next) - 1u : 0xFFFFFFFFu);
                const uint32_t rb = __shfl_sync(0xFFFFFFFFu, my_rb, p);
                const bool owner = __shfl_sync(0xFFFFFFFFu, my_head ? 1 : 0, p) != 0;
                const uint32_t b_last = owner ? cta_of(o, (rb + 1) * n_kc - 1) : b;
#pragma unroll
                for (int m = 0; m < kPer; ++m) {
                    const int e = threadIdx.x + m * kThreads;
                    if (e >= kPartial) break;
                    const int lsrc = e / kAcc, idx = e % kAcc, q = idx & 3, rn = idx >> 2;
                    const int rt = rn / NT, nt = rn % NT, h = rt / TW;
                    int64_t row;
                    int col;
                    coords(lsrc, rt, nt, q, rb, &row, &col);
                    if (row >= out_f || col >= C) continue;
                    const int off = lsrc * kAccW + ((rt - h * TW) * NT + nt) * 4 + q;
                    float v = 0.f;
                    for (uint32_t mm = members & sub_mask[h]; mm != 0u; mm &= mm - 1u)
                        v += park[(__ffs(mm) - 1) * kParkW + off];
                    if (owner) {
                        // the other CTAs' partials, in CTA order, four loads in flight at a time;
                        // the missing ones polled together where the registers allow it (one
                        // n-tile, two ring slots per worker, symmetric units), else one at a time
                        if constexpr (NT == 1 && R == 2 && !KQ) {
                            for (uint32_t bb = b + 1; bb <= b_last; bb += 4) {
                                unsigned long long w4[4];
                                uint32_t pend = 0u;
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    w4[i] = 0ull;
                                    if (bb + i <= b_last) {
                                        w4[i] = ld_tagged(part + (size_t)(bb + i) * kPartialMax + e);
                                        pend |= 1u << i;
                                    }
                                }
                                for (uint32_t it = 0;; ++it) {
#pragma unroll
                                    for (int i = 0; i < 4; ++i)
                                        if ((uint32_t)(w4[i] >> 32) == tag) pend &= ~(1u << i);
                                    if (pend == 0u) break;
                                    if (it >= s_wc.limit || wait_stopped(&s_wc)) {
                                        wait_fail(&s_wc, kStPartial);
                                        break;
                                    }
                                    if (it > 64) __nanosleep(64);
#pragma unroll
                                    for (int i = 0; i < 4; ++i)
                                        if (pend & (1u << i)) w4[i] = ld_tagged(part + (size_t)(bb + i) * kPartialMax + e);
                                }
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (bb + i <= b_last) v += __uint_as_float((uint32_t)w4[i]);
                            }
                        } else {
                            for (uint32_t bb = b + 1; bb <= b_last; bb += 4) {
                                unsigned long long w4[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (bb + i <= b_last) w4[i] = ld_tagged(part + (size_t)(bb + i) * kPartialMax + e);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    if (bb + i > b_last) break;
                                    const float x = (uint32_t)(w4[i] >> 32) == tag
                                                        ? __uint_as_float((uint32_t)w4[i])
                                                        : wait_tagged(part + (size_t)(bb + i) * kPartialMax + e, tag, &s_wc);
                                    v += x;
                                }
                            }
                        }
                        o.Y[(int64_t)col * out_f + row] = v;
                    } else {
                        st_tagged(part + (size_t)b * kPartialMax + e, v, tag);
                    }
                }
                if constexpr (NT == 1 && TW == kTiles && MAXOPS == 1) {
                    // the lm_head epilogue of a block finished here: noted, done after the runs
                    if (P.stats != nullptr && owner && threadIdx.x == 0 && s_nown < 2 * NW) s_own[s_nown++] = rb;
                }
            }
        }
        if constexpr (NT == 1 && TW == kTiles && MAXOPS == 1) {
            // the lm_head epilogue of the blocks this CTA finished from partials: one warp per
            // (block, column), from the outputs just written (read back through L2: rows lane
            // and lane + 32), all of them at once
            if (P.stats != nullptr) {
                __syncthreads();
                const int n_pairs = (int)s_nown * C;
                constexpr int kPP = 4;  // (block, column) pairs per warp and round, loads first
                for (int base = warp * kPP; base < n_pairs; base += NW * kPP) {
                    float v2[kPP][2];
#pragma unroll
                    for (int i = 0; i < kPP; ++i) {
                        const int pc = base + i;
                        const uint32_t rb = pc < n_pairs ? s_own[pc / C] : 0u;
                        const int col = pc < n_pairs ? pc % C : 0;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int64_t row = (int64_t)rb * kRowsPerBlock + lane + 32 * hh;
                            v2[i][hh] = (pc < n_pairs && row < out_f) ? __ldcg(o.Y + (int64_t)col * out_f + row)
                                                                      : __int_as_float(0x7fc00000);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kPP; ++i) {
                        const int pc = base + i;
                        if (pc >= n_pairs) break;  // uniform across the warp
                        const uint32_t rb = s_own[pc / C];
                        const int col = pc % C;
                        float bv = 0.f;
                        int bi = -1;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            if (v2[i][hh] == v2[i][hh])
                                stat_argmax(bv, bi, v2[i][hh], (int)((int64_t)rb * kRowsPerBlock + lane + 32 * hh));
#pragma unroll
                        for (int m = 1; m < 32; m <<= 1)
                            stat_argmax(bv, bi, __shfl_xor_sync(0xFFFFFFFFu, bv, m), __shfl_xor_sync(0xFFFFFFFFu, bi, m));
                        float sum = 0.f;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            if (v2[i][hh] == v2[i][hh]) sum += exp2f((v2[i][hh] - bv) * P.stat_k);
#pragma unroll
                        for (int m = 1; m < 32; m <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, m);
                        if (lane == 0)
                            P.stats[(size_t)rb * C + col] = make_float4(bi >= 0 ? bv : -INFINITY, sum, __int_as_float(bi), 0.f);
                    }
                }
            }
        }
        SVD_PROBE(gi, 2);
    }
    // after a give-up: wait (bounded) for the group's copies that may still be in flight -- the
    // last copy issued into each slot -- so that none lands in shared memory after the CTA exits
    if (sub == 0 && lane == 0 && wait_stopped(&s_wc)) {
        for (uint32_t k = c_issued > (uint32_t)R ? c_issued - R : 0u; k < c_issued; ++k)
            mbar_wait_ok(full0 + 8 * (k % R), (k / R) & 1u, kDrainLimit);
    }
    // the last CTA out returns the barrier counters to zero and advances the epoch; when the
    // partial tags are about to repeat it also clears every partial slot
    __syncthreads();
    if (threadIdx.x == 0) {
        s_last = 0u;
        if (atom_add_acqrel_gpu(gbar + kBarExit, 1u) == G - 1u) {
            gbar[kBarCount] = 0u;
            gbar[kBarExit] = 0u;
            gbar[kBarEpoch] = epoch + 1u;
            s_last = partial_epoch24(epoch + 1u) == 1u ? 1u : 0u;
        }
    }
    __syncthreads();
    if (s_last)
        for (uint32_t i = threadIdx.x; i < part_entries; i += kThreads) part[i] = 0ull;
}

// ---- the CUDA-core kernel (canonical layout) -------------------------------------------
// One warp per output row; lane l takes 32-input blocks l, l+32, ...: one 16-byte load of 32
// nibbles, value (c - 8) built exactly as float(2^23 + c) - (2^23 + 8), C fp32 FMAs per
// weight against activations held in shared memory as fp32 (one pad word every 32 to spread
// the lanes over the banks), the block sum scaled by its fp16 scale, then a butterfly
// reduction over the warp.
template <int CC>
__global__ void __launch_bounds__(256)
vl_simt_kernel(const uint8_t *__restrict__ codes, const uint16_t *__restrict__ scales,
               const __nv_bfloat16 *__restrict__ X, float *__restrict__ Y, int64_t in_f,
               int64_t out_f) {
    extern __shared__ float xs[];
    const int64_t pitch = in_f + in_f / 32;
    griddep_wait();
    for (int64_t i = threadIdx.x; i < CC * in_f; i += blockDim.x) {
        const int64_t c = i / in_f, k = i % in_f;
        xs[c * pitch + k + k / 32] = __bfloat162float(X[i]);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nblk = in_f / 32;
    for (int64_t row = (int64_t)blockIdx.x * 8 + warp; row < out_f; row += (int64_t)gridDim.x * 8) {
        float acc[CC];
#pragma unroll
        for (int c = 0; c < CC; ++c) acc[c] = 0.f;
        for (int64_t blk = lane; blk < nblk; blk += 32) {
            const uint4 q = ldg_nc_v4(codes + row * (in_f / 2) + blk * 16);
            const float s = __half2float(__ushort_as_half(scales[row * nblk + blk]));
            const uint32_t words[4] = {q.x, q.y, q.z, q.w};
            float part[CC];
#pragma unroll
            for (int c = 0; c < CC; ++c) part[c] = 0.f;
            const float *xb = xs + blk * 32 + blk;
#pragma unroll
            for (int wi = 0; wi < 4; ++wi)
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    const uint32_t nib = (words[wi] >> (4 * n)) & 15u;
                    const float wv = __uint_as_float(0x4B000000u | nib) - 8388616.0f;
#pragma unroll
                    for (int c = 0; c < CC; ++c) part[c] = fmaf(wv, xb[c * pitch + wi * 8 + n], part[c]);
                }
#pragma unroll
            for (int c = 0; c < CC; ++c) acc[c] = fmaf(s, part[c], acc[c]);
        }
#pragma unroll
        for (int c = 0; c < CC; ++c) {
            float v = acc[c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[c] = v;
        }
        if (lane == 0)
#pragma unroll
            for (int c = 0; c < CC; ++c) Y[(int64_t)c * out_f + row] = acc[c];
    }
}

#include "verify_linear_tc.cuh"

// ---- host side ---------------------------------------------------------------------------
#ifndef SVD_NW1
#define SVD_NW1 16
#endif
#ifndef SVD_R1
#define SVD_R1 2
#endif
#ifndef SVD_U
#define SVD_U 2
#endif
constexpr int kNW1 = SVD_NW1;     // warps per CTA, C <= 8
constexpr int kR1 = SVD_R1;       // ring slots per warp, C <= 5
constexpr int kU = SVD_U;         // units per slot (one pair of bulk copies)
constexpr int kR1w = 4;           // 6..8 columns: four one-unit slots per warp (the same ring
constexpr int kU1w = 1;           // bytes; 1-3 % faster there, no gain at 5 columns or fewer)
constexpr int kNW2 = 16;          // warps per CTA, 8 < C <= 16: two warps per unit,
constexpr int kTW2 = 2;           // each on two of its four 16-row tiles
constexpr int kR2 = 2;            // ring slots per worker group, C <= 32
constexpr int kNW4 = 8;           // warps per CTA, 16 < C <= 32: one warp per unit (all four row
constexpr int kTW4 = 4;           // tiles), so each activation fragment serves four tiles; 255
                                  // registers a thread hold the accumulators (16 warps spill)
#ifndef SVD_TWQ
#define SVD_TWQ 2
#endif
#ifndef SVD_RQ
#define SVD_RQ 2
#endif
#ifndef SVD_NWQ
#define SVD_NWQ 16
#endif
constexpr int kNWq = SVD_NWQ;     // Q4_K units (64 rows x 256 inputs, 9 KB), C <= 8: two warps
constexpr int kTWq = SVD_TWQ;     // per unit, each on two 16-row tiles; one unit per slot, two
constexpr int kRq = SVD_RQ;       // slots per worker group
constexpr int kUq = 1;
constexpr int kTWq2 = 1;          // Q4_K, 8 < C <= 16: four warps per unit, one 16-row tile each,
constexpr int kRq2 = 4;           // four slots per group (the accumulators of two n-tiles)
constexpr int kMaxCtasPerSm = 2;  // the workspace holds partial slots for this many
constexpr int kChainMax = 256;    // ops per chain launch (kernel parameters, ~16 KB)

static int ntiles_for(int C) { return C <= 8 ? 1 : (C <= 16 ? 2 : 4); }

// Workspace: [partial slots: SMs x kMaxCtasPerSm CTAs x kPartialMax tagged 64-bit entries]
//            [barrier words, 256 bytes: grid-barrier counter, exit counter, launch epoch]
//            [17..32 columns only: the fp16 B tiles of the op's activations, 4 KB per 64
//             inputs of the widest op, 1024-byte aligned].
// Up to 16 columns it has the same size for every matrix, so calls of any shape can share one
// zero-filled workspace; every launch returns the counters to zero and advances the epoch that
// tags its partials.
static size_t partial_entries() { return (size_t)sm_count() * kMaxCtasPerSm * kPartialMax; }
static size_t partial_region_bytes() {
    return align_up((size_t)sm_count() * kMaxCtasPerSm * kPartialMax * sizeof(unsigned long long),
                    256);
}
constexpr size_t kBarrierBytes = 256;
static_assert((kBarEpoch + 1) * sizeof(unsigned) <= kBarrierBytes, "barrier words");
// B tiles of the tensor-core kernel (C > 16), after the barrier words; 1 KB of alignment slack
static size_t tc_xb_region(int64_t max_in_f, int C) {
    return C > 16 ? tc_xb_bytes(max_in_f) + 1024 : 0;
}
static uint8_t *tc_xb_ptr(void *ws) {
    const uintptr_t p = reinterpret_cast<uintptr_t>(ws) + partial_region_bytes() + kBarrierBytes;
    return reinterpret_cast<uint8_t *>((p + 1023) & ~(uintptr_t)1023);
}

size_t vl_workspace_bytes(int64_t in_f, int64_t out_f, int C) {
    (void)out_f;
    return partial_region_bytes() + kBarrierBytes + tc_xb_region(in_f, C);
}

template <int NT, int NW, int TW, int R, int U, int MAXOPS, int KQ = 0>
static cudaError_t launch_stream(const VlOps<MAXOPS> &P, void *ws, bool pdl, bool coop,
                                 int64_t max_units, cudaStream_t stream) {
    using Cfg = VlCfg<NT, NW, TW, R, U, MAXOPS, KQ>;
    auto kern = vl_stream_kernel<NT, NW, TW, R, U, MAXOPS, KQ>;
    static int per_sm_cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int per_sm = (dev >= 0 && dev < 64) ? per_sm_cache[dev] : 0;
    if (per_sm == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::kThreads, Cfg::kSmem);
        if (e != cudaSuccess) return e;
        per_sm = per_sm < 1 ? 1 : (per_sm > kMaxCtasPerSm ? kMaxCtasPerSm : per_sm);
        if (dev >= 0 && dev < 64) per_sm_cache[dev] = per_sm;
    }
    int64_t G = (int64_t)sm_count() * per_sm;
    if (!coop && G > max_units) G = max_units;  // a lone op never needs idle CTAs
    if (G < 1) G = 1;
    uint8_t *base = reinterpret_cast<uint8_t *>(ws);
    auto *part = reinterpret_cast<unsigned long long *>(base);
    unsigned *gbar = reinterpret_cast<unsigned *>(base + partial_region_bytes());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (coop) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    } else if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, P, part, (uint32_t)partial_entries(), gbar);
}

static VlOp make_op(const svd_qweight *W, const void *X, float *Y) {
    const NativeGeom ng = W->layout == SVD_LAYOUT_Q4K_NATIVE ? kq_geom(W->in_features, W->out_features)
                                                             : native_geom(W->in_features, W->out_features);
    VlOp o;
    o.codes = reinterpret_cast<const uint8_t *>(W->codes);
    o.scales = reinterpret_cast<const uint8_t *>(W->scales);
    o.X = reinterpret_cast<const __nv_bfloat16 *>(X);
    o.Y = Y;
    o.in_f = W->in_features;
    o.out_f = W->out_features;
    o.n_kc = (uint32_t)ng.n_kc;
    o.n_units = (uint32_t)ng.n_units;
    return o;
}

// The tensor-core kernel: one CTA per SM (a cooperative launch for a chain), each holding
// kTcTmemCols TMEM columns, so two CTAs overlapping under programmatic dependent launch fit in
// one SM's 512.
template <int MAXOPS>
static cudaError_t launch_tc(const VlOps<MAXOPS> &P, void *ws, bool pdl, bool coop, cudaStream_t stream) {
    auto kern = vl_tc_kernel<MAXOPS>;
    constexpr size_t smem = TcCfg<MAXOPS>::kSmem;
    static bool ready[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !ready[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        if (dev >= 0 && dev < 64) ready[dev] = true;
    }
    int64_t max_units = 0;  // MMA units (128 rows x 64 inputs) of the largest op
    for (int i = 0; i < P.n; ++i) {
        const int64_t n_rb = P.op[i].n_units / P.op[i].n_kc;
        const int64_t u = (n_rb + 1) / 2 * (int64_t)P.op[i].n_kc;
        max_units = u > max_units ? u : max_units;
    }
    int64_t G = sm_count();
    if (!coop && G > max_units) G = max_units;
    if (G < 1) G = 1;
    uint8_t *base = reinterpret_cast<uint8_t *>(ws);
    auto *part = reinterpret_cast<unsigned long long *>(base);
    unsigned *gbar = reinterpret_cast<unsigned *>(base + partial_region_bytes());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (coop) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    } else if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, P, part, (uint32_t)partial_entries(), gbar, tc_xb_ptr(ws));
}

// 17..32 columns run on the tensor-core kernel unless the caller asks for the fragment kernel.
// Q4_K native ops (C <= 8, checked by the callers) run the stream kernel on Q4_K units.
template <int MAXOPS>
static cudaError_t launch_ops(const VlOps<MAXOPS> &P, void *ws, bool pdl, cudaStream_t stream,
                              bool fragment_mma = false, bool q4k = false) {
    int64_t max_units = 0;
    for (int i = 0; i < P.n; ++i)
        max_units = (int64_t)P.op[i].n_units > max_units ? (int64_t)P.op[i].n_units : max_units;
    const bool coop = P.n > 1;
    if (q4k) {
        if (P.C <= 8) return launch_stream<1, kNWq, kTWq, kRq, kUq, MAXOPS, 1>(P, ws, pdl, coop, max_units, stream);
        return launch_stream<2, kNWq, kTWq2, kRq2, kUq, MAXOPS, 1>(P, ws, pdl, coop, max_units, stream);
    }
    switch (ntiles_for(P.C)) {
        case 1:
            if (P.C >= 6) return launch_stream<1, kNW1, kTiles, kR1w, kU1w, MAXOPS>(P, ws, pdl, coop, max_units, stream);
            return launch_stream<1, kNW1, kTiles, kR1, kU, MAXOPS>(P, ws, pdl, coop, max_units, stream);
        case 2: return launch_stream<2, kNW2, kTW2, kR2, kU, MAXOPS>(P, ws, pdl, coop, max_units, stream);
        default:
            if (!fragment_mma) return launch_tc<MAXOPS>(P, ws, pdl, coop, stream);
            return launch_stream<4, kNW4, kTW4, kR2, kU, MAXOPS>(P, ws, pdl, coop, max_units, stream);
    }
}

template <int CC>
static cudaError_t launch_simt(const svd_qweight *W, const void *X, float *Y, bool pdl,
                               cudaStream_t stream) {
    auto kern = vl_simt_kernel<CC>;
    const int64_t in_f = W->in_features;
    const size_t smem = (size_t)CC * (in_f + in_f / 32) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)sm_count() * per_sm;
    const int64_t need = (W->out_features + 7) / 8;
    if (grid > need) grid = need;
    return launch(kern, dim3((unsigned)grid), dim3(256), smem, stream, pdl,
                  reinterpret_cast<const uint8_t *>(W->codes),
                  reinterpret_cast<const uint16_t *>(W->scales),
                  reinterpret_cast<const __nv_bfloat16 *>(X), Y, in_f, W->out_features);
}

static int check_qweight(const svd_qweight *W) {
    if (!W || !W->codes) return SVD_ERR_INVALID_ARG;
    if (W->in_features <= 0 || W->out_features <= 0 || W->in_features % 32 != 0)
        return SVD_ERR_INVALID_ARG;
    if (W->reserved != 0) return SVD_ERR_INVALID_ARG;
    if (W->layout == SVD_LAYOUT_Q4K) {  // super-blocks only: no separate scales
        if (W->scales || W->in_features % 256 != 0 || !aligned16(W->codes)) return SVD_ERR_INVALID_ARG;
        return SVD_OK;
    }
    if (!W->scales) return SVD_ERR_INVALID_ARG;
    if (W->layout == SVD_LAYOUT_Q4K_NATIVE && W->in_features % 256 != 0) return SVD_ERR_INVALID_ARG;
    if (W->layout != SVD_LAYOUT_CANONICAL && W->layout != SVD_LAYOUT_NATIVE &&
        W->layout != SVD_LAYOUT_Q4K_NATIVE)
        return SVD_ERR_INVALID_ARG;
    if (!aligned16(W->codes) || !aligned16(W->scales)) return SVD_ERR_INVALID_ARG;
    return SVD_OK;
}

int verify_linear_q4k(const svd_qweight *W, const void *X, int C, float *Y, bool pdl,
                      cudaStream_t stream);

// The stream-K kernel does its unit arithmetic in 32 bits: n_units * (workers + 1) must
// stay below 2^32 (about 880 thousand units, 3.6 billion weights, on 152 SMs).
static int check_native_size(const svd_qweight *W) {
    const NativeGeom ng = W->layout == SVD_LAYOUT_Q4K_NATIVE ? kq_geom(W->in_features, W->out_features)
                                                             : native_geom(W->in_features, W->out_features);
    const uint64_t workers = (uint64_t)sm_count() * kMaxCtasPerSm * 16 + 1;
    if ((uint64_t)ng.n_units * workers > 0xFFFFFFFFull) return SVD_ERR_UNSUPPORTED;
    return SVD_OK;
}

// verify_linear with the lm_head epilogue: when stats is not null, C <= 8 and W is NATIVE, the
// launch also writes the per-block statistics described at VlOps (and *stats_done = true).
int verify_linear_ex(const svd_qweight *W, const void *X, int C, float *Y, void *ws,
                     size_t ws_bytes, int flags, float4 *stats, float stat_k, bool *stats_done,
                     cudaStream_t stream) {
    if (stats_done) *stats_done = false;
    int rc = check_qweight(W);
    if (rc != SVD_OK) return rc;
    if (!X || !Y || C < 1 || C > SVD_C_MAX || !aligned16(X)) return SVD_ERR_INVALID_ARG;
    if (flags & ~(SVD_F_PDL | SVD_F_FRAGMENT_MMA)) return SVD_ERR_INVALID_ARG;
    const bool pdl = (flags & SVD_F_PDL) != 0;
    if (sm_count() < 1) return SVD_ERR_CUDA;
    if (W->layout == SVD_LAYOUT_NATIVE || W->layout == SVD_LAYOUT_Q4K_NATIVE) {
        const bool q4k = W->layout == SVD_LAYOUT_Q4K_NATIVE;
        if (q4k && C > 16) return SVD_ERR_UNSUPPORTED;
        rc = check_native_size(W);
        if (rc != SVD_OK) return rc;
        if (!ws || ws_bytes < vl_workspace_bytes(W->in_features, W->out_features, C))
            return SVD_ERR_WORKSPACE;
        VlOps<1> P;
        P.n = 1;
        P.C = C;
        P.op[0] = make_op(W, X, Y);
        if (stats && !q4k && ntiles_for(C) == 1) {
            P.stats = stats;
            P.stat_k = stat_k;
            if (stats_done) *stats_done = true;
        }
        SVD_CUDA_TRY(launch_ops(P, ws, pdl, stream, (flags & SVD_F_FRAGMENT_MMA) != 0, q4k));
        return SVD_OK;
    }
    if (W->layout == SVD_LAYOUT_Q4K) {  // K-quant super-blocks: CUDA-core kernel (kquant.cu)
        if (C > 8) return SVD_ERR_UNSUPPORTED;
        return verify_linear_q4k(W, X, C, Y, pdl, stream);
    }
    // canonical layout: CUDA-core kernel
    if ((int64_t)C * W->in_features * 4 > 196608) return SVD_ERR_UNSUPPORTED;
    cudaError_t e;
    switch (C) {
        case 1: e = launch_simt<1>(W, X, Y, pdl, stream); break;
        case 2: e = launch_simt<2>(W, X, Y, pdl, stream); break;
        case 3: e = launch_simt<3>(W, X, Y, pdl, stream); break;
        case 4: e = launch_simt<4>(W, X, Y, pdl, stream); break;
        case 5: e = launch_simt<5>(W, X, Y, pdl, stream); break;
        case 6: e = launch_simt<6>(W, X, Y, pdl, stream); break;
        case 7: e = launch_simt<7>(W, X, Y, pdl, stream); break;
        case 8: e = launch_simt<8>(W, X, Y, pdl, stream); break;
        default: return SVD_ERR_UNSUPPORTED;
    }
    SVD_CUDA_TRY(e);
    return SVD_OK;
}

int verify_linear(const svd_qweight *W, const void *X, int C, float *Y, void *ws,
                  size_t ws_bytes, int flags, cudaStream_t stream) {
    return verify_linear_ex(W, X, C, Y, ws, ws_bytes, flags, nullptr, 0.f, nullptr, stream);
}

size_t chain_workspace_bytes(const svd_linear_op *ops, int n_ops, int C) {
    int64_t max_in = 0;
    for (int i = 0; ops && i < n_ops; ++i)
        max_in = ops[i].W.in_features > max_in ? ops[i].W.in_features : max_in;
    return partial_region_bytes() + kBarrierBytes + tc_xb_region(max_in, C);
}

int verify_chain(const svd_linear_op *ops, int n_ops, int C, void *ws, size_t ws_bytes, int flags,
                 cudaStream_t stream) {
    if (!ops || n_ops < 1 || C < 1 || C > SVD_C_MAX) return SVD_ERR_INVALID_ARG;
    if (flags & ~(SVD_F_PDL | SVD_F_FRAGMENT_MMA)) return SVD_ERR_INVALID_ARG;
    // one layout for the whole chain: native, or Q4_K native (up to 8 columns)
    const bool q4k = ops[0].W.layout == SVD_LAYOUT_Q4K_NATIVE;
    if (q4k && C > 16) return SVD_ERR_UNSUPPORTED;
    for (int i = 0; i < n_ops; ++i) {
        const int rc = check_qweight(&ops[i].W);
        if (rc != SVD_OK) return rc;
        if (ops[i].W.layout != (q4k ? SVD_LAYOUT_Q4K_NATIVE : SVD_LAYOUT_NATIVE)) return SVD_ERR_INVALID_ARG;
        if (check_native_size(&ops[i].W) != SVD_OK) return SVD_ERR_UNSUPPORTED;
        if (!ops[i].X || !ops[i].Y || !aligned16(ops[i].X)) return SVD_ERR_INVALID_ARG;
    }
    if (sm_count() < 1) return SVD_ERR_CUDA;
    if (!ws || ws_bytes < chain_workspace_bytes(ops, n_ops, C)) return SVD_ERR_WORKSPACE;
    // host staging of the kernel parameters (copied into the launch)
    std::unique_ptr<VlOps<kChainMax>> Pp(new VlOps<kChainMax>);
    VlOps<kChainMax> &P = *Pp;
    for (int first = 0; first < n_ops; first += kChainMax) {
        const int n = (n_ops - first) < kChainMax ? (n_ops - first) : kChainMax;
        if (n == 1) {
            VlOps<1> P1;
            P1.n = 1;
            P1.C = C;
            P1.op[0] = make_op(&ops[first].W, ops[first].X, ops[first].Y);
            SVD_CUDA_TRY(launch_ops(P1, ws, first == 0 && (flags & SVD_F_PDL), stream, (flags & SVD_F_FRAGMENT_MMA) != 0, q4k));
            continue;
        }
        P.n = n;
        P.C = C;
        for (int i = 0; i < n; ++i) P.op[i] = make_op(&ops[first + i].W, ops[first + i].X, ops[first + i].Y);
        SVD_CUDA_TRY(launch_ops(P, ws, false, stream, (flags & SVD_F_FRAGMENT_MMA) != 0, q4k));
    }
    return SVD_OK;
}

int native_sizes(int64_t in_f, int64_t out_f, size_t *cb, size_t *sb) {
    if (in_f <= 0 || out_f <= 0 || in_f % 32 != 0) return SVD_ERR_INVALID_ARG;
    const NativeGeom ng = native_geom(in_f, out_f);
    if (cb) *cb = (size_t)ng.n_units * kUnitCodeBytes;
    if (sb) *sb = (size_t)ng.n_units * kUnitScaleBytes;
    return SVD_OK;
}

int kq_native_sizes(int64_t in_f, int64_t out_f, size_t *cb, size_t *hb) {
    if (in_f <= 0 || out_f <= 0 || in_f % kKqIn != 0) return SVD_ERR_INVALID_ARG;
    const NativeGeom ng = kq_geom(in_f, out_f);
    if (cb) *cb = (size_t)ng.n_units * kKqUnitCodeBytes;
    if (hb) *hb = (size_t)ng.n_units * kKqUnitHdrBytes;
    return SVD_OK;
}

static int kq_repack(const svd_qweight *src, void *dc, void *dh, cudaStream_t stream) {
    if (!dc || !dh || !aligned16(dc) || !aligned16(dh)) return SVD_ERR_INVALID_ARG;
    const NativeGeom ng = kq_geom(src->in_features, src->out_features);
    const int64_t n_words = ng.n_units * (kKqUnitCodeBytes / 4);
    const int64_t n_rows = ng.n_units * kRowsPerBlock;
    kq_repack_codes_kernel<<<(unsigned)((n_words + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint8_t *>(src->codes), reinterpret_cast<uint32_t *>(dc),
        src->in_features, src->out_features, ng.n_kc, n_words);
    SVD_CUDA_TRY(cudaGetLastError());
    kq_repack_hdr_kernel<<<(unsigned)((n_rows + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint8_t *>(src->codes), reinterpret_cast<uint4 *>(dh),
        src->in_features, src->out_features, ng.n_kc, n_rows);
    SVD_CUDA_TRY(cudaGetLastError());
    return SVD_OK;
}

static int kq_unpack(const svd_qweight *src, void *dst, void *dnull, cudaStream_t stream) {
    if (!dst || dnull) return SVD_ERR_INVALID_ARG;
    const NativeGeom ng = kq_geom(src->in_features, src->out_features);
    const int64_t nb = src->out_features * (src->in_features / kKqIn * kKqBlockBytes);
    kq_unpack_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint32_t *>(src->codes), reinterpret_cast<const uint8_t *>(src->scales),
        reinterpret_cast<uint8_t *>(dst), src->in_features, src->out_features, ng.n_kc);
    SVD_CUDA_TRY(cudaGetLastError());
    return SVD_OK;
}

int repack(const svd_qweight *src, void *dc, void *ds, cudaStream_t stream) {
    int rc = check_qweight(src);
    if (rc != SVD_OK) return rc;
    if (src->layout == SVD_LAYOUT_Q4K) return kq_repack(src, dc, ds, stream);
    if (src->layout != SVD_LAYOUT_CANONICAL || !dc || !ds || !aligned16(dc) || !aligned16(ds))
        return SVD_ERR_INVALID_ARG;
    const NativeGeom ng = native_geom(src->in_features, src->out_features);
    const int64_t n_words = ng.n_units * (kUnitCodeBytes / 4);
    const int64_t n_halves = ng.n_units * (kUnitScaleBytes / 2);
    repack_codes_kernel<<<(unsigned)((n_words + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint8_t *>(src->codes), reinterpret_cast<uint32_t *>(dc),
        src->in_features, src->out_features, ng.n_kc, n_words);
    SVD_CUDA_TRY(cudaGetLastError());
    repack_scales_kernel<<<(unsigned)((n_halves + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint16_t *>(src->scales), reinterpret_cast<uint16_t *>(ds),
        src->in_features, src->out_features, ng.n_kc, n_halves);
    SVD_CUDA_TRY(cudaGetLastError());
    return SVD_OK;
}

int unpack(const svd_qweight *src, void *dc, void *ds, cudaStream_t stream) {
    int rc = check_qweight(src);
    if (rc != SVD_OK) return rc;
    if (src->layout == SVD_LAYOUT_Q4K_NATIVE) return kq_unpack(src, dc, ds, stream);
    if (src->layout != SVD_LAYOUT_NATIVE || !dc || !ds) return SVD_ERR_INVALID_ARG;
    const NativeGeom ng = native_geom(src->in_features, src->out_features);
    const int64_t nb = src->out_features * (src->in_features / 2);
    const int64_t ns = src->out_features * (src->in_features / 32);
    unpack_codes_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint32_t *>(src->codes), reinterpret_cast<uint8_t *>(dc),
        src->in_features, src->out_features, ng.n_kc);
    SVD_CUDA_TRY(cudaGetLastError());
    unpack_scales_kernel<<<(unsigned)((ns + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint16_t *>(src->scales), reinterpret_cast<uint16_t *>(ds),
        src->in_features, src->out_features, ng.n_kc);
    SVD_CUDA_TRY(cudaGetLastError());
    return SVD_OK;
}

// ---- failure detection: the workspace's status word and the stall injection -------------
__global__ void set_word_kernel(unsigned *p, unsigned v) { *p = v; }

static unsigned *workspace_counters(const void *ws) {
    return reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(const_cast<void *>(ws)) +
                                        partial_region_bytes());
}

int verify_status(const void *ws, size_t ws_bytes, uint32_t *bits, cudaStream_t stream) {
    if (sm_count() < 1) return SVD_ERR_CUDA;
    if (!ws || ws_bytes < partial_region_bytes() + kBarrierBytes) return SVD_ERR_WORKSPACE;
    unsigned *st = workspace_counters(ws) + kBarStatus;
    unsigned v = 0;
    SVD_CUDA_TRY(cudaMemcpyAsync(&v, st, sizeof(v), cudaMemcpyDeviceToHost, stream));
    SVD_CUDA_TRY(cudaStreamSynchronize(stream));
    if (bits) *bits = v;
    if (v == 0u) return SVD_OK;
    set_word_kernel<<<1, 1, 0, stream>>>(st, 0u);
    SVD_CUDA_TRY(cudaGetLastError());
    SVD_CUDA_TRY(cudaStreamSynchronize(stream));
    return SVD_ERR_TIMEOUT;
}

int verify_inject_stall(void *ws, size_t ws_bytes, uint32_t polls, cudaStream_t stream) {
    if (sm_count() < 1) return SVD_ERR_CUDA;
    if (!ws || ws_bytes < partial_region_bytes() + kBarrierBytes) return SVD_ERR_WORKSPACE;
    const unsigned word = polls == SVD_POLL_DEFAULT ? 0u : polls + 1u;  // 0 keeps the default
    set_word_kernel<<<1, 1, 0, stream>>>(workspace_counters(ws) + kBarPoll, word);
    SVD_CUDA_TRY(cudaGetLastError());
    return SVD_OK;
}

// ---- verify linear without caller scratch ----------------------------------------------
// The stream-K kernel needs a small scratch area (tagged partial sums of row blocks split
// between CTAs, and the barrier words).  svd_verify_linear takes it from the caller;
// this variant takes it from a fixed array in the library's own device memory instead, for
// callers that cannot allocate device memory.  The array is reserved when the library's
// module is loaded on a device and stays there until the process exits.
constexpr int kNoAllocMaxSms = 160;
constexpr size_t kNoAllocPartialBytes =
    (size_t)kNoAllocMaxSms * kMaxCtasPerSm * kPartialMax * sizeof(unsigned long long);
constexpr size_t kNoAllocBytes = kNoAllocPartialBytes + kBarrierBytes;
static_assert(kNoAllocBytes <= SVD_NOALLOC_SCRATCH_BYTES, "scratch bound in svd.h");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch, looked up with the device current (in host code the
// symbol is only a host-side handle and must never reach a kernel).  It is looked up again on
// every call made outside stream capture, so a new context on the device (after
// cudaDeviceReset) never sees a stale address; during capture the last address is used.
static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[64] = {nullptr};

int verify_linear_noalloc(const svd_qweight *W, const void *X, int C, float *Y, int flags,
                          cudaStream_t stream) {
    int rc = check_qweight(W);
    if (rc != SVD_OK) return rc;
    if (W->layout != SVD_LAYOUT_NATIVE) return SVD_ERR_INVALID_ARG;
    if (!X || !Y || C < 1 || C > SVD_C_MAX || !aligned16(X)) return SVD_ERR_INVALID_ARG;
    if (flags & ~(SVD_F_PDL | SVD_F_FRAGMENT_MMA)) return SVD_ERR_INVALID_ARG;
    if (W->out_features > SVD_NOALLOC_MAX_OUT_FEATURES) return SVD_ERR_UNSUPPORTED;
    if (sm_count() >= 1 && check_native_size(W) != SVD_OK) return SVD_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms < 1) return SVD_ERR_CUDA;
    if (sms > kNoAllocMaxSms) return SVD_ERR_UNSUPPORTED;
    int dev = 0;
    SVD_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return SVD_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    SVD_CUDA_TRY(cudaStreamIsCapturing(stream, &cap));
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev] || cap == cudaStreamCaptureStatusNone) {
            if (cap != cudaStreamCaptureStatusNone) return SVD_ERR_UNSUPPORTED;  // first call captured
            void *p = nullptr;
            SVD_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
            g_noalloc_ptr[dev] = p;
        }
        base = g_noalloc_ptr[dev];
    }
    // Same layout as a caller workspace: partial slots, then the barrier words.  Every call
    // clears the counters (and the status word and poll limit) on the stream before its
    // kernel, so a call never depends on what an earlier call left behind; the epoch word (the
    // last one) is kept, so partials written by earlier calls never carry the tag of a later
    // one.
    unsigned char *counters = reinterpret_cast<unsigned char *>(base) + partial_region_bytes();
    SVD_CUDA_TRY(cudaMemsetAsync(counters, 0, kBarEpoch * sizeof(unsigned), stream));
    VlOps<1> P;
    P.n = 1;
    P.C = C;
    P.op[0] = make_op(W, X, Y);
    // above 16 columns the fixed array has no room for the tensor-core kernel's B tiles: the
    // warp-level kernel runs instead
    SVD_CUDA_TRY(launch_ops(P, base, (flags & SVD_F_PDL) != 0, stream, true));
    return SVD_OK;
}

}  // namespace svd

