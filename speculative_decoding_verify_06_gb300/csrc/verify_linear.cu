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
// Two kernels:
//  * vl_mma_kernel (NATIVE layout) -- persistent stream-K over (64-row block, 64-input chunk)
//    units.  Each warp owns a cp.async ring of its units in shared memory (codes + scales,
//    2304 bytes per unit), dequantises nibbles straight into bf16 A fragments with one lop3 and
//    one bf16x2 subtract per pair (value 128 + c built from the exponent pattern 0x4300, then
//    minus 136 gives c - 8 exactly), and runs mma.sync m16n8k16 (bf16 in, fp32 accumulate)
//    against the activations as the B operand.  Every 32-input block gets a fresh accumulator
//    that is scaled by its fp16 scale in fp32, so the only rounding is fp32 accumulation.
//    Warps of a CTA interleave the chunks of a row block; partial row blocks at the edges of a
//    CTA's range are combined through a small workspace by the last CTA to arrive (an atomic
//    ticket per row block, summed in CTA order: deterministic, no spinning).
//  * vl_simt_kernel (CANONICAL layout) -- the plain CUDA-core version: one warp per output
//    row, each lane one 32-input block at a time, fp32 FMAs, warp-shuffle reduction.
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
constexpr int kUnitBytes = kUnitCodeBytes + kUnitScaleBytes;

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

// ---- device building blocks -----------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Bulk (TMA-engine) copies into shared memory completing on an mbarrier.
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(mbar)
        : "memory");
}
// Waits for phase `parity` of an mbarrier; gives up after a bounded number of polls (each poll
// may suspend the thread briefly), so a broken pipeline cannot hang the GPU.
__device__ __forceinline__ void mbar_wait(uint32_t mbar, uint32_t parity) {
    for (int it = 0; it < (1 << 22); ++it) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
            "selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(mbar), "r"(parity)
            : "memory");
        if (ok) return;
    }
}

// Four bf16x2 A registers from one native word: (bits >> 4p) & 0x000F000F | 0x43004300 is the
// pair (128 + c_lo, 128 + c_hi) exactly; subtracting (136, 136) leaves (c - 8) exactly.  With
// MULHI the three right shifts are taken as mul.hi by 2^28, 2^24, 2^20 held in registers (the
// integer-multiply unit), which leaves only the lop3s on the integer ALU.
template <bool MULHI>
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t a[4], uint32_t m4, uint32_t m8,
                                             uint32_t m12) {
    const uint32_t magic = 0x43004300u, bias = 0x43084308u;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t v, sh;
        if (MULHI) {
            sh = (p == 0) ? w : __umulhi(w, p == 1 ? m4 : (p == 2 ? m8 : m12));
        } else {
            sh = w >> (4 * p);
        }
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(sh), "r"(0x000F000Fu), "r"(magic));
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(a[p]) : "r"(v), "r"(bias));
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
    int64_t in_f, out_f, n_kc, n_units;
};

template <int MAXOPS>
struct VlOps {
    int n;
    int C;
    uint32_t m4, m8, m12;  // 2^28, 2^24, 2^20: shift multipliers kept opaque to the compiler
    VlOp op[MAXOPS];
};

// The units of an op are split into G_op = min(G, n_units) contiguous CTA ranges
// [b n / G_op, (b+1) n / G_op); every CTA below G_op owns at least one unit.
// owner_cta(n) is the CTA whose range holds unit n.
__device__ __forceinline__ int64_t owner_cta(int64_t n, int64_t Gop, int64_t n_units) {
    return ((n + 1) * Gop - 1) / n_units;
}

// ---- the tensor-core stream-K kernel ---------------------------------------------------
constexpr int kPartialSlotFloats = 32 * kTiles * 4 * 4;  // largest warp partial (4 n-tiles)

template <int NT, int NW, int D, bool ASYNC>
struct MmaCfg {
    static constexpr int kAcc = kTiles * NT * 4;              // fp32 accumulators per lane
    static constexpr int kPartial = 32 * kAcc;                // floats per warp partial
    static constexpr size_t kRing = (size_t)NW * D * kUnitBytes;
    static constexpr size_t kSmem =
        kRing + (size_t)(ASYNC ? 2 : 1) * NW * kPartial * sizeof(float);
};

// Runs every op of P in order on a persistent grid.  Each warp keeps a ring of D unit slots
// in shared memory filled by cp.async; the issue cursor walks the warp's units op after op,
// so the weights of op g+1 stream in while op g finishes.  Activations of op g+1 are read
// only after the grid barrier that ends op g (a chain of more than one op is launched
// cooperatively), or, for op 0, after griddepcontrol.wait.
//
// A row block ends asynchronously: each warp drops its partial sums into one of two shared
// buffers and takes a shared ticket; the last warp to arrive sums the eight partials (in warp
// order) and writes the rows or the CTA's stream-K partial, while the other warps go on
// streaming.  A buffer is reused two row blocks later, after its reducer has released it.
template <int NT, int NW, int D, int MAXOPS, int MINB, bool MULHI, bool ASYNC, bool BULK>
__global__ void __launch_bounds__(NW * 32, MINB)
vl_mma_kernel(const __grid_constant__ VlOps<MAXOPS> P, float *__restrict__ ws_part,
              unsigned int *__restrict__ ws_cnt) {
    using Cfg = MmaCfg<NT, NW, D, ASYNC>;
    constexpr int kAcc = Cfg::kAcc, kPartial = Cfg::kPartial;
    constexpr int kPerLane = kPartial / 32;  // reduced elements per lane of the reducer warp
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ unsigned s_tick[2], s_free[2];
    __shared__ __align__(8) uint64_t s_mbar[BULK ? NW * D : 1];
    float *red = reinterpret_cast<float *>(smem + Cfg::kRing);  // [2][NW][kPartial]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int C = P.C;
    uint8_t *ring = smem + (size_t)warp * D * kUnitBytes;
    if (threadIdx.x < 2) {
        s_tick[threadIdx.x] = 0u;
        s_free[threadIdx.x] = 0u;
    }
    const uint32_t mbar0 = smem_u32(&s_mbar[0]) + (BULK ? warp * D * 8 : 0);
    if (BULK && lane == 0) {
        for (int i = 0; i < D; ++i) mbar_init(mbar0 + 8 * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    // ---- issue cursor: (op ig, unit ij of iJ), source pointers, ring slot ------------------
    int ig = -1, ij = 0, iJ = 0, islot = 0;
    const uint8_t *pc = nullptr, *ps = nullptr;
    auto iseek = [&]() {
        while (ij >= iJ) {
            if (++ig >= P.n) return;
            const VlOp &o = P.op[ig];
            const int64_t Gop = min(G, o.n_units);
            ij = 0;
            iJ = 0;
            if (b >= Gop) continue;
            const int64_t st = b * o.n_units / Gop, en = (b + 1) * o.n_units / Gop;
            const int64_t span = en - st;
            iJ = span > warp ? (int)((span - warp + NW - 1) / NW) : 0;
            pc = o.codes + (st + warp) * kUnitCodeBytes + lane * 16;
            ps = o.scales + (st + warp) * kUnitScaleBytes + lane * 16;
        }
    };
    auto issue_one = [&]() {
        if (ig < P.n) {
            if constexpr (BULK) {
                if (lane == 0) {
                    const uint32_t slot = smem_u32(ring + islot * kUnitBytes);
                    const uint32_t mb = mbar0 + 8 * islot;
                    // the slot was last read through the generic proxy: order those reads
                    // before the bulk copy (async proxy) overwrites it
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(mb, kUnitBytes);
                    bulk_g2s(slot, pc - lane * 16, kUnitCodeBytes, mb);
                    bulk_g2s(slot + kUnitCodeBytes, ps - lane * 16, kUnitScaleBytes, mb);
                }
            } else {
                uint8_t *slot = ring + islot * kUnitBytes + lane * 16;
#pragma unroll
                for (int r = 0; r < kTiles; ++r) cp_async16(slot + r * 512, pc + r * 512);
                if (lane < kUnitScaleBytes / 16) cp_async16(slot + kUnitCodeBytes, ps);
            }
            pc += NW * kUnitCodeBytes;
            ps += NW * kUnitScaleBytes;
            ++ij;
            islot = (islot + 1 == D) ? 0 : islot + 1;
            iseek();
        }
        if constexpr (!BULK) cp_async_commit();
    };
    iseek();
    // Weights never depend on earlier kernels or ops: start streaming before any wait.
#pragma unroll
    for (int s = 0; s < D - 1; ++s) issue_one();
    __syncthreads();  // s_tick / s_free initialised

    float acc[kTiles][NT][4];
#pragma unroll
    for (int r = 0; r < kTiles; ++r)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[r][nt][q] = 0.f;

    int cslot = 0;
    uint32_t cphase = 0;  // parity of the slot's current use (bulk copies)
    unsigned seg = 0;  // row-block segments this CTA has finished (all ops)
    for (int gi = 0; gi < P.n; ++gi) {
        const VlOp &o = P.op[gi];
        if (gi == 0) {
            griddep_wait();
            griddep_launch_dependents();
        } else {
            cooperative_groups::this_grid().sync();
        }
        const int64_t Gop = min(G, o.n_units);
        if (b >= Gop) continue;
        const int64_t n_kc = o.n_kc, n_units = o.n_units, in_f = o.in_f, out_f = o.out_f;
        const int64_t start = b * n_units / Gop, end = (b + 1) * n_units / Gop;
        const int64_t span = end - start;
        const int J = span > warp ? (int)((span - warp + NW - 1) / NW) : 0;

        // this lane's activation rows (B operand: column nt*8 + g4, inputs from t4*8)
        const __nv_bfloat16 *xrow[NT];
        bool xok[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g4;
            xok[nt] = col < C;
            xrow[nt] = o.X + (int64_t)(xok[nt] ? col : 0) * in_f + t4 * 8;
        }
        const bool tail32 = (in_f & 63) != 0;  // the last chunk holds a single 32-input block
        auto load_x = [&](int64_t kc, uint4 (&xr)[NT][2]) {
            const bool lastc = tail32 && (kc == n_kc - 1);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const __nv_bfloat16 *src = xrow[nt] + kc * kChunk;
                xr[nt][0] = xok[nt] ? ldg_nc_v4(src) : make_uint4(0u, 0u, 0u, 0u);
                xr[nt][1] = (xok[nt] && !lastc) ? ldg_nc_v4(src + 32) : make_uint4(0u, 0u, 0u, 0u);
            }
        };

        int64_t u = start + warp;
        int64_t kc = u % n_kc;
        uint4 xr[NT][2];
        if (J > 0) load_x(kc, xr);
        int j = 0;
        const int64_t rb_first = start / n_kc, rb_last = (end - 1) / n_kc;
        for (int64_t rb = rb_first; rb <= rb_last; ++rb, ++seg) {
            const int64_t seg_lo = max(start, rb * n_kc), seg_hi = min(end, (rb + 1) * n_kc);
            while (j < J && u < seg_hi) {
                issue_one();
                if constexpr (BULK) {
                    mbar_wait(mbar0 + 8 * cslot, cphase);
                } else {
                    cp_async_wait<D - 1>();
                    __syncwarp();
                }
                uint4 xc[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    xc[nt][0] = xr[nt][0];
                    xc[nt][1] = xr[nt][1];
                }
                int64_t kn = kc + NW;
                while (kn >= n_kc) kn -= n_kc;
                if (j + 1 < J) load_x(kn, xr);
                const uint8_t *slot = ring + cslot * kUnitBytes;
                uint4 cw[kTiles];
                uint2 sc[kTiles];
#pragma unroll
                for (int r = 0; r < kTiles; ++r) {
                    cw[r] = *reinterpret_cast<const uint4 *>(slot + r * 512 + lane * 16);
                    sc[r] = *reinterpret_cast<const uint2 *>(slot + kUnitCodeBytes + r * 64 + g4 * 8);
                }
#pragma unroll
                for (int r = 0; r < kTiles; ++r) {
                    const float2 s_lo = __half22float2(*reinterpret_cast<const __half2 *>(&sc[r].x));
                    const float2 s_hi = __half22float2(*reinterpret_cast<const __half2 *>(&sc[r].y));
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        uint32_t a0[4], a1[4];
                        dequant_word<MULHI>(blk ? cw[r].z : cw[r].x, a0, P.m4, P.m8, P.m12);
                        dequant_word<MULHI>(blk ? cw[r].w : cw[r].y, a1, P.m4, P.m8, P.m12);
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
                __syncwarp();  // every lane is done with this slot before it is refilled
                if (++cslot == D) {
                    cslot = 0;
                    cphase ^= 1u;
                }
                ++j;
                u += NW;
                kc = kn;
            }

            // ---- end of row block rb ---------------------------------------------------------
            if constexpr (!ASYNC) {
                // All threads of the CTA combine the warps' partials, two elements each.
                {
                    float4 *dst = reinterpret_cast<float4 *>(red + warp * kPartial + lane * kAcc);
#pragma unroll
                    for (int r = 0; r < kTiles; ++r)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            dst[r * NT + nt] = make_float4(acc[r][nt][0], acc[r][nt][1],
                                                           acc[r][nt][2], acc[r][nt][3]);
                            acc[r][nt][0] = acc[r][nt][1] = acc[r][nt][2] = acc[r][nt][3] = 0.f;
                        }
                }
                __syncthreads();
                constexpr int kPer = kPartial / (NW * 32);
                float vals[kPer];
#pragma unroll
                for (int m = 0; m < kPer; ++m) {
                    const int e = threadIdx.x + m * NW * 32;
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) v += red[w * kPartial + e];
                    vals[m] = v;
                }
                auto coords = [&](int e, int64_t *row, int *col) {
                    const int lsrc = e / kAcc, idx = e % kAcc, q = idx & 3, rn = idx >> 2;
                    const int r = rn / NT, nt = rn % NT;
                    *row = rb * kRowsPerBlock + 16 * r + (lsrc >> 2) + ((q >> 1) ? 8 : 0);
                    *col = nt * 8 + (lsrc & 3) * 2 + (q & 1);
                };
                const bool full = (seg_lo == rb * n_kc) && (seg_hi == (rb + 1) * n_kc);
                if (full) {
#pragma unroll
                    for (int m = 0; m < kPer; ++m) {
                        int64_t row;
                        int col;
                        coords(threadIdx.x + m * NW * 32, &row, &col);
                        if (row < out_f && col < C) o.Y[(int64_t)col * out_f + row] = vals[m];
                    }
                } else {
                    // Stream-K fix-up: publish this CTA's partial, take a ticket (one thread,
                    // release); the last CTA of the row block sums every partial in CTA order.
                    const int slot_id = (rb == rb_first) ? 0 : 1;
                    float *mine = ws_part + (b * 2 + slot_id) * (int64_t)kPartialSlotFloats;
#pragma unroll
                    for (int m = 0; m < kPer; ++m) mine[threadIdx.x + m * NW * 32] = vals[m];
                    __threadfence();
                    __syncthreads();
                    const int64_t b_first = owner_cta(rb * n_kc, Gop, n_units);
                    const int64_t b_last = owner_cta((rb + 1) * n_kc - 1, Gop, n_units);
                    if (threadIdx.x == 0) {
                        __threadfence();
                        const unsigned old = atomicAdd(ws_cnt + rb, 1u);
                        s_tick[0] = (old == (unsigned)(b_last - b_first)) ? 1u : 0u;
                    }
                    __syncthreads();
                    if (s_tick[0]) {
                        __threadfence();
#pragma unroll
                        for (int m = 0; m < kPer; ++m) {
                            const int e = threadIdx.x + m * NW * 32;
                            float v = 0.f;
                            for (int64_t bb = b_first; bb <= b_last; ++bb) {
                                const int64_t bb_first_rb = (bb * n_units / Gop) / n_kc;
                                const int sid = (rb == bb_first_rb) ? 0 : 1;
                                v += __ldcg(ws_part + (bb * 2 + sid) * (int64_t)kPartialSlotFloats + e);
                            }
                            int64_t row;
                            int col;
                            coords(e, &row, &col);
                            if (row < out_f && col < C) o.Y[(int64_t)col * out_f + row] = v;
                        }
                        if (threadIdx.x == 0) ws_cnt[rb] = 0u;
                    }
                }
                __syncthreads();  // red and s_tick are free again
                continue;
            }

            // ---- asynchronous variant: the last warp of the row block reduces ----------------
            const int buf = seg & 1;
            if (seg >= 2) {  // the reducer of segment seg - 2 must have released the buffer
                const unsigned need = seg >> 1;
                for (int spin = 0; spin < (1 << 24); ++spin) {
                    if (*reinterpret_cast<volatile unsigned *>(&s_free[buf]) >= need) break;
                    __nanosleep(32);
                }
            }
            {
                float4 *dst = reinterpret_cast<float4 *>(red + (buf * NW + warp) * kPartial + lane * kAcc);
#pragma unroll
                for (int r = 0; r < kTiles; ++r)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        dst[r * NT + nt] = make_float4(acc[r][nt][0], acc[r][nt][1],
                                                       acc[r][nt][2], acc[r][nt][3]);
                        acc[r][nt][0] = acc[r][nt][1] = acc[r][nt][2] = acc[r][nt][3] = 0.f;
                    }
            }
            __syncwarp();
            unsigned ticket = 0;
            if (lane == 0) {
                __threadfence_block();
                ticket = atomicAdd(&s_tick[buf], 1u);
            }
            ticket = __shfl_sync(0xffffffffu, ticket, 0);
            if (ticket != NW - 1) continue;  // another warp reduces this row block

            // ---- the reducer: the last warp of the CTA to finish row block rb ----------------
            __threadfence_block();
            const float *rbuf = red + buf * NW * kPartial;
            float vals[kPerLane];
#pragma unroll
            for (int m = 0; m < kPerLane; ++m) {
                const int e = lane + 32 * m;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) v += rbuf[w * kPartial + e];
                vals[m] = v;
            }
            auto out_coords = [&](int e, int64_t *row, int *col) {
                const int lsrc = e / kAcc, idx = e % kAcc, q = idx & 3, rn = idx >> 2;
                const int r = rn / NT, nt = rn % NT;
                *row = rb * kRowsPerBlock + 16 * r + (lsrc >> 2) + ((q >> 1) ? 8 : 0);
                *col = nt * 8 + (lsrc & 3) * 2 + (q & 1);
            };
            const bool full = (seg_lo == rb * n_kc) && (seg_hi == (rb + 1) * n_kc);
            if (full) {
#pragma unroll
                for (int m = 0; m < kPerLane; ++m) {
                    int64_t row;
                    int col;
                    out_coords(lane + 32 * m, &row, &col);
                    if (row < out_f && col < C) o.Y[(int64_t)col * out_f + row] = vals[m];
                }
            } else {
                // Stream-K fix-up: publish this CTA's partial, take a ticket; the last CTA of
                // the row block sums every partial in CTA order and resets the ticket.
                const int slot_id = (rb == rb_first) ? 0 : 1;
                float *mine = ws_part + (b * 2 + slot_id) * (int64_t)kPartialSlotFloats;
#pragma unroll
                for (int m = 0; m < kPerLane; ++m) mine[lane + 32 * m] = vals[m];
                __threadfence();
                __syncwarp();
                const int64_t b_first = owner_cta(rb * n_kc, Gop, n_units);
                const int64_t b_last = owner_cta((rb + 1) * n_kc - 1, Gop, n_units);
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(ws_cnt + rb, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old == (unsigned)(b_last - b_first)) {
                    __threadfence();
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) {
                        const int e = lane + 32 * m;
                        float v = 0.f;
                        for (int64_t bb = b_first; bb <= b_last; ++bb) {
                            const int64_t bb_first_rb = (bb * n_units / Gop) / n_kc;
                            const int sid = (rb == bb_first_rb) ? 0 : 1;
                            v += __ldcg(ws_part + (bb * 2 + sid) * (int64_t)kPartialSlotFloats + e);
                        }
                        int64_t row;
                        int col;
                        out_coords(e, &row, &col);
                        if (row < out_f && col < C) o.Y[(int64_t)col * out_f + row] = v;
                    }
                    if (lane == 0) ws_cnt[rb] = 0u;
                }
            }
            __syncwarp();
            if (lane == 0) {
                s_tick[buf] = 0u;
                __threadfence_block();
                atomicAdd(&s_free[buf], 1u);
            }
        }
    }
    if constexpr (!BULK) cp_async_wait<0>();
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

// ---- host side ---------------------------------------------------------------------------
#ifndef SVD_NW
#define SVD_NW 16
#endif
#ifndef SVD_D1
#define SVD_D1 5
#endif
#ifndef SVD_MINB1
#define SVD_MINB1 1
#endif
#ifndef SVD_MULHI
#define SVD_MULHI false
#endif
#ifndef SVD_ASYNC
#define SVD_ASYNC false
#endif
#ifndef SVD_BULK
#define SVD_BULK true
#endif
constexpr int kNW = SVD_NW;        // warps per CTA
constexpr int kD1 = SVD_D1;        // ring depth, C <= 8
constexpr int kD2 = 4;             // ring depth, C <= 16 / 32
constexpr int kMinB1 = SVD_MINB1;  // CTAs per SM the C <= 8 kernel is compiled for
constexpr bool kMulHi = SVD_MULHI;
constexpr bool kAsyncRed = SVD_ASYNC;  // row-block reduction by the last warp (else all threads)
constexpr bool kBulk = SVD_BULK;       // weights by bulk copies (else per-lane cp.async)
constexpr int kMaxCtasPerSm = 2;   // the workspace holds partial slots for this many
constexpr int kChainMax = 256;     // ops per chain launch (kernel parameters, ~16 KB)

static int ntiles_for(int C) { return C <= 8 ? 1 : (C <= 16 ? 2 : 4); }

// Workspace: [partial slots: SMs x kMaxCtasPerSm CTAs x 2 x kPartialSlotFloats][tickets].  The
// partial region has the same size and place for every matrix and C, so calls of any shape
// can share one zero-filled workspace; the tickets after it are per 64-row block.
static size_t partial_region_bytes() {
    return align_up((size_t)sm_count() * kMaxCtasPerSm * 2 * kPartialSlotFloats * sizeof(float),
                    256);
}

size_t vl_workspace_bytes(int64_t in_f, int64_t out_f, int C) {
    (void)C;
    const NativeGeom ng = native_geom(in_f, out_f);
    return partial_region_bytes() + align_up((size_t)ng.n_rb * sizeof(unsigned), 256);
}

template <int NT, int D, int MAXOPS>
static cudaError_t launch_mma(const VlOps<MAXOPS> &P, void *ws, bool pdl, bool coop,
                              int64_t max_units, cudaStream_t stream) {
    constexpr int NW = (NT == 4 && kNW > 8) ? 8 : kNW;  // four n-tiles: partials fill smem
    using Cfg = MmaCfg<NT, NW, D, kAsyncRed>;
    auto kern = vl_mma_kernel<NT, NW, D, MAXOPS, (NT == 1 ? kMinB1 : 1), kMulHi, kAsyncRed, kBulk>;
    static int per_sm_cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int per_sm = (dev >= 0 && dev < 64) ? per_sm_cache[dev] : 0;
    if (per_sm == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, Cfg::kSmem);
        if (e != cudaSuccess) return e;
        per_sm = per_sm < 1 ? 1 : (per_sm > kMaxCtasPerSm ? kMaxCtasPerSm : per_sm);
        if (dev >= 0 && dev < 64) per_sm_cache[dev] = per_sm;
    }
    int64_t G = (int64_t)sm_count() * per_sm;
    if (!coop && G > max_units) G = max_units;  // a lone op never needs idle CTAs
    if (G < 1) G = 1;
    float *part = reinterpret_cast<float *>(ws);
    unsigned *cnt = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(ws) +
                                                 partial_region_bytes());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(NW * 32);
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
    return cudaLaunchKernelEx(&cfg, kern, P, part, cnt);
}

template <int MAXOPS>
static void set_shift_multipliers(VlOps<MAXOPS> &P) {
    P.m4 = 1u << 28;
    P.m8 = 1u << 24;
    P.m12 = 1u << 20;
}

static VlOp make_op(const svd_qweight *W, const void *X, float *Y) {
    const NativeGeom ng = native_geom(W->in_features, W->out_features);
    VlOp o;
    o.codes = reinterpret_cast<const uint8_t *>(W->codes);
    o.scales = reinterpret_cast<const uint8_t *>(W->scales);
    o.X = reinterpret_cast<const __nv_bfloat16 *>(X);
    o.Y = Y;
    o.in_f = W->in_features;
    o.out_f = W->out_features;
    o.n_kc = ng.n_kc;
    o.n_units = ng.n_units;
    return o;
}

template <int MAXOPS>
static cudaError_t launch_ops(const VlOps<MAXOPS> &P, void *ws, bool pdl, cudaStream_t stream) {
    int64_t max_units = 0;
    for (int i = 0; i < P.n; ++i) max_units = P.op[i].n_units > max_units ? P.op[i].n_units : max_units;
    const bool coop = P.n > 1;
    switch (ntiles_for(P.C)) {
        case 1: return launch_mma<1, kD1, MAXOPS>(P, ws, pdl, coop, max_units, stream);
        case 2: return launch_mma<2, kD2, MAXOPS>(P, ws, pdl, coop, max_units, stream);
        default: return launch_mma<4, kD2, MAXOPS>(P, ws, pdl, coop, max_units, stream);
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
    if (!W || !W->codes || !W->scales) return SVD_ERR_INVALID_ARG;
    if (W->in_features <= 0 || W->out_features <= 0 || W->in_features % 32 != 0)
        return SVD_ERR_INVALID_ARG;
    if (W->reserved != 0) return SVD_ERR_INVALID_ARG;
    if (W->layout != SVD_LAYOUT_CANONICAL && W->layout != SVD_LAYOUT_NATIVE)
        return SVD_ERR_INVALID_ARG;
    if (!aligned16(W->codes) || !aligned16(W->scales)) return SVD_ERR_INVALID_ARG;
    return SVD_OK;
}

int verify_linear(const svd_qweight *W, const void *X, int C, float *Y, void *ws,
                  size_t ws_bytes, int flags, cudaStream_t stream) {
    int rc = check_qweight(W);
    if (rc != SVD_OK) return rc;
    if (!X || !Y || C < 1 || C > SVD_C_MAX || !aligned16(X)) return SVD_ERR_INVALID_ARG;
    if (flags & ~SVD_F_PDL) return SVD_ERR_INVALID_ARG;
    const bool pdl = (flags & SVD_F_PDL) != 0;
    if (sm_count() < 1) return SVD_ERR_CUDA;
    if (W->layout == SVD_LAYOUT_NATIVE) {
        if (!ws || ws_bytes < vl_workspace_bytes(W->in_features, W->out_features, C))
            return SVD_ERR_WORKSPACE;
        VlOps<1> P;
        P.n = 1;
        P.C = C;
        set_shift_multipliers(P);
        P.op[0] = make_op(W, X, Y);
        SVD_CUDA_TRY(launch_ops(P, ws, pdl, stream));
        return SVD_OK;
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

size_t chain_workspace_bytes(const svd_linear_op *ops, int n_ops, int C) {
    int64_t n_rb = 1;
    for (int i = 0; i < n_ops; ++i) {
        const NativeGeom ng = native_geom(ops[i].W.in_features, ops[i].W.out_features);
        n_rb = ng.n_rb > n_rb ? ng.n_rb : n_rb;
    }
    (void)C;
    return partial_region_bytes() + align_up((size_t)n_rb * sizeof(unsigned), 256);
}

int verify_chain(const svd_linear_op *ops, int n_ops, int C, void *ws, size_t ws_bytes, int flags,
                 cudaStream_t stream) {
    if (!ops || n_ops < 1 || C < 1 || C > SVD_C_MAX) return SVD_ERR_INVALID_ARG;
    if (flags & ~SVD_F_PDL) return SVD_ERR_INVALID_ARG;
    for (int i = 0; i < n_ops; ++i) {
        const int rc = check_qweight(&ops[i].W);
        if (rc != SVD_OK) return rc;
        if (ops[i].W.layout != SVD_LAYOUT_NATIVE) return SVD_ERR_INVALID_ARG;
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
            set_shift_multipliers(P1);
            P1.op[0] = make_op(&ops[first].W, ops[first].X, ops[first].Y);
            SVD_CUDA_TRY(launch_ops(P1, ws, first == 0 && (flags & SVD_F_PDL), stream));
            continue;
        }
        P.n = n;
        P.C = C;
        set_shift_multipliers(P);
        for (int i = 0; i < n; ++i) P.op[i] = make_op(&ops[first + i].W, ops[first + i].X, ops[first + i].Y);
        SVD_CUDA_TRY(launch_ops(P, ws, false, stream));
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

int repack(const svd_qweight *src, void *dc, void *ds, cudaStream_t stream) {
    int rc = check_qweight(src);
    if (rc != SVD_OK) return rc;
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

// ---- verify linear without caller scratch ----------------------------------------------
// The stream-K kernel needs a small scratch area (partial sums of row blocks split between
// CTAs, and one ticket counter per 64-row block).  svd_verify_linear takes it from the caller;
// this variant takes it from a fixed array in the library's own device memory instead, for
// callers that cannot allocate device memory.  The array is reserved when the library's
// module is loaded on a device and stays there until the process exits.
constexpr int kNoAllocMaxSms = 160;
constexpr int64_t kNoAllocMaxRowBlocks = SVD_NOALLOC_MAX_OUT_FEATURES / kRowsPerBlock;
constexpr size_t kNoAllocPartialBytes =
    (size_t)kNoAllocMaxSms * kMaxCtasPerSm * 2 * kPartialSlotFloats * sizeof(float);
constexpr size_t kNoAllocBytes = kNoAllocPartialBytes + kNoAllocMaxRowBlocks * sizeof(unsigned);
static_assert(kNoAllocBytes <= SVD_NOALLOC_SCRATCH_BYTES, "scratch bound in svd.h");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch, looked up once per device with that device current
// (in host code the symbol is only a host-side handle and must never reach a kernel).
static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[64] = {nullptr};

int verify_linear_noalloc(const svd_qweight *W, const void *X, int C, float *Y, int flags,
                          cudaStream_t stream) {
    int rc = check_qweight(W);
    if (rc != SVD_OK) return rc;
    if (W->layout != SVD_LAYOUT_NATIVE) return SVD_ERR_INVALID_ARG;
    if (!X || !Y || C < 1 || C > SVD_C_MAX || !aligned16(X)) return SVD_ERR_INVALID_ARG;
    if (flags & ~SVD_F_PDL) return SVD_ERR_INVALID_ARG;
    if (W->out_features > SVD_NOALLOC_MAX_OUT_FEATURES) return SVD_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms < 1) return SVD_ERR_CUDA;
    if (sms > kNoAllocMaxSms) return SVD_ERR_UNSUPPORTED;
    int dev = 0;
    SVD_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return SVD_ERR_UNSUPPORTED;
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            SVD_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
            g_noalloc_ptr[dev] = p;
        }
        base = g_noalloc_ptr[dev];
    }
    // Same layout as a caller workspace: partial slots, then the tickets, which must start at
    // zero.  Every call clears them again on the stream before its kernel, so a call never
    // depends on what the previous one left behind.
    const NativeGeom ng = native_geom(W->in_features, W->out_features);
    unsigned char *tickets = reinterpret_cast<unsigned char *>(base) + partial_region_bytes();
    SVD_CUDA_TRY(cudaMemsetAsync(tickets, 0, (size_t)ng.n_rb * sizeof(unsigned), stream));
    VlOps<1> P;
    P.n = 1;
    P.C = C;
    set_shift_multipliers(P);
    P.op[0] = make_op(W, X, Y);
    SVD_CUDA_TRY(launch_ops(P, base, (flags & SVD_F_PDL) != 0, stream));
    return SVD_OK;
}

}  // namespace svd

