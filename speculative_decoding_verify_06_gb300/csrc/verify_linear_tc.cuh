// verify_linear_tc.cuh -- the batched verify GEMM (17..32 activation columns) on the fifth-
// generation tensor cores: tcgen05.mma with fp32 accumulators in tensor memory.
//
// "100 tokens per second from a 27B model on a 24 GB AMD card", section "Why a hiring company
// is writing this", and "Decode is memory-bound ...", section "Rules I use" (rule 2): batching
// several sequences' windows amortises the one weight read of a pass over more columns.  At
// C = 32 the legacy fragment path pays one fp32 FMA per weight for the per-block rescale and
// reloads every activation fragment per warp; here the block scale is folded into the A operand
// and the activations are converted once per op and staged per block in shared memory, where
// the tensor core reads them.
//
// Arithmetic.  A = fp16(s * (c - 8)): (c - 8) is built exactly from the exponent pattern 0x6400
// (1024 + c, minus 1032), then multiplied by the block's fp16 scale with one rounding (relative
// error <= 2^-11 per weight).  B = the activations rounded from bf16 to fp16 (exact for
// |x| in [2^-14, 65504]; smaller values become fp16 subnormals, absolute error <= 2^-25).  The
// products are accumulated in fp32 in tensor memory.  The error per output is therefore at most
// 2^-11 * sum |w x| plus fp32 accumulation and the subnormal term, inside the 1e-3 * sum |w x|
// bound of the verify GEMM.
//
// Decomposition.  An MMA unit is 128 weight rows (native row blocks 2q and 2q+1) x one 64-input
// chunk; units are ordered row-group-major, and the grid splits them into contiguous ranges,
// one per CTA (stream-K).  A CTA runs three PIPES of four warps, each with an MMA warp.  The CTA's
// range is cut into blocks of up to two units of one row group, dealt to the pipes round-robin.
// At the start of each op all CTAs convert the op's activations from bf16 into fp16 B tiles
// in the workspace (a share of the chunks each) and pass a grid barrier.  A pipe streams its
// blocks through a ring of two slots (per block four bulk copies of weights, one per warp: the
// codes and the scales of the two row blocks, and one of the block's B tiles); its warps
// dequantise each unit into an fp16 A stage (warp j: rows 32j..32j+31) and arrive on the stage's
// barrier.  The pipe's MMA warp takes its stages in order and issues four tcgen05.mma (M 128,
// N 32, K 16) per stage into the pipe's accumulator (32 TMEM columns; two sets, by the parity of
// the row-group segment).  When a
// segment (one row group of the range) is done, the pipes' warps add the accumulators of the
// segment in pipe order -- pipe p takes token groups p and p + 3 (8 TMEM columns each), warp j
// of a pipe rows 32j..32j+31 (its TMEM lane quarter) -- and write Y, or store a tagged partial
// if an earlier CTA owns the row group; the owner adds the later CTAs' partials in CTA order.
// Summation order is fixed: results are deterministic.
//
// Every wait is bounded (the WaitCtl of the stream-K kernel): a wait that runs out sets a status
// bit, later waits return at once, and before exiting the CTA waits a bounded time for its
// tensor-core operations and bulk copies.
//
// Included by verify_linear.cu inside namespace svd, after the stream-K kernel whose op
// descriptors, partial tags and bounded waits it shares.
#pragma once

constexpr int kTcPipes = 3;           // pipes per CTA
constexpr int kTcPipeWarps = 4;       // warps per pipe (one per TMEM lane quarter)
constexpr int kTcMmaWarp = kTcPipes * kTcPipeWarps;   // first of the pipes' MMA warps
constexpr int kTcThreads = (kTcMmaWarp + kTcPipes) * 32;
constexpr int kTcU = 2;               // units per block (per bulk copy)
constexpr int kTcR = 2;               // ring slots per pipe
constexpr int kTcS = 2;               // A stages per pipe
constexpr int kTcN = 32;              // MMA N: activation columns
constexpr int kTcRows = 2 * kRowsPerBlock;            // MMA M: 128 weight rows
constexpr int kTcAStage = kTcRows * kChunk * 2;       // 128 rows x 64 inputs fp16
constexpr int kTcBTile = kTcN * kChunk * 2;           // 32 tokens x 64 inputs fp16 (one chunk)
// a ring slot: the B tiles of the block's units, then the codes of its two row blocks, then
// their scales
constexpr int kTcSlotCodes = kTcU * kTcBTile;
constexpr int kTcSlotScales = kTcSlotCodes + 2 * kTcU * kUnitCodeBytes;
constexpr int kTcSlotBytes = kTcSlotScales + 2 * kTcU * kUnitScaleBytes;
// per pipe: the A stages, then the ring (all 1024-byte aligned for the swizzle)
constexpr int kTcPipeBytes = kTcS * kTcAStage + kTcR * kTcSlotBytes;
constexpr int kTcAccCols = kTcN;                      // TMEM columns per accumulator
constexpr uint32_t kTcTmemCols = 256;                 // kTcPipes * 2 * kTcAccCols, rounded to 2^k
constexpr int kTcPartial = kTcRows * kTcN;            // entries of a CTA's partial
static_assert(kTcPartial <= 2 * kPartialMax, "a tensor-core CTA uses two stream-K partial slots");
static_assert(kRowsPerBlock == 64 && kChunk == 64, "the MMA unit is two 64-row native blocks x 64 inputs");
static_assert(kTcPipes * 2 * kTcAccCols <= (int)kTcTmemCols, "accumulators fit the allocation");
static_assert(kTcPipeBytes % 1024 == 0 && kTcAStage % 1024 == 0 && kTcSlotBytes % 1024 == 0 &&
                  kTcBTile % 1024 == 0,
              "stages and B tiles stay on the swizzle's 1024-byte period");

// The fp16 B layout of an op's activations (one 4 KB tile per 64-input chunk, written once per
// op into the workspace and bulk-copied with each block's weights): token n at 128 n, the
// inputs 32 h + 8 t .. + 7 of the chunk (scale block h) in piece 2 t + h, stored at piece
// (2 t + h) ^ (n & 7) -- the 128-byte swizzle, and the permutation that makes the A stores
// conflict-free.
__host__ __device__ constexpr size_t tc_xb_bytes(int64_t in_f) {
    return (size_t)((in_f + kChunk - 1) / kChunk) * kTcBTile;
}

template <int MAXOPS>
struct TcCfg {
    // + 1 KB to align the stages to the 1024-byte period of the 128-byte swizzle
    static constexpr size_t kSmem = (size_t)kTcPipes * kTcPipeBytes + (size_t)MAXOPS * sizeof(VlOp) + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

// ---- tcgen05 / TMEM -----------------------------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand stored with the 128-byte swizzle: each row
// holds 64 fp16 inputs (128 bytes), row r at 128 r, and its 16-byte piece c sits at piece
// c ^ (r & 7) (address bits 4-6 XOR bits 7-9).  Fields: start >> 4, leading offset (unused by
// swizzled K-major layouts) >> 4 at bit 16, stride between 8-row groups (8 x 128 = 1024 bytes)
// >> 4 at bit 32, the descriptor version bit 46, layout 2 (128-byte swizzle) at bits 61-63.  The
// operand must lie in a 1024-byte-aligned region; a K step of 16 advances the start by 32 bytes.
__device__ __forceinline__ uint64_t tc_sdesc_sw128(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(16u >> 4) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B fp16 (bits 7-9, 10-12 =
// 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t tc_idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The mbarrier completes one arrival when every tcgen05 operation this thread issued before has
// completed.
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Eight consecutive TMEM columns of the warp's 32 lanes (one row per lane).
__device__ __forceinline__ void tc_ld8(uint32_t taddr, uint32_t v[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Four fp16x2 A values from one native word (see native_word_coords): register p of the word
// holds rows g (p even) / g + 8 (p odd), inputs 2 (p >> 1) + h.  Nibbles at bits 0-3 | 16-19
// give 1024 + c exactly under the pattern 0x6400, minus 1032 = c - 8; nibbles at bits 4-7 |
// 20-23 give 1024 + 16 c, times 1/16 minus 72 = c - 8 (exact); the shifted word gives p = 2, 3
// the same way.  Each is then scaled by its row's block scale with one fp16 rounding.
__device__ __forceinline__ void dequant_word_f16(uint32_t w, uint32_t s_g, uint32_t s_g8, uint32_t o[4]) {
    const uint32_t magic = 0x64006400u;
    const uint32_t w8 = w >> 8;
    uint32_t v0, v1, v2, v3;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v0) : "r"(w), "r"(0x000F000Fu), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v1) : "r"(w), "r"(0x00F000F0u), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v2) : "r"(w8), "r"(0x000F000Fu), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v3) : "r"(w8), "r"(0x00F000F0u), "r"(magic));
    const uint32_t bias = 0x64086408u;      // (1032, 1032)
    const uint32_t sixteenth = 0x2C002C00u;  // (1/16, 1/16)
    const uint32_t m72 = 0xD480D480u;        // (-72, -72)
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(v0) : "r"(bias));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(v1) : "r"(sixteenth), "r"(m72));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(v2) : "r"(bias));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(v3) : "r"(sixteenth), "r"(m72));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[0]) : "r"(v0), "r"(s_g));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[1]) : "r"(v1), "r"(s_g8));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[2]) : "r"(v2), "r"(s_g));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[3]) : "r"(v3), "r"(s_g8));
}
// Two bf16 (one word) to two fp16, round to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- schedule ----------------------------------------------------------------------------
// MMA units of an op (row groups of 128 rows x chunks), the CTA's contiguous range of them, and
// the CTA holding unit u.  n_units * (CTAs + 1) < 2^32 is checked on the host.
__device__ __forceinline__ uint32_t tc_units(const VlOp &o) {
    const uint32_t n_rb = o.n_units / o.n_kc;
    return ((n_rb + 1u) / 2u) * o.n_kc;
}
__device__ __forceinline__ void tc_range(const VlOp &o, uint32_t G, uint32_t b, uint32_t *lo, uint32_t *hi) {
    const uint32_t n = tc_units(o), Gop = min(G, n);
    if (b < Gop) {
        *lo = b * n / Gop;
        *hi = (b + 1u) * n / Gop;
    } else {
        *lo = *hi = 0u;
    }
}
__device__ __forceinline__ uint32_t tc_cta_of(const VlOp &o, uint32_t G, uint32_t u) {
    const uint32_t n = tc_units(o), Gop = min(G, n);
    return ((u + 1u) * Gop - 1u) / n;
}
// A SEGMENT is the part of the CTA's range inside one row group: [s0, s1).  Its blocks (up to
// kTcU units each) are numbered on from cb, the CTA's blocks before it, and block cb + j goes to
// pipe (cb + j) mod kTcPipes.  First block of pipe p in a segment:
__device__ __forceinline__ uint32_t tc_first_block(uint32_t p, uint32_t cb) {
    return (p + kTcPipes - cb % kTcPipes) % kTcPipes;
}
__device__ __forceinline__ uint32_t tc_blocks(uint32_t s0, uint32_t s1) {
    return (s1 - s0 + kTcU - 1u) / kTcU;
}

// A pipe's blocks in order, across the segments and ops of the launch (the copy cursor, run
// ahead of the consumer; it walks exactly the consumer's loops).
struct TcIter {
    int op;               // current op; n_ops when exhausted
    uint32_t lo, hi;      // the CTA's range of that op
    uint32_t s0, s1, rg;  // current segment and its row group
    uint32_t jb, nb, cb;  // next block of this pipe in the segment, blocks in it, blocks before it

    __device__ __forceinline__ void start() {
        op = -1;
        lo = hi = s0 = s1 = rg = 0u;
        jb = nb = cb = 0u;
    }
    // Next block of pipe p: op index, first unit, unit count and row group; false when there is
    // none.
    __device__ __forceinline__ bool next(uint32_t p, const VlOp *ops, int n_ops, uint32_t G, uint32_t b,
                                         int *op_out, uint32_t *u0, uint32_t *n, uint32_t *rg_out) {
        for (;;) {
            if (op >= n_ops) return false;
            if (op >= 0 && jb < nb) {
                *op_out = op;
                *u0 = s0 + kTcU * jb;
                *n = min((uint32_t)kTcU, s1 - *u0);
                *rg_out = rg;
                jb += kTcPipes;
                return true;
            }
            cb += nb;
            nb = 0u;
            if (op >= 0 && s1 < hi) {
                const uint32_t n_kc = ops[op].n_kc;
                s0 = s1;
                rg = s0 / n_kc;
                s1 = min(hi, (rg + 1u) * n_kc);
                nb = tc_blocks(s0, s1);
                jb = tc_first_block(p, cb);
                continue;
            }
            if (++op >= n_ops) return false;
            tc_range(ops[op], G, b, &lo, &hi);
            s0 = s1 = lo;
        }
    }
};

// One segment awaiting its epilogue.
struct TcSeg {
    uint32_t s0, s1, rg, cb, nb, k;
};

// What a pipe's stage holds, written by its warp 0 for the MMA warp: flags in bits 0-3, the
// segment number k above them.
constexpr uint32_t kTcMetaMma = 1u;     // a unit: issue its four MMAs
constexpr uint32_t kTcMetaFirst = 2u;   // the pipe's first unit of the segment: start the accumulator
constexpr uint32_t kTcMetaSegEnd = 4u;  // the pipe's last stage of the segment: signal its accumulator
constexpr uint32_t kTcMetaEnd = 8u;     // the pipe has no more stages
constexpr uint32_t kTcMetaBlockEnd = 16u;  // the block's last unit: its ring slot's B tiles are free after
constexpr int kTcMetaSlotShift = 5;     // ring slot of the unit (its B tile), 1 bit
constexpr int kTcMetaUnitShift = 6;     // unit within the block, 1 bit
constexpr int kTcMetaKShift = 8;        // segment number

template <int MAXOPS>
__global__ void __launch_bounds__(kTcThreads, 1)
vl_tc_kernel(const __grid_constant__ VlOps<MAXOPS> P, unsigned long long *__restrict__ part,
             uint32_t part_entries, unsigned *__restrict__ gbar, uint8_t *__restrict__ xb) {
    extern __shared__ __align__(128) uint8_t smem[];  // aligned to 1 KB below
    __shared__ __align__(8) uint64_t s_full[kTcPipes * kTcR];   // a ring slot's copies landed
    __shared__ __align__(8) uint64_t s_stage[kTcPipes * kTcS];  // a stage is written (its 4 warps)
    __shared__ __align__(8) uint64_t s_bfree[kTcPipes * kTcR];  // a slot's B tiles have been read
    __shared__ __align__(8) uint64_t s_empty[kTcPipes * kTcS];  // a stage's MMAs have read it
    __shared__ __align__(8) uint64_t s_done[kTcPipes * 2];      // a pipe's MMAs of a segment (per set)
    __shared__ __align__(8) uint64_t s_free[2];                 // a set's accumulators have been read
    __shared__ __align__(8) uint64_t s_final[kTcPipes];         // every MMA of a pipe, at exit
    __shared__ uint32_t s_meta[kTcPipes * kTcS];
    __shared__ uint32_t s_bblk[kTcPipes * kTcR][3];             // a slot's block: op, first chunk, units
    __shared__ uint32_t s_tmem, s_epoch, s_last;
    __shared__ WaitCtl s_wc;
    uint8_t *const sm0 = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
    VlOp *ops = reinterpret_cast<VlOp *>(sm0 + (size_t)kTcPipes * kTcPipeBytes);
    const int n_ops = P.n;
    const int C = P.C;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool mma_warp = warp >= kTcMmaWarp;  // warp kTcMmaWarp + p issues pipe p's MMAs
    const uint32_t pipe = mma_warp ? (uint32_t)(warp - kTcMmaWarp) : (uint32_t)warp / kTcPipeWarps;
    const int wj = warp % kTcPipeWarps;  // warp in the pipe = its TMEM lane quarter
    const uint32_t G = gridDim.x, b = blockIdx.x;
    uint8_t *const ring = sm0 + (size_t)pipe * kTcPipeBytes + kTcS * kTcAStage;
    const uint32_t astage0 = smem_u32(sm0) + pipe * kTcPipeBytes;
    const uint32_t ring0 = smem_u32(ring);
    const uint32_t full0 = smem_u32(&s_full[pipe * kTcR]);
    const uint32_t stage0 = smem_u32(&s_stage[pipe * kTcS]);
    const uint32_t empty0 = smem_u32(&s_empty[pipe * kTcS]);

    {
        static_assert(sizeof(VlOp) % 8 == 0, "op descriptor copied in 8-byte words");
        const uint64_t *src = reinterpret_cast<const uint64_t *>(&P.op[0]);
        uint64_t *dst = reinterpret_cast<uint64_t *>(ops);
        for (int i = threadIdx.x; i < n_ops * (int)(sizeof(VlOp) / 8); i += kTcThreads) dst[i] = src[i];
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcPipes * kTcR; ++i) {
            mbar_init(smem_u32(&s_full[i]), kTcPipeWarps + 1);  // four weight parts and the B tiles
            mbar_init(smem_u32(&s_bfree[i]), 1);
        }
        for (int i = 0; i < kTcPipes * kTcS; ++i) {
            mbar_init(smem_u32(&s_stage[i]), kTcPipeWarps);
            mbar_init(smem_u32(&s_empty[i]), 1);
        }
        for (int i = 0; i < kTcPipes * 2; ++i) mbar_init(smem_u32(&s_done[i]), 1);
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&s_free[i]), kTcMmaWarp);
        for (int i = 0; i < kTcPipes; ++i) mbar_init(smem_u32(&s_final[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_wc.stop = 0u;
    }
    __syncthreads();

    // Copy cursor of a pipe (uniform across its warps).  Warp wj copies one part of every block:
    // the codes (wj even) or the scales (wj odd) of row block 2q + (wj >> 1), which are read by
    // warps wj & ~1 and wj | 1 only; a row block past the matrix's end is not copied (its rows
    // are never stored).  Warp 1 also copies the block's B tiles, but only once its op's
    // activations have been converted (the weights of later ops stream ahead of that) and the
    // MMAs of the block that used the slot before have read its B tiles.
    TcIter it;
    it.start();
    uint32_t c_issued = 0, b_next = 0;  // blocks whose weights / B tiles have been issued
    int conv_op = -1;                   // ops up to this one have their B layout in the workspace
    auto issue_b = [&]() {
        while (b_next < c_issued) {
            const uint32_t slot = b_next % kTcR;
            const uint32_t *bi = s_bblk[pipe * kTcR + slot];
            if ((int)bi[0] > conv_op) return;
            if (b_next >= (uint32_t)kTcR)
                slot_wait(smem_u32(&s_bfree[pipe * kTcR + slot]), ((b_next / kTcR) - 1u) & 1u, &s_wc);
            if (lane == 0) {
                const uint32_t bar = full0 + 8u * slot, bytes = bi[2] * (uint32_t)kTcBTile;
                mbar_expect_tx(bar, bytes);
                bulk_g2s(ring0 + slot * kTcSlotBytes, xb + (size_t)bi[1] * kTcBTile, bytes, bar);
            }
            ++b_next;
        }
    };
    auto issue = [&]() {
        int op;
        uint32_t u0, n, rg;
        if (!it.next(pipe, ops, n_ops, G, b, &op, &u0, &n, &rg)) return;
        const VlOp &o = ops[op];
        const uint32_t slot = c_issued % kTcR, bar = full0 + 8u * slot;
        const uint32_t kc = u0 - rg * o.n_kc;
        if (lane == 0) {
            const uint32_t h = (uint32_t)wj >> 1, rb = 2u * rg + h;
            if ((uint64_t)rb * o.n_kc < o.n_units) {
                const size_t nu = (size_t)rb * o.n_kc + kc;  // native unit index
                uint32_t dst, bytes;
                const uint8_t *src;
                if ((wj & 1) == 0) {
                    bytes = n * kUnitCodeBytes;
                    dst = ring0 + slot * kTcSlotBytes + kTcSlotCodes + h * (kTcU * kUnitCodeBytes);
                    src = o.codes + nu * kUnitCodeBytes;
                } else {
                    bytes = n * kUnitScaleBytes;
                    dst = ring0 + slot * kTcSlotBytes + kTcSlotScales + h * (kTcU * kUnitScaleBytes);
                    src = o.scales + nu * kUnitScaleBytes;
                }
                mbar_expect_tx(bar, bytes);
                bulk_g2s(dst, src, bytes, bar);
            } else {
                mbar_arrive(bar);
            }
            if (wj == 1) {
                s_bblk[pipe * kTcR + slot][0] = (uint32_t)op;
                s_bblk[pipe * kTcR + slot][1] = kc;
                s_bblk[pipe * kTcR + slot][2] = n;
            }
        }
        __syncwarp();
        ++c_issued;
        if (wj == 1) issue_b();
    };
    if (!mma_warp) {
        // The stall injection (workspace word kBarPoll, written only by the test hook): no copy.
        if (*reinterpret_cast<volatile unsigned *>(gbar + kBarPoll) != 0u) it.op = n_ops;
        // weights never depend on earlier kernels: start streaming before waiting for them
        for (int i = 0; i < kTcR; ++i) issue();
    }

    griddep_wait();
    griddep_launch_dependents();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        s_epoch = *reinterpret_cast<volatile unsigned *>(gbar + kBarEpoch);
        const unsigned lim = *reinterpret_cast<volatile unsigned *>(gbar + kBarPoll);
        s_wc.limit = lim ? lim - 1u : kPollLimit;
        s_wc.status = gbar + kBarStatus;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem, epoch = s_epoch;

    if (mma_warp) {
        // ---- a pipe's MMA warp: the pipe's stages in order -------------------------------
        // (blocking waits are safe here: a pipe's warps never wait on another pipe's MMA warp,
        // and the epilogue of segment k - 2 that segment k waits for needs only the MMAs of
        // segments up to k - 2, all issued before)
        constexpr uint32_t kIdesc = tc_idesc_f16(kTcRows, kTcN);
        const uint32_t abase0 = astage0, ring00 = ring0;
        uint32_t ctr = 0u, kfree = 1u;  // segments up to kfree need no wait for a free set
        for (;;) {
            const uint32_t st = ctr % kTcS;
            if (!slot_wait(stage0 + 8u * st, (ctr / kTcS) & 1u, &s_wc)) break;
            const uint32_t meta = *reinterpret_cast<volatile uint32_t *>(&s_meta[pipe * kTcS + st]);
            if (meta & kTcMetaEnd) break;
            const uint32_t k = meta >> kTcMetaKShift, set = k & 1u;
            const uint32_t slot = (meta >> kTcMetaSlotShift) & 1u, unit = (meta >> kTcMetaUnitShift) & 1u;
            // segment k reuses set k & 1: the epilogue of segment k - 2 must have read it
            if (k > kfree) {
                slot_wait(smem_u32(&s_free[set]), ((k >> 1) - 1u) & 1u, &s_wc);
                kfree = k;
            }
            if (lane == 0) {
                tc_fence_after();
                if (meta & kTcMetaMma) {
                    const uint32_t dcol = tmem + (pipe * 2u + set) * kTcAccCols;
                    const uint64_t da = tc_sdesc_sw128(abase0 + st * kTcAStage);
                    const uint64_t db = tc_sdesc_sw128(ring00 + slot * kTcSlotBytes + unit * kTcBTile);
                    const uint32_t acc0 = (meta & kTcMetaFirst) ? 0u : 1u;
#pragma unroll
                    for (uint32_t kq = 0; kq < 4; ++kq)  // K step of 16 = 32 bytes = 2 in the start field
                        tc_mma_f16(dcol, da + 2u * kq, db + 2u * kq, kIdesc, kq ? 1u : acc0);
                }
                tc_commit(empty0 + 8u * st);
                if (meta & kTcMetaBlockEnd) tc_commit(smem_u32(&s_bfree[pipe * kTcR + slot]));
                if (meta & kTcMetaSegEnd) tc_commit(smem_u32(&s_done[pipe * 2u + set]));
            }
            __syncwarp();
            ++ctr;
        }
        // every tensor-core operation of the pipe complete before the accumulators are released
        if (lane == 0) {
            tc_commit(smem_u32(&s_final[pipe]));
            mbar_wait_ok(smem_u32(&s_final[pipe]), 0u);
        }
        __syncwarp();
    } else {
        // ---- the pipes: copies, dequantisation, activations, epilogues ----
        const int g4 = lane >> 2, t4 = lane & 3;
        const int hrb = wj >> 1;       // this warp's row block in the MMA unit (rows 32 wj .. 32 wj + 31)
        const int t0 = 2 * (wj & 1);   // its first 16-row tile there
        // This lane's places in a stage (128-byte swizzle: row R at 128 R, piece c at c ^ (R & 7)).
        // A: row g of tile t0 + r is R = 64 hrb + 16 (t0 + r) + g (so R & 7 = g), row g + 8 is 1024
        // bytes further; its inputs 32 hc + 8 t4 .. + 7 (scale block hc) go to piece 2 t4 + hc, so
        // that the two rows a quarter-warp stores cover eight distinct bank groups.  The B tiles
        // use the same pieces (tc_xb_bytes), so the MMA's k-th 16 inputs (pieces 2k and 2k + 1)
        // are inputs 8k .. 8k + 7 and 32 + 8k .. 32 + 8k + 7 of the chunk in A and B alike.
        const uint32_t a_row = (uint32_t)(64 * hrb + 16 * t0 + g4) * 128u;
        const uint32_t pc0 = (uint32_t)((2 * t4) ^ g4) * 16u, pc1 = (uint32_t)((2 * t4 + 1) ^ g4) * 16u;
        uint32_t nbar = 0;  // grid barriers passed
        constexpr uint32_t kQuarter = 1u << 16;  // TMEM lane field
        const uint32_t pair_bar = 1u + pipe * 2u + (uint32_t)hrb;  // the two warps of one row block
        uint32_t k = 0, cb = 0, stage_ctr = 0, slot_ctr = 0;

        // the next stage of this pipe, once the MMAs that read it last are done
        auto stage_begin = [&]() {
            const uint32_t st = stage_ctr % kTcS;
            if (stage_ctr >= (uint32_t)kTcS) slot_wait(empty0 + 8u * st, ((stage_ctr / kTcS) - 1u) & 1u, &s_wc);
            return st;
        };
        // hands a written stage to the MMA warp
        auto post = [&](uint32_t st, uint32_t meta) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (wj == 0) s_meta[pipe * kTcS + st] = meta;
                mbar_arrive(stage0 + 8u * st);
            }
            ++stage_ctr;
        };

        // a barrier of the pipes' warps (the MMA warps run on), then of the grid
        auto grid_sync = [&]() {
            asm volatile("bar.sync 15, %0;" ::"r"(kTcMmaWarp * 32) : "memory");
            ++nbar;
            if (threadIdx.x == 0) grid_barrier(gbar + kBarCount, nbar * G, &s_wc);
            asm volatile("bar.sync 15, %0;" ::"r"(kTcMmaWarp * 32) : "memory");
        };
        for (int gi = 0; gi < n_ops; ++gi) {
            const VlOp &o = ops[gi];
            if (gi > 0) grid_sync();  // op gi - 1 has written its outputs
            const uint32_t n_kc = o.n_kc;
            const int64_t in_f = o.in_f, out_f = o.out_f;
            const uint32_t tag = (partial_epoch24(epoch) << 8) | (uint32_t)(gi & 255);
            // This CTA's share of the op's B tiles: chunks [G0, G1), one 16-byte piece (8
            // activations of one token) per thread and step, zero past C or in_f.  The generic
            // writes are fenced against the bulk copies (async proxy) that read them after the
            // grid barrier.
            {
                const uint32_t k0 = (uint32_t)((uint64_t)b * n_kc / G), k1 = (uint32_t)((uint64_t)(b + 1) * n_kc / G);
                for (uint32_t idx = threadIdx.x; idx < (k1 - k0) * 256u; idx += kTcMmaWarp * 32) {
                    const uint32_t kc = k0 + idx / 256u, n = (idx / 8u) % 32u, p16 = idx % 8u;
                    const int64_t col = (int64_t)kc * kChunk + 8 * p16;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if ((int)n < C && col < in_f) {
                        const __nv_bfloat16 *src = o.X + (int64_t)n * in_f + col;
                        if constexpr (MAXOPS > 1) v = ldg_cg_v4(src);
                        else v = ldg_nc_v4(src);
                    }
                    const uint32_t pc = 2u * (p16 & 3u) + (p16 >> 2);
                    *reinterpret_cast<uint4 *>(xb + (size_t)kc * kTcBTile + n * 128u + ((pc ^ (n & 7u)) * 16u)) =
                        make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                                   bf16x2_to_f16x2(v.w));
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            grid_sync();  // every CTA's share of the B tiles is written
            conv_op = gi;
            if (wj == 1) issue_b();  // the B tiles of this op's blocks already in flight
            uint32_t lo, hi;
            tc_range(o, G, b, &lo, &hi);

            // Epilogue of a segment: the pipes' accumulators of its set added in pipe order, then
            // Y -- or a tagged partial when an earlier CTA owns the row group; an owner whose row
            // group runs on into later CTAs adds their partials in CTA order (only at the end of
            // its range).  This pipe takes token groups pipe and pipe + kTcPipes (8 columns each).
            auto epilogue = [&](const TcSeg &sg) {
                const uint32_t set = sg.k & 1u;
                for (uint32_t pp = 0; pp < (uint32_t)kTcPipes; ++pp)
                    slot_wait(smem_u32(&s_done[pp * 2u + set]), (sg.k >> 1) & 1u, &s_wc);
                tc_fence_after();
                float v[2][8];
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[gq][e] = 0.f;
                    const uint32_t cg = pipe + (uint32_t)gq * kTcPipes;
                    if (cg >= (uint32_t)(kTcN / 8) || (int)(8 * cg) >= C) continue;
                    for (uint32_t pp = 0; pp < (uint32_t)kTcPipes; ++pp) {
                        if (tc_first_block(pp, sg.cb) >= sg.nb) continue;  // no block of pipe pp here
                        uint32_t r[8];
                        tc_ld8(tmem + (uint32_t)wj * 32u * kQuarter + (pp * 2u + set) * kTcAccCols + 8u * cg, r);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[gq][e] += __uint_as_float(r[e]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s_free[set]));

                const uint32_t rl = 32u * (uint32_t)wj + (uint32_t)lane;
                const int64_t row = (int64_t)sg.rg * kTcRows + rl;
                const bool owner = sg.s0 == sg.rg * n_kc, whole = sg.s1 == (sg.rg + 1u) * n_kc;
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    const uint32_t cg = pipe + (uint32_t)gq * kTcPipes;
                    const int c0 = 8 * (int)cg;
                    if (cg >= (uint32_t)(kTcN / 8) || c0 >= C) continue;
                    if (!owner) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (c0 + e < C)
                                st_tagged(part + (size_t)b * kTcPartial + (size_t)(c0 + e) * kTcRows + rl, v[gq][e], tag);
                    } else if (row < out_f) {
                        if (!whole) {
                            // the later CTAs' partials, two CTAs at a time: all sixteen loads in
                            // flight together, the missing ones polled together, then added in
                            // CTA order
                            const uint32_t b_last = tc_cta_of(o, G, (sg.rg + 1u) * n_kc - 1u);
                            for (uint32_t bb = b + 1u; bb <= b_last; bb += 2u) {
                                const bool two = bb + 1u <= b_last;
                                const unsigned long long *src = part + (size_t)bb * kTcPartial + rl;
                                unsigned long long w[2][8];
                                uint32_t pend = 0u;
#pragma unroll
                                for (int i = 0; i < 2; ++i)
#pragma unroll
                                    for (int e = 0; e < 8; ++e) {
                                        w[i][e] = 0ull;
                                        if (c0 + e < C && (i == 0 || two)) {
                                            w[i][e] = ld_tagged(src + (size_t)i * kTcPartial + (size_t)(c0 + e) * kTcRows);
                                            pend |= 1u << (8 * i + e);
                                        }
                                    }
                                for (uint32_t it = 0;; ++it) {
#pragma unroll
                                    for (int i = 0; i < 2; ++i)
#pragma unroll
                                        for (int e = 0; e < 8; ++e)
                                            if ((uint32_t)(w[i][e] >> 32) == tag) pend &= ~(1u << (8 * i + e));
                                    if (pend == 0u) break;
                                    if (it >= s_wc.limit || wait_stopped(&s_wc)) {
                                        wait_fail(&s_wc, kStPartial);
                                        break;
                                    }
                                    if (it > 64) __nanosleep(64);
#pragma unroll
                                    for (int i = 0; i < 2; ++i)
#pragma unroll
                                        for (int e = 0; e < 8; ++e)
                                            if (pend & (1u << (8 * i + e)))
                                                w[i][e] = ld_tagged(src + (size_t)i * kTcPartial + (size_t)(c0 + e) * kTcRows);
                                }
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    if (c0 + e < C) {
                                        v[gq][e] += __uint_as_float((uint32_t)w[0][e]);
                                        if (two) v[gq][e] += __uint_as_float((uint32_t)w[1][e]);
                                    }
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (c0 + e < C) o.Y[(int64_t)(c0 + e) * out_f + row] = v[gq][e];
                    }
                }
            };

            // Segments in order; the epilogue of each runs after the next one's stages are posted
            // (or at the end of the range), while the next one fills the other accumulator set.
            TcSeg prev;
            bool have_prev = false;
            for (uint32_t s0 = lo, s1;; s0 = s1) {
                if (s0 >= hi) {
                    if (have_prev) epilogue(prev);
                    break;
                }
                const uint32_t rg = s0 / n_kc;
                s1 = min(hi, (rg + 1u) * n_kc);
                const uint32_t nb = tc_blocks(s0, s1), kmeta = k << kTcMetaKShift;
                const uint32_t jb0 = tc_first_block(pipe, cb);
                uint32_t first = kTcMetaFirst;
                if (jb0 >= nb) post(stage_begin(), kmeta | kTcMetaSegEnd);  // no block of this pipe here
                for (uint32_t jb = jb0; jb < nb; jb += kTcPipes) {
                    const uint32_t u0 = s0 + kTcU * jb, n = min((uint32_t)kTcU, s1 - u0);
                    const bool last_block = jb + kTcPipes >= nb;
                    const uint32_t slot = slot_ctr % kTcR;
                    // a wait that gave up ends the pipe's copies (the slot may still be filling)
                    if (!slot_wait(full0 + 8u * slot, (slot_ctr / kTcR) & 1u, &s_wc)) it.op = n_ops;
                    const uint8_t *sl = ring + slot * kTcSlotBytes;
#pragma unroll
                    for (int i = 0; i < kTcU; ++i) {
                        if (i >= (int)n) break;
                        const uint8_t *cbase = sl + kTcSlotCodes + hrb * (kTcU * kUnitCodeBytes) + i * kUnitCodeBytes + lane * 16;
                        const uint8_t *sbase = sl + kTcSlotScales + hrb * (kTcU * kUnitScaleBytes) +
                                               i * kUnitScaleBytes + g4 * 8;
                        uint4 cw[2];
                        uint2 sc[2];
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            cw[r] = *reinterpret_cast<const uint4 *>(cbase + (t0 + r) * 512);
                            sc[r] = *reinterpret_cast<const uint2 *>(sbase + (t0 + r) * 64);
                        }
                        const uint32_t st = stage_begin();
                        const uint32_t abase = astage0 + st * kTcAStage;
#pragma unroll
                        for (int r = 0; r < 2; ++r)
#pragma unroll
                            for (int hc = 0; hc < 2; ++hc) {
                                const uint32_t sel = hc ? 0x3232u : 0x1010u;  // block hc's scale, both halves
                                const uint32_t sg = __byte_perm(sc[r].x, sc[r].x, sel);
                                const uint32_t sg8 = __byte_perm(sc[r].y, sc[r].y, sel);
                                uint32_t o0[4], o1[4];
                                dequant_word_f16(hc ? cw[r].z : cw[r].x, sg, sg8, o0);
                                dequant_word_f16(hc ? cw[r].w : cw[r].y, sg, sg8, o1);
                                const uint32_t at = abase + a_row + (uint32_t)r * 2048u + (hc ? pc1 : pc0);
                                st_shared_v4(at, o0[0], o0[2], o1[0], o1[2]);
                                st_shared_v4(at + 1024u, o0[1], o0[3], o1[1], o1[3]);
                            }
                        const bool blk_end = i + 1 == (int)n, seg_end = last_block && blk_end;
                        post(st, kmeta | kTcMetaMma | first | (seg_end ? kTcMetaSegEnd : 0u) |
                                     (blk_end ? kTcMetaBlockEnd : 0u) | (slot << kTcMetaSlotShift) |
                                     ((uint32_t)i << kTcMetaUnitShift));
                        first = 0u;
                    }
                    // both warps reading this row block's part of the slot are done with it: refill
                    asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
                    issue();
                    ++slot_ctr;
                }
                if (have_prev) epilogue(prev);
                prev = TcSeg{s0, s1, rg, cb, nb, k};
                have_prev = true;
                cb += nb;
                ++k;
            }
        }
        post(stage_begin(), kTcMetaEnd);  // this pipe has no more stages
    }
    // after a give-up: wait (bounded) for copies that may still be in flight -- the last part
    // this warp copied into each slot -- so that none lands in shared memory after the CTA exits
    if (!mma_warp && lane == 0 && wait_stopped(&s_wc)) {
        for (uint32_t kk = c_issued > (uint32_t)kTcR ? c_issued - kTcR : 0u; kk < c_issued; ++kk)
            mbar_wait_ok(full0 + 8u * (kk % kTcR), (kk / kTcR) & 1u, kDrainLimit);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols)
                     : "memory");
    // the last CTA out returns the barrier counters to zero and advances the epoch; when the
    // partial tags are about to repeat it also clears every partial slot
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
        for (uint32_t i = threadIdx.x; i < part_entries; i += kTcThreads) part[i] = 0ull;
}
