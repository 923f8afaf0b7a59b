// verify_linear_tc.cuh -- the batched verify GEMM (17..32 activation columns) on the fifth-
// generation tensor cores: tcgen05.mma with fp32 accumulators in tensor memory.
//
// "100 tokens per second from a 27B model on a 24 GB AMD card", section "Why a hiring company
// is writing this", and "Decode is memory-bound ...", section "Rules I use" (rule 2): batching
// several sequences' windows amortises the one weight read of a pass over more columns.  At
// C = 32 the legacy fragment path pays one fp32 FMA per weight for the per-block rescale and
// reloads every activation fragment per warp; here the block scale is folded into the A operand
// and the activations are staged once per CTA in shared memory, where the tensor core reads
// them.
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
// one per CTA (stream-K).  A CTA runs four PIPES of four warps.  The CTA's range is cut into
// blocks of up to two units of one row group, dealt to the pipes round-robin; each pipe streams
// its blocks through a ring of two slots (per block four bulk copies, one per warp: the codes and
// the scales of the two row blocks), dequantises each half-chunk (128 rows x 32 inputs) into an
// fp16 A stage, converts the activations of that half-chunk into an fp16 B stage, and issues two
// tcgen05.mma (M 128, N 32, K 16) into its own accumulator (32 TMEM columns; two sets, by the
// parity of the row-group segment).  When a segment (one row group of the range) is done, the
// sixteen warps add the pipes' accumulators in pipe order -- pipe p reads TMEM columns 8p..8p+7
// (tokens), warp j of a pipe rows 32j..32j+31 (its TMEM lane quarter) -- and write Y, or store a
// tagged partial if an earlier CTA owns the row group; the owner adds the later CTAs' partials in
// CTA order.  Summation order is fixed: results are deterministic.
//
// Every wait is bounded (the WaitCtl of the stream-K kernel): a wait that runs out sets a status
// bit, later waits return at once, and before exiting the CTA waits a bounded time for its
// tensor-core operations and bulk copies.
// Included by verify_linear.cu inside namespace svd, after the stream-K kernel whose op
// descriptors, partial tags and bounded waits it shares.
#pragma once

constexpr int kTcPipes = 4;           // pipes per CTA
constexpr int kTcPipeWarps = 4;       // warps per pipe (one per TMEM lane quarter)
constexpr int kTcThreads = kTcPipes * kTcPipeWarps * 32;
constexpr int kTcU = 2;               // units per block (per bulk copy)
constexpr int kTcR = 2;               // ring slots per pipe
constexpr int kTcS = 3;               // A/B stages per pipe
constexpr int kTcN = 32;              // MMA N: activation columns
constexpr int kTcRows = 2 * kRowsPerBlock;            // MMA M: 128 weight rows
constexpr int kTcSlotBytes = 2 * kTcU * kUnitBytes;   // codes rb0, codes rb1, scales rb0, rb1
constexpr int kTcAStage = kTcRows * 32 * 2;           // 128 rows x 32 inputs fp16
constexpr int kTcBStage = kTcN * 32 * 2;              // 32 tokens x 32 inputs fp16
constexpr int kTcPipeBytes = kTcR * kTcSlotBytes + kTcS * (kTcAStage + kTcBStage);
constexpr int kTcAccCols = kTcN;                      // TMEM columns per accumulator
constexpr uint32_t kTcTmemCols = kTcPipes * 2 * kTcAccCols;  // 256 (power of two)
constexpr int kTcPartial = kTcRows * kTcN;            // entries of a CTA's partial
static_assert(kTcPartial <= 2 * kPartialMax, "a tensor-core CTA uses two stream-K partial slots");
static_assert(kRowsPerBlock == 64, "the MMA unit is two 64-row native blocks");

template <int MAXOPS>
struct TcCfg {
    // + 1 KB to align the stages to the 512-byte period of the 64-byte swizzle
    static constexpr size_t kSmem = (size_t)kTcPipes * kTcPipeBytes + (size_t)MAXOPS * sizeof(VlOp) + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

// ---- tcgen05 / TMEM -----------------------------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand stored with the 64-byte swizzle: each row
// holds 32 fp16 inputs (64 bytes), row r at 64 r, and its 16-byte piece c sits at piece
// c ^ ((r >> 1) & 3) (address bits 4-5 XOR bits 7-8), so a quarter-warp storing two rows writes
// one contiguous 128 bytes.  Fields: start >> 4, leading offset (unused by swizzled K-major
// layouts) >> 4 at bit 16, stride between 8-row groups (8 x 64 = 512 bytes) >> 4 at bit 32, the
// descriptor version bit 46, layout 4 (64-byte swizzle) at bits 61-63.  The operand must lie
// in a 512-byte-aligned region; a K step of 16 advances the start by 32 bytes.
__device__ __forceinline__ uint64_t tc_sdesc_sw64(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(16u >> 4) << 16) |
           ((uint64_t)(512u >> 4) << 32) | (1ull << 46) | (4ull << 61);
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
    uint32_t s0, s1;      // current segment
    uint32_t jb, nb, cb;  // next block of this pipe in the segment, blocks in it, blocks before it

    __device__ __forceinline__ void start() {
        op = -1;
        lo = hi = s0 = s1 = 0u;
        jb = nb = cb = 0u;
    }
    // Next block of pipe p: op index, first unit and unit count; false when there is none.
    __device__ __forceinline__ bool next(uint32_t p, const VlOp *ops, int n_ops, uint32_t G, uint32_t b,
                                         int *op_out, uint32_t *u0, uint32_t *n) {
        for (;;) {
            if (op >= n_ops) return false;
            if (op >= 0 && jb < nb) {
                *op_out = op;
                *u0 = s0 + kTcU * jb;
                *n = min((uint32_t)kTcU, s1 - *u0);
                jb += kTcPipes;
                return true;
            }
            cb += nb;
            nb = 0u;
            if (op >= 0 && s1 < hi) {
                const uint32_t n_kc = ops[op].n_kc;
                s0 = s1;
                s1 = min(hi, (s0 / n_kc + 1u) * n_kc);
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

template <int MAXOPS>
__global__ void __launch_bounds__(kTcThreads, 1)
vl_tc_kernel(const __grid_constant__ VlOps<MAXOPS> P, unsigned long long *__restrict__ part,
             uint32_t part_entries, unsigned *__restrict__ gbar) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_full[kTcPipes * kTcR];   // a ring slot's copies landed
    __shared__ __align__(8) uint64_t s_empty[kTcPipes * kTcS];  // a stage's MMAs have read it
    __shared__ __align__(8) uint64_t s_done[kTcPipes * 2];      // a pipe's MMAs of a segment (per set)
    __shared__ __align__(8) uint64_t s_free[2];                 // a set's accumulators have been read
    __shared__ __align__(8) uint64_t s_final[kTcPipes];         // every MMA of a pipe, at exit
    __shared__ uint32_t s_tmem, s_epoch, s_last;
    __shared__ WaitCtl s_wc;
    uint8_t *const sm0 = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);  // 1 KB aligned
    VlOp *ops = reinterpret_cast<VlOp *>(sm0 + (size_t)kTcPipes * kTcPipeBytes);
    const int n_ops = P.n;
    const int C = P.C;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t pipe = (uint32_t)warp / kTcPipeWarps;
    const int wj = warp % kTcPipeWarps;  // warp in the pipe = its TMEM lane quarter
    const uint32_t G = gridDim.x, b = blockIdx.x;
    const bool elected = wj == 0 && lane == 0;  // issues the pipe's MMAs
    uint8_t *const ring = sm0 + (size_t)pipe * kTcPipeBytes;
    const uint32_t ring0 = smem_u32(ring);
    const uint32_t astage0 = ring0 + kTcR * kTcSlotBytes;
    const uint32_t bstage0 = astage0 + kTcS * kTcAStage;
    const uint32_t full0 = smem_u32(&s_full[pipe * kTcR]);
    const uint32_t empty0 = smem_u32(&s_empty[pipe * kTcS]);

    {
        static_assert(sizeof(VlOp) % 8 == 0, "op descriptor copied in 8-byte words");
        const uint64_t *src = reinterpret_cast<const uint64_t *>(&P.op[0]);
        uint64_t *dst = reinterpret_cast<uint64_t *>(ops);
        for (int i = threadIdx.x; i < n_ops * (int)(sizeof(VlOp) / 8); i += kTcThreads) dst[i] = src[i];
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcPipes * kTcR; ++i) mbar_init(smem_u32(&s_full[i]), kTcPipeWarps);
        for (int i = 0; i < kTcPipes * kTcS; ++i) mbar_init(smem_u32(&s_empty[i]), 1);
        for (int i = 0; i < kTcPipes * 2; ++i) mbar_init(smem_u32(&s_done[i]), 1);
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&s_free[i]), kTcPipes * kTcPipeWarps);
        for (int i = 0; i < kTcPipes; ++i) mbar_init(smem_u32(&s_final[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_wc.stop = 0u;
    }
    __syncthreads();

    // Copy cursor of this pipe (uniform across its warps).  Warp wj copies one part of every
    // block: wj = 0, 1 the codes of row block 2q + wj, wj = 2, 3 the scales of row block
    // 2q + wj - 2; a row block past the matrix's end is not copied (its rows are never stored).
    TcIter it;
    it.start();
    uint32_t c_issued = 0;
    auto issue = [&]() {
        int op;
        uint32_t u0, n;
        if (!it.next(pipe, ops, n_ops, G, b, &op, &u0, &n)) return;
        const VlOp &o = ops[op];
        const uint32_t slot = c_issued % kTcR, bar = full0 + 8u * slot;
        if (lane == 0) {
            const uint32_t q = u0 / o.n_kc, kc = u0 - q * o.n_kc, h = (uint32_t)wj & 1u;
            const uint32_t rb = 2u * q + h, n_rb = o.n_units / o.n_kc;
            if (rb < n_rb) {
                const size_t nu = (size_t)rb * o.n_kc + kc;  // native unit index
                uint32_t dst, bytes;
                const uint8_t *src;
                if (wj < 2) {
                    bytes = n * kUnitCodeBytes;
                    dst = ring0 + slot * kTcSlotBytes + h * (kTcU * kUnitCodeBytes);
                    src = o.codes + nu * kUnitCodeBytes;
                } else {
                    bytes = n * kUnitScaleBytes;
                    dst = ring0 + slot * kTcSlotBytes + 2u * kTcU * kUnitCodeBytes + h * (kTcU * kUnitScaleBytes);
                    src = o.scales + nu * kUnitScaleBytes;
                }
                mbar_expect_tx(bar, bytes);
                bulk_g2s(dst, src, bytes, bar);
            } else {
                mbar_arrive(bar);
            }
        }
        ++c_issued;
    };
    // The consumer's next block (for the activation prefetch): one block ahead of it.
    TcIter la;
    la.start();
    {
        int op_;
        uint32_t u_, n_;
        la.next(pipe, ops, n_ops, G, b, &op_, &u_, &n_);
    }
    // The stall injection (workspace word kBarPoll, written only by the test hook): no copy.
    if (*reinterpret_cast<volatile unsigned *>(gbar + kBarPoll) != 0u) it.op = n_ops;
    // weights never depend on earlier kernels: start streaming before waiting for them
    for (int i = 0; i < kTcR; ++i) issue();

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

    const int g4 = lane >> 2, t4 = lane & 3;
    const int hrb = wj >> 1;       // this warp's row block in the MMA unit (rows 32 wj .. 32 wj + 31)
    const int t0 = 2 * (wj & 1);   // its first 16-row tile there
    constexpr uint32_t kIdesc = tc_idesc_f16(kTcRows, kTcN);
    // This lane's places in a stage (64-byte swizzle).  A: row g of tile t0 + r is row
    // 64 hrb + 16 (t0 + r) + g of the unit, its inputs 8 t4 .. 8 t4 + 7 piece t4 ^ ((g >> 1) & 3);
    // row g + 8 is 512 bytes further.  B: token 8 wj + g4, the same piece.
    const uint32_t piece = (uint32_t)(t4 ^ ((g4 >> 1) & 3)) * 16u;
    const uint32_t a_off = (uint32_t)(64 * hrb + 16 * t0 + g4) * 64u + piece;
    const uint32_t b_off = (uint32_t)(8 * wj + g4) * 64u + piece;
    const int xtok = 8 * wj + g4;  // the activation column this lane converts
    constexpr uint32_t kQuarter = 1u << 16;  // TMEM lane field

    uint32_t k = 0, cb = 0, stage_ctr = 0, slot_ctr = 0;
    for (int gi = 0; gi < n_ops; ++gi) {
        const VlOp &o = ops[gi];
        if (gi > 0) {
            __syncthreads();
            if (threadIdx.x == 0) grid_barrier(gbar + kBarCount, (unsigned)gi * G, &s_wc);
            __syncthreads();
        }
        const uint32_t n_kc = o.n_kc;
        const int64_t in_f = o.in_f, out_f = o.out_f;
        const uint32_t tag = (partial_epoch24(epoch) << 8) | (uint32_t)(gi & 255);
        const __nv_bfloat16 *xrow = o.X + (int64_t)(xtok < C ? xtok : 0) * in_f + 8 * t4;
        // this lane's 8 activations of the half-chunk starting at input col (zero past C or in)
        auto load_x = [&](int64_t col) {
            if (xtok >= C || col >= in_f) return make_uint4(0u, 0u, 0u, 0u);
            if constexpr (MAXOPS > 1) return ldg_cg_v4(xrow + col);
            else return ldg_nc_v4(xrow + col);
        };
        uint4 xcur = make_uint4(0u, 0u, 0u, 0u);
        bool xpre = false;  // xcur holds the next stage's activations
        uint32_t lo, hi;
        tc_range(o, G, b, &lo, &hi);

        // Epilogue of a segment: the pipes' accumulators of its set added in pipe order (this
        // pipe takes tokens 8 pipe .. 8 pipe + 7, this warp its 32 rows), then Y -- or a tagged
        // partial when an earlier CTA owns the row group; an owner whose row group runs on into
        // later CTAs adds their partials in CTA order (only at the end of its range).
        auto epilogue = [&](const TcSeg &sg) {
            const uint32_t set = sg.k & 1u;
            for (uint32_t pp = 0; pp < (uint32_t)kTcPipes; ++pp)
                slot_wait(smem_u32(&s_done[pp * 2u + set]), (sg.k >> 1) & 1u, &s_wc);
            tc_fence_after();
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
            for (uint32_t pp = 0; pp < (uint32_t)kTcPipes; ++pp) {
                if (tc_first_block(pp, sg.cb) >= sg.nb) continue;  // no block of pipe pp here
                uint32_t r[8];
                tc_ld8(tmem + (uint32_t)wj * 32u * kQuarter + (pp * 2u + set) * kTcAccCols + 8u * pipe, r);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] += __uint_as_float(r[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s_free[set]));

            const uint32_t rl = 32u * (uint32_t)wj + (uint32_t)lane;
            const int64_t row = (int64_t)sg.rg * kTcRows + rl;
            const int c0 = 8 * (int)pipe;
            const bool owner = sg.s0 == sg.rg * n_kc, whole = sg.s1 == (sg.rg + 1u) * n_kc;
            if (!owner) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (c0 + e < C) st_tagged(part + (size_t)b * kTcPartial + (size_t)(c0 + e) * kTcRows + rl, v[e], tag);
            } else if (row < out_f) {
                if (!whole) {
                    const uint32_t b_last = tc_cta_of(o, G, (sg.rg + 1u) * n_kc - 1u);
                    for (uint32_t bb = b + 1u; bb <= b_last; ++bb) {
                        const unsigned long long *src = part + (size_t)bb * kTcPartial + rl;
                        unsigned long long w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (c0 + e < C) w[e] = ld_tagged(src + (size_t)(c0 + e) * kTcRows);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (c0 + e < C)
                                v[e] += (uint32_t)(w[e] >> 32) == tag
                                            ? __uint_as_float((uint32_t)w[e])
                                            : wait_tagged(src + (size_t)(c0 + e) * kTcRows, tag, &s_wc);
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (c0 + e < C) o.Y[(int64_t)(c0 + e) * out_f + row] = v[e];
            }
        };

        // Segments in order; the epilogue of each runs after the next one's MMAs are issued
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
            const uint32_t nb = tc_blocks(s0, s1), set = k & 1u;
            const uint32_t dcol = tmem + (pipe * 2u + set) * kTcAccCols;
            // the elected thread waits, before the segment's first MMA or its end, until the
            // epilogue of segment k - 2 (same set) has read the accumulators
            bool need_free = k >= 2u;
            uint32_t accum = 0u;
            for (uint32_t jb = tc_first_block(pipe, cb); jb < nb; jb += kTcPipes) {
                const uint32_t u0 = s0 + kTcU * jb, n = min((uint32_t)kTcU, s1 - u0);
                const uint32_t kc0 = u0 - rg * n_kc;
                // the pipe's next block, if it belongs to this op: its first activations are
                // prefetched during this block's last stage
                int nop;
                uint32_t nu0, nn;
                const bool nxt = la.next(pipe, ops, n_ops, G, b, &nop, &nu0, &nn) && nop == gi;
                const uint32_t slot = slot_ctr % kTcR;
                // a wait that gave up ends the pipe's copies (the slot may still be filling)
                if (!slot_wait(full0 + 8u * slot, (slot_ctr / kTcR) & 1u, &s_wc)) it.op = n_ops;
                const uint8_t *sl = ring + slot * kTcSlotBytes;
#pragma unroll
                for (int i = 0; i < kTcU; ++i) {
                    if (i >= (int)n) break;
                    const uint8_t *cbase = sl + hrb * (kTcU * kUnitCodeBytes) + i * kUnitCodeBytes + lane * 16;
                    const uint8_t *sbase = sl + 2 * kTcU * kUnitCodeBytes + hrb * (kTcU * kUnitScaleBytes) +
                                           i * kUnitScaleBytes + g4 * 8;
                    uint4 cw[2];
                    uint2 sc[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        cw[r] = *reinterpret_cast<const uint4 *>(cbase + (t0 + r) * 512);
                        sc[r] = *reinterpret_cast<const uint2 *>(sbase + (t0 + r) * 64);
                    }
#pragma unroll
                    for (int hc = 0; hc < 2; ++hc) {
                        // this stage's activations (prefetched by the previous stage, else now),
                        // then the next stage's
                        if (!xpre) xcur = load_x((int64_t)(kc0 + i) * kChunk + 32 * hc);
                        const uint4 xv = xcur;
                        xpre = true;
                        if (hc == 0)
                            xcur = load_x((int64_t)(kc0 + i) * kChunk + 32);
                        else if (i + 1 < (int)n)
                            xcur = load_x((int64_t)(kc0 + i + 1) * kChunk);
                        else if (nxt)
                            xcur = load_x((int64_t)(nu0 - (nu0 / n_kc) * n_kc) * kChunk);
                        else
                            xpre = false;
                        const uint32_t st = stage_ctr % kTcS;
                        if (stage_ctr >= (uint32_t)kTcS)
                            slot_wait(empty0 + 8u * st, ((stage_ctr / kTcS) - 1u) & 1u, &s_wc);
                        const uint32_t abase = astage0 + st * kTcAStage, bbase = bstage0 + st * kTcBStage;
                        const uint32_t sel = hc ? 0x3232u : 0x1010u;  // block hc's scale in both halves
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const uint32_t w0 = hc ? cw[r].z : cw[r].x, w1 = hc ? cw[r].w : cw[r].y;
                            const uint32_t sg = __byte_perm(sc[r].x, sc[r].x, sel);
                            const uint32_t sg8 = __byte_perm(sc[r].y, sc[r].y, sel);
                            uint32_t o0[4], o1[4];
                            dequant_word_f16(w0, sg, sg8, o0);
                            dequant_word_f16(w1, sg, sg8, o1);
                            st_shared_v4(abase + a_off + r * 1024u, o0[0], o0[2], o1[0], o1[2]);
                            st_shared_v4(abase + a_off + r * 1024u + 512u, o0[1], o0[3], o1[1], o1[3]);
                        }
                        st_shared_v4(bbase + b_off, bf16x2_to_f16x2(xv.x), bf16x2_to_f16x2(xv.y),
                                     bf16x2_to_f16x2(xv.z), bf16x2_to_f16x2(xv.w));
                        fence_proxy_async_smem();
                        asm volatile("bar.sync %0, %1;" ::"r"(1 + pipe), "r"(kTcPipeWarps * 32) : "memory");
                        if (elected) {
                            if (need_free) {
                                slot_wait(smem_u32(&s_free[set]), ((k >> 1) - 1u) & 1u, &s_wc);
                                need_free = false;
                            }
                            tc_fence_after();
#pragma unroll
                            for (uint32_t kq = 0; kq < 2; ++kq)
                                tc_mma_f16(dcol, tc_sdesc_sw64(abase + 32u * kq), tc_sdesc_sw64(bbase + 32u * kq),
                                           kIdesc, accum | kq);
                            tc_commit(empty0 + 8u * st);
                        }
                        accum = 1u;
                        ++stage_ctr;
                    }
                }
                // every warp of the pipe has read the slot (the barrier above): refill it
                issue();
                ++slot_ctr;
            }
            if (elected) {
                if (need_free) slot_wait(smem_u32(&s_free[set]), ((k >> 1) - 1u) & 1u, &s_wc);
                tc_commit(smem_u32(&s_done[pipe * 2u + set]));
            }
            if (have_prev) epilogue(prev);
            prev = TcSeg{s0, s1, rg, cb, nb, k};
            have_prev = true;
            cb += nb;
            ++k;
        }
    }

    // every tensor-core operation of the pipe is complete before the accumulators are released
    if (elected) {
        tc_commit(smem_u32(&s_final[pipe]));
        mbar_wait_ok(smem_u32(&s_final[pipe]), 0u);
    }
    // after a give-up: wait (bounded) for copies that may still be in flight -- the last part
    // this warp copied into each slot -- so that none lands in shared memory after the CTA exits
    if (lane == 0 && wait_stopped(&s_wc)) {
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
