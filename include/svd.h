/*
 * svd.h -- C ABI of the speculative-decoding verify pass for GB300 (sm_103a).
 *
 * The verify pass of speculative decoding scores K drafted tokens with one forward pass of the
 * target model: every weight matrix is read from memory once and applied to the K+1 activation
 * columns of the window; the target produces one distribution per window position; an
 * acceptance rule keeps a prefix of the drafts and the target's own token caps the window.
 * Sources:
 *   "100 tokens per second from a 27B model on a 24 GB AMD card" (curriculo.me), sections
 *     "The wall" and "How speculative decoding gets past a per-token wall";
 *   "Decode is memory-bound: the ~59 tok/s ceiling on an RTX 4090, and how speculative decoding
 *     gets past it" (trefon.com), sections "The ceiling", "Speculative decoding", "Two things
 *     the math says to do";
 *   the Hacker News thread on speculative decoding (hn.shard-db.dev, item 49596054): the
 *     comments on parallel verification and on the [positions, vocabulary] output tensor.
 *
 * Conventions for every entry point:
 *   - Buffers are DEVICE pointers unless stated; the caller allocates and owns all of them.
 *     The library never allocates device memory, keeps no per-call state and never
 *     synchronises the stream: every call only enqueues work on `stream` (cudaStream_t; NULL
 *     is the legacy default stream) and returns.
 *   - The return value is SVD_OK (0) or a negative SVD_ERR_* code; nothing is enqueued when a
 *     call returns an error.  svd_error_string() names a code; svd_last_cuda_error() gives the
 *     CUDA error behind the most recent SVD_ERR_CUDA of the calling thread.
 *   - Errors in the CONTENT of device inputs (a draft id out of range, a NaN probability) are
 *     not return codes: they are reported per window in a device status word (SVD_ST_*).
 *   - Pointers handed to the vector loads must be 16-byte aligned where stated.
 */
#ifndef SVD_H_
#define SVD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#pragma GCC visibility push(default) /* exported even when built with -fvisibility=hidden */
#endif

typedef struct CUstream_st *svd_stream_t; /* identical to cudaStream_t */

/* Return codes. */
enum {
    SVD_OK = 0,
    SVD_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer          */
    SVD_ERR_UNSUPPORTED = -2, /* a valid request this build does not implement       */
    SVD_ERR_CUDA = -3,        /* a CUDA call failed (see svd_last_cuda_error)        */
    SVD_ERR_WORKSPACE = -4,   /* workspace null or smaller than the query said       */
    SVD_ERR_TIMEOUT = -5      /* a bounded wait of a kernel gave up (svd_verify_status) */
};

/* Per-window status bits written by svd_accept (0 = clean). */
enum {
    SVD_ST_BAD_TOKEN = 1,     /* a draft id outside [0, V): that position is rejected */
    SVD_ST_Q_ZERO = 2,        /* q_i(x_i) == 0 for a drafted token                    */
    SVD_ST_BAD_PROB = 4,      /* a probability read was NaN, infinite, < 0 or > 1;    */
                              /* it was clamped into [0, 1]                           */
    SVD_ST_ZERO_RESIDUAL = 8, /* (p - q)+ had zero mass; the draw used p instead      */
    SVD_ST_EMPTY = 16         /* the distribution drawn from had zero mass: no token  */
};

/* Weight layouts. */
enum {
    SVD_LAYOUT_CANONICAL = 0, /* codes[out][in/2] bytes, input 2t in the low nibble,
                                 input 2t+1 in the high nibble; scales[out][in/32] fp16 */
    SVD_LAYOUT_NATIVE = 1,    /* the tensor-core fragment order made by
                                 svd_repack_weights (opaque; same byte count, rows
                                 padded to 64, inputs padded to 64)                   */
    SVD_LAYOUT_Q4K = 2        /* K-quant 4-bit super-blocks (the 4-bit tensors of the pages'
                                 Q4_K_M / UD-Q4_K_XL checkpoints; "100 tokens per second
                                 ...", "The wall"): codes -> [out][in/256] blocks of 144
                                 bytes = fp16 d, fp16 dmin, 12 bytes of packed 6-bit
                                 sub-block scales and mins, 128 bytes of 4-bit codes;
                                 weight = d sc[j] q - dmin m[j] for sub-block j of 32;
                                 scales must be NULL; in_features % 256 == 0.  Read by a
                                 CUDA-core kernel (svd_verify_linear only, C <= 8)       */,
    SVD_LAYOUT_Q4K_NATIVE = 3 /* the same super-blocks repacked by svd_repack_weights for the
                                 tensor-core stream kernel (opaque; same byte count, rows
                                 padded to 64): codes -> units of 64 rows x 256 inputs,
                                 8192 bytes of codes in fragment order; scales -> the
                                 units' 64 super-block headers (16 bytes each).  Streamed
                                 by svd_verify_linear and svd_verify_chain, C <= 16     */
};

/* Flags for svd_verify_linear. */
enum {
    SVD_F_PDL = 1, /* launch with programmatic dependent launch: the kernel may start while the
                     previous kernel on the stream is still running and stream its weights
                     early; it waits for that kernel before reading X or the workspace.  Set
                     only when nothing in flight on the stream writes the weights. */
    SVD_F_FRAGMENT_MMA = 2 /* native layout, 17..32 columns: run the warp-level mma.sync kernel
                     (bf16 operands, exact dequantisation, per-block fp32 rescale) instead of the
                     tcgen05 kernel (fp16 operands: the block scale is folded into the weights
                     with one fp16 rounding, activations rounded from bf16 to fp16).  Kept as the
                     comparison for the tensor-core path; no effect for C <= 16. */
};

#define SVD_C_MAX 32 /* most activation columns (K+1 positions x sequences) per call */
#define SVD_K_MAX 32 /* most drafted tokens per window                                */

/* A block-quantised 4-bit weight matrix W (in_features x out_features): code c in 0..15
 * stands for s * (c - 8) with one fp16 scale s per 32 consecutive inputs of an output row
 * (4.5 bits per weight).  codes and scales are device pointers, 16-byte aligned. */
typedef struct svd_qweight {
    const void *codes;
    const void *scales;
    int64_t in_features;  /* multiple of 32 */
    int64_t out_features; /* >= 1 */
    int32_t layout;       /* SVD_LAYOUT_* */
    int32_t reserved;     /* must be 0 */
} svd_qweight;

/* Sampler settings ("Decode is memory-bound ...", "Two things the math says to do":
 * temperature 0.6, top-p 0.95, min-p 0.05).  greedy != 0 ignores the other fields. */
typedef struct svd_sampler {
    float temperature; /* > 0 */
    float top_p;       /* (0, 1]; 1 disables the top-p filter */
    float min_p;       /* [0, 1); 0 disables the min-p filter */
    int32_t greedy;
} svd_sampler;

/* ---- errors ------------------------------------------------------------------------- */
const char *svd_error_string(int code);
int svd_last_cuda_error(void); /* cudaError_t of the thread's last SVD_ERR_CUDA */

/* ---- load time: weight repack ------------------------------------------------------- */
/* Byte sizes of the native layout of an in x out matrix (rows padded to 64, inputs padded to
 * 64).  Returns SVD_ERR_INVALID_ARG for in % 32 != 0 or non-positive sizes. */
int svd_native_sizes(int64_t in_features, int64_t out_features, size_t *codes_bytes,
                     size_t *scales_bytes);

/* Byte sizes of the Q4_K native layout (rows padded to 64): codes_bytes = 8192 per unit of 64
 * rows x 256 inputs, headers_bytes = 1024 per unit.  SVD_ERR_INVALID_ARG for in % 256 != 0 or
 * non-positive sizes. */
int svd_q4k_native_sizes(int64_t in_features, int64_t out_features, size_t *codes_bytes,
                         size_t *headers_bytes);

/* Permute a CANONICAL matrix into the NATIVE layout the tensor-core kernel streams: for each
 * 64-row block and each 64-input chunk, the 16-byte word every lane of a warp loads holds its
 * A-fragment nibbles for four k16 MMA steps, and the scales follow in fragment order.  A pure
 * bit permutation (padding codes are 8, padding scales 0); svd_unpack_weights is its inverse.
 * dst buffers must hold svd_native_sizes() bytes and must not overlap src. */
int svd_repack_weights(const svd_qweight *src_canonical, void *dst_codes, void *dst_scales,
                       svd_stream_t stream);
/* A Q4K matrix (src->layout SVD_LAYOUT_Q4K, scales NULL) is repacked into SVD_LAYOUT_Q4K_NATIVE
 * instead: dst_codes receives the units' codes (the nibble of input i of a unit's 64-input
 * sub-chunk at the place the NATIVE layout gives it, value q), dst_scales the headers, sizes
 * from svd_q4k_native_sizes; padding rows have code 0 and a zero header. */
/* Inverse of svd_repack_weights (drops the padding).  For SVD_LAYOUT_Q4K_NATIVE the raw Q4K
 * bytes [out][in/256 * 144] go to dst_codes and dst_scales must be NULL. */
int svd_unpack_weights(const svd_qweight *src_native, void *dst_codes, void *dst_scales,
                       svd_stream_t stream);

/* ---- (a) verify linear -------------------------------------------------------------- */
/* Y[c][j] = sum_i s[j][i/32] * (code[j][i] - 8) * X[c][i]  for c < C, j < out, in fp32
 * ("100 tokens per second ...", "How speculative decoding gets past a per-token wall": the
 * weights are read once and applied to the K-wide batch of the window).
 *   X: bf16 [C][in] row-major (token-major), 16-byte aligned.  Y: fp32 [C][out].
 *   C in 1..SVD_C_MAX.
 *   NATIVE weights run a tensor-core stream-K kernel.  C <= 16: warp-level bf16 MMA with the
 *   codes dequantised exactly, fp32 accumulate, one fresh accumulator per 32-input block,
 *   scaled in fp32.  17 <= C <= 32 ("Why a hiring company is writing this": several
 *   sequences' windows in one pass): tcgen05.mma with fp32 accumulators in tensor memory, the
 *   A operand fp16(s * (code - 8)) (one fp16 rounding, relative 2^-11) and the B operand X
 *   rounded to fp16 (|X| must stay below 65504; |X| < 2^-14 loses relative precision as an fp16
 *   subnormal), which keeps |error| <= 2^-11 * sum |w x| plus fp32 accumulation;
 *   SVD_F_FRAGMENT_MMA selects the warp-level kernel there too.  It needs a workspace of
 *   svd_verify_linear_workspace_bytes() bytes that is ZERO-FILLED before its first use (it
 *   holds barrier counters, which every call returns to zero, a launch epoch, a status word,
 *   and partial sums of row blocks split between CTAs, tagged with the launch that wrote
 *   them; for 17..32 columns also the fp16 B tiles of the activations, 4 KB per 64 inputs), so
 *   one zeroed workspace serves any number of calls issued in stream order, for any matrix shape
 *   and C whose size it covers (up to 16 columns the size does not depend on the shape); calls
 *   that may run concurrently need separate workspaces.  Every wait
 *   inside the kernel is bounded: one that gives up leaves Y undefined and records itself in
 *   the workspace (svd_verify_status).
 *   CANONICAL weights run the CUDA-core warp-shuffle kernel (no workspace; needs
 *   C * in * 4 <= 196608 bytes, else SVD_ERR_UNSUPPORTED).
 *   The result is deterministic: the same inputs give the same bits on every call. */
size_t svd_verify_linear_workspace_bytes(int64_t in_features, int64_t out_features, int C);
int svd_verify_linear(const svd_qweight *W, const void *X, int C, float *Y, void *workspace,
                      size_t workspace_bytes, int flags, svd_stream_t stream);

/* A chain of verify-linear launches executed in order: op i+1 may read what op i wrote. */
typedef struct svd_linear_op {
    svd_qweight W;  /* NATIVE layout */
    const void *X;  /* bf16 [C][W.in_features], 16-byte aligned */
    float *Y;       /* fp32 [C][W.out_features] */
} svd_linear_op;

/* The verify linear of every op of a model's pass in ONE persistent cooperative launch per 256
 * ops: each CTA streams its share of op 0, op 1, ... through the same shared-memory ring, so
 * the weights of op i+1 are already in flight while op i finishes; a grid-wide barrier between
 * ops orders op i's writes before op i+1 reads its activations ("100 tokens per second ...",
 * "How speculative decoding gets past a per-token wall": every weight matrix of the pass read
 * once for the whole window).  Results equal n_ops calls of svd_verify_linear bit for bit.
 * ops is a HOST array; the weights must not change while the chain runs.  SVD_F_PDL applies
 * to a chain of one op only.  The workspace is zero-filled before first use, as for
 * svd_verify_linear. */
size_t svd_verify_chain_workspace_bytes(const svd_linear_op *ops, int n_ops, int C);
int svd_verify_chain(const svd_linear_op *ops, int n_ops, int C, void *workspace,
                     size_t workspace_bytes, int flags, svd_stream_t stream);

/* Failure detection of svd_verify_linear / svd_verify_chain / svd_lm_head_softmax.  Each wait
 * of their kernel (a bulk copy landing, a partial sum from another CTA, the grid barrier
 * between the ops of a chain) is bounded; a wait that runs out sets a bit in the workspace's
 * status word, every later wait of the CTA returns at once, the kernel runs to its end, lets
 * its own copies in flight land and returns, and its outputs are undefined.
 * svd_verify_status waits for `stream`, reads the status word of `workspace` (a workspace of
 * at least svd_verify_linear_workspace_bytes() bytes; for svd_lm_head_softmax, the start of
 * its workspace), clears it, stores the bits in *bits (when bits != NULL; 1 = a copy, 2 = a
 * partial sum, 4 = the grid barrier) and returns SVD_OK when no wait gave up,
 * SVD_ERR_TIMEOUT when one did.  It synchronises the stream.
 * svd_verify_inject_stall (a test hook; no counterpart on the source pages) enqueues on `stream`
 * a write into the workspace that makes the kernels launched with it afterwards issue no
 * weight copy, as if the copy engine had stopped, and give up a wait after `polls` polls
 * (checked every 256 polls), so that a wait really runs out; SVD_POLL_DEFAULT turns it off. */
#define SVD_POLL_DEFAULT 0xFFFFFFFFu
int svd_verify_status(const void *workspace, size_t workspace_bytes, uint32_t *bits,
                      svd_stream_t stream);
int svd_verify_inject_stall(void *workspace, size_t workspace_bytes, uint32_t polls,
                            svd_stream_t stream);

/* ---- verify linear without caller scratch -------------------------------------------- */
/* (This entry point has no counterpart on the source pages; it is a deployment convenience.)
 * Some callers cannot allocate device memory at the point where they run the verify pass:
 * code that executes while another component owns every allocation (a host framework's
 * memory pool, a pre-reserved arena), inside callbacks or real-time threads where cudaMalloc's
 * implicit synchronisation is not allowed, or in plugins that are handed only the tensors they
 * read and write.  svd_verify_linear_noalloc computes exactly what svd_verify_linear computes
 * for a NATIVE matrix, with the same arguments minus the workspace: its scratch (stream-K
 * partial sums and barrier words) is a fixed array of SVD_NOALLOC_SCRATCH_BYTES in the
 * library's own device memory, reserved on every GPU that loads the library until the
 * process exits.  It calls no allocator of any kind.
 *   - out_features <= SVD_NOALLOC_MAX_OUT_FEATURES and at most 160 SMs, else
 *     SVD_ERR_UNSUPPORTED (other limits as for svd_verify_linear).
 *   - For 17..32 columns it runs the warp-level kernel (as svd_verify_linear with
 *     SVD_F_FRAGMENT_MMA): the array has no room for the tensor-core kernel's B tiles.
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture (a first call inside a capture
 *     returns SVD_ERR_UNSUPPORTED).  Every later call outside a capture looks it up again, so a
 *     new context on the device (after cudaDeviceReset) is handled; captured calls use the
 *     address of the last call outside capture.
 *   - Every call clears the barrier counters with a memset on `stream` and then launches the
 *     kernel.
 *     All calls share the one array, so calls that may overlap on the GPU (different streams
 *     without ordering between them) race and give wrong results; issue them in one stream or
 *     order them with events. */
#define SVD_NOALLOC_MAX_OUT_FEATURES 262144
#define SVD_NOALLOC_SCRATCH_BYTES (5u * 1024u * 1024u + 32u * 1024u)
int svd_verify_linear_noalloc(const svd_qweight *W, const void *X, int C, float *Y, int flags,
                              svd_stream_t stream);

/* ---- (b) sampler and lm_head -------------------------------------------------------- */
/* Per row of logits [rows][V] fp32: p = softmax(logits / T); keep v iff p[v] >= min_p *
 * max p and v lies in the shortest prefix, in the order (p descending, id ascending), whose
 * mass reaches top_p (the crossing token included); renormalise the kept mass to one.  Both
 * filters read the same un-renormalised p ("Decode is memory-bound ...", "Two things the math
 * says to do").  Writes probs [rows][V] fp32 and argmax [rows] (lowest id on ties; NaN
 * logits never win).  greedy writes the one-hot distribution of the argmax.
 *   probs must not alias logits.  rows in 1..SVD_C_MAX, V in 1..2^24. */
size_t svd_sampler_workspace_bytes(int rows, int64_t V);
int svd_sampler_probs(const float *logits, int rows, int64_t V, const svd_sampler *sampler,
                      float *probs, int32_t *argmax, void *workspace, size_t workspace_bytes,
                      svd_stream_t stream);

/* lm_head projection of every window position followed by the sampler: logits = W_lm^T H
 * ([positions][vocabulary], the HN thread's [4, vocabulary_size] tensor), then
 * svd_sampler_probs.  W_lm must be NATIVE (hidden x vocabulary).  H: bf16 [C][hidden].
 * logits: fp32 [C][V] (written).  For C <= 8 the GEMM's epilogue also produces, per block of
 * 64 vocabulary rows and position, the online-softmax statistics of the block -- its max, the
 * sum of exp((l - max) / T) over it and its argmax (lowest id on ties, NaN logits skipped) --
 * and the sampler merges those instead of scanning the logits for the row max (Milakov and
 * Gimelshein's online normaliser; the pages' [positions, vocabulary] output).  lse (nullable,
 * fp32 [C]) receives log sum_v exp(logits[c][v] / T), natural log, for a non-greedy sampler:
 * from the epilogue's block sums when C <= 8, else from the sampler's exact mass.  The
 * workspace (zero-filled before first use, as for svd_verify_linear) holds
 * svd_lm_head_workspace_bytes() bytes. */
size_t svd_lm_head_workspace_bytes(int64_t hidden, int64_t vocab, int C);
int svd_lm_head_softmax(const svd_qweight *W_lm, const void *H, int C,
                        const svd_sampler *sampler, float *logits, float *probs,
                        int32_t *argmax, float *lse, void *workspace, size_t workspace_bytes,
                        svd_stream_t stream);

/* ---- (c) acceptance ----------------------------------------------------------------- */
/* One verify window per w in [0, n_windows) with k drafts x_0..x_{k-1} (draft [n][k]).
 * Row i of the target distribution of window w is p + p_rows[w*(k+1)+i] * V when p_rows is
 * given, else p + (w*(k+1)+i) * V (i = 0..k); the drafter's rows likewise through q_rows
 * ([n][k]) or q + (w*k+i) * V.  Rows are fp32 probability vectors of length V.
 * Greedy (q == NULL): emit x_i while x_i equals the target's argmax at position i (from
 *   target_argmax [n][k+1] when given, else from p, lowest id on ties); at the first mismatch
 *   j emit argmax_j; if all k match emit argmax_k ("100 tokens per second ...", "How
 *   speculative decoding gets past a per-token wall"; the HN thread's "D E F" example).
 * Sampled (q != NULL): for i = 0..k-1 accept x_i iff u_i * q_i(x_i) < p_i(x_i) (decided
 *   exactly in double precision), i.e. with probability min(1, p/q); at the first rejection j
 *   emit a draw from the normalised (p_j - q_j)+ with u'_j; if all k are accepted emit a
 *   draw from p_k with u'_k, the target's own token capping the window ("Decode is
 *   memory-bound ...", "Speculative decoding"; Leviathan et al. 2023, Chen et al. 2023).  A
 *   draw from weights r emits the smallest v whose running sum exceeds u' * sum(r); the sums
 *   are exact 128-bit fixed point (2^-62 per unit), so the draw does not depend on thread
 *   order.
 *   u_i, u'_i are words 0 and 1 of Philox4x32-10 (Salmon et al., SC'11) with key = seed and
 *   counter = (window low 32 bits, window high 32 bits, i, 0), window = window_offset + w,
 *   each mapped to (word >> 8) * 2^-24.  uniforms ([n][k+1][2] fp32, multiples of 2^-24 in
 *   [0,1)) replaces them when non-NULL (a test hook).
 * Outputs: out_tokens [n][k+1] (emitted tokens then -1), n_emitted [n] in [1, k+1] for a
 *   clean window, status [n] (SVD_ST_* bits; 0 = clean).
 * k in 1..SVD_K_MAX, V in 1..2^31-1, n_windows >= 0 (0 enqueues nothing). */
int svd_accept(const float *p, const int64_t *p_rows, const float *q, const int64_t *q_rows,
               const int32_t *target_argmax, const int32_t *draft, int64_t n_windows, int k,
               int64_t V, uint64_t seed, uint64_t window_offset, const float *uniforms,
               int32_t *out_tokens, int32_t *n_emitted, int32_t *status, svd_stream_t stream);

/* ---- pass orchestration ------------------------------------------------------------- */
/* Record every call the thread makes on `stream` between svd_graph_begin and svd_graph_end
 * into one CUDA graph (stream capture), instantiate it and return an opaque handle; the
 * verify pass of a whole model (256 verify-linear launches for 64 layers, the lm_head, the
 * sampler and the acceptance) then replays with one svd_graph_launch.  Kernels recorded with
 * SVD_F_PDL keep their programmatic dependencies inside the graph.  The handle owns host
 * memory and the instantiated graph, no device buffers; free it with svd_graph_destroy. */
typedef struct svd_graph svd_graph;
int svd_graph_begin(svd_stream_t stream);
int svd_graph_end(svd_stream_t stream, svd_graph **out);
int svd_graph_launch(svd_graph *g, svd_stream_t stream);
void svd_graph_destroy(svd_graph *g);

/* Number of streaming multiprocessors of the current device (what the workspace queries
 * size for); -1 on error. */
int svd_device_sm_count(void);

/* ---- KV-read attention of a verify window ------------------------------------------------ */
/* "Decode is memory-bound ..." ("The ceiling"): at long context attention reads the whole KV
 * cache on every pass, beside the weights; "100 tokens per second ..." ("The wall"): the
 * target's cache at q8_0 keys and q4_0 values, 32K context.
 *
 * Canonical cache arrays of one layer (device, caller-owned), ld positions per kv head:
 *   k_codes  int8  [Hkv][ld][128]     key value = d * q
 *   k_scales fp16  [Hkv][ld][4]       one d per 32 dimensions
 *   v_codes  uint8 [Hkv][ld][64]      value = d * (c - 8); dimension 2t in the low nibble
 *   v_scales fp16  [Hkv][ld][4]
 * Native cache: units of 16 positions of one kv head, SVD_KV_UNIT_BYTES each, laid out
 * [Hkv][ceil(capacity / 16)][unit] (key codes, value codes, key scales, value scales in the
 * tensor-core fragment order of the attention kernel); 16-byte aligned.
 *
 * svd_kv_cache_bytes: bytes of a native cache for `capacity` positions (0 on bad sizes).
 * svd_kv_repack: writes positions [pos_begin, pos_end) of every kv head from the canonical
 *   arrays into the native cache (the append of a window's keys and values, or a whole cache);
 *   other positions are untouched.  svd_kv_unpack is its inverse (canonical arrays written for
 *   those positions).  Both return SVD_ERR_INVALID_ARG for null pointers, a misaligned cache,
 *   pos_end > capacity or pos_end > ld.
 * svd_kv_attention: for window position c = 0..C-1 (cache position n_past + c, its key and value
 *   already written) and query head h (kv head h / (Hq / Hkv)):
 *     o[c][h] = sum_{j <= n_past + c} softmax_j(scale * <q[c][h], k_j>) v_j
 *   q: bf16 [C][Hq][128]; out: fp32 [C][Hq][128]; both and the cache 16-byte aligned.
 *   Queries are used as f16: exact for bf16 values of magnitude in [2^-14, 65504] (and 0),
 *   rounded outside.  Positions of the cache beyond n_past + C are never read into the result,
 *   whatever their bytes.  The workspace (svd_kv_attention_workspace_bytes, 16-byte aligned)
 *   holds per-split partials; its first 32-bit word gets bit 0 set if a bounded wait of the
 *   kernel gave up (zero it once to watch it); its second word, when non-zero, is one more than
 *   the number of polls after which such a wait gives up (a test hook: 1 makes every wait give
 *   up at once; 0, the zero-filled value, keeps the default of about a second).  Two kernels are enqueued (the split pass and its
 *   merge, the latter a programmatic dependent launch).  The split pass starts copying cache
 *   units that lie wholly before position n_past before it waits for the kernel ahead of it on
 *   the stream: positions before n_past must not be written by a kernel still in flight there
 *   (an append of positions n_past.. is fine).  Errors: SVD_ERR_INVALID_ARG for null or
 *   misaligned pointers, Hq % Hkv != 0, C < 1, n_past < 0, n_past + C > capacity or a scale that
 *   is not positive and finite; SVD_ERR_WORKSPACE for a short workspace.
 */
#define SVD_KV_HEAD_DIM 128
#define SVD_KV_UNIT_POSITIONS 16
#define SVD_KV_UNIT_BYTES 3328
size_t svd_kv_cache_bytes(int n_kv_heads, int capacity);
int svd_kv_repack(const int8_t *k_codes, const uint16_t *k_scales, const uint8_t *v_codes,
                  const uint16_t *v_scales, int n_kv_heads, int ld, int pos_begin, int pos_end,
                  void *cache, int capacity, svd_stream_t stream);
int svd_kv_unpack(const void *cache, int capacity, int n_kv_heads, int pos_begin, int pos_end,
                  int8_t *k_codes, uint16_t *k_scales, uint8_t *v_codes, uint16_t *v_scales,
                  int ld, svd_stream_t stream);
/* svd_kv_append: the cache's write side for a verify window -- quantises the window's fp32 keys
 *   and values (position c at k + c * ld and v + c * ld, kv heads consecutive, 128 values each;
 *   ld >= Hkv * 128 floats, e.g. the k and v columns of the fused q|k|v output) to q8_0 keys and
 *   q4_0 values, per block of 32 in fp32 (READING: the llama.cpp block types of these names:
 *   q8_0 d = max|x|/127, q = round-half-away(x/d); q4_0 d = m/-8 with m the value of largest
 *   magnitude (lowest dimension on ties), c = min(15, trunc(x/d + 8.5)); 1/d is taken as 0 when
 *   d = 0; d stored as fp16, round to nearest even), and writes them at cache positions
 *   n_past .. n_past + C - 1 of the native cache.  Other positions are untouched.  One kernel
 *   (a programmatic dependent launch: it reads k and v only after the preceding kernel on the
 *   stream has completed).  Errors:
 *   SVD_ERR_INVALID_ARG for null or misaligned pointers, non-positive sizes, ld < Hkv * 128 or
 *   n_past + C > capacity. */
int svd_kv_append(const float *k, const float *v, int ld, int C, int n_kv_heads, int n_past,
                  void *cache, int capacity, svd_stream_t stream);
size_t svd_kv_attention_workspace_bytes(int n_q_heads, int n_kv_heads, int C);
/* svd_kv_attention_append: svd_kv_append of the window (k, v, ld as there) followed by
 *   svd_kv_attention, in one kernel when C * Hq / Hkv <= 24 (the CTAs whose units hold the
 *   window's positions quantise them into the cache before streaming those units; the last
 *   split of the context is made a little shorter to absorb that work), else as the two
 *   launches.  The cache is written as by svd_kv_append; the output is that of svd_kv_append
 *   followed by svd_kv_attention up to the order of the fp32 sums.  Errors as for both. */
int svd_kv_attention_append(const uint16_t *q, const float *k, const float *v, int ld, void *cache,
                            int capacity, int n_q_heads, int n_kv_heads, int n_past, int C,
                            float scale, float *out, void *workspace, size_t workspace_bytes,
                            svd_stream_t stream);
int svd_kv_attention(const uint16_t *q, const void *cache, int capacity, int n_q_heads,
                     int n_kv_heads, int n_past, int C, float scale, float *out, void *workspace,
                     size_t workspace_bytes, svd_stream_t stream);

/* ---- host-side companions: depth policy and n-gram drafter ----------------------------- */
/* No GPU work; safe to call from any host thread (a handle is not shared between threads
 * without the caller's locking).
 *
 * Tokens per pass and speedup ("Decode is memory-bound ...", section "Speculative decoding"):
 * with i.i.d. acceptance alpha in [0, 1] and depth k >= 0, a pass yields
 * (1 - alpha^(k+1)) / (1 - alpha) tokens (k + 1 at alpha = 1); if one draft step costs
 * draft_cost (>= 0) of a target pass, the speedup is that over (k * draft_cost + 1).  NaN on
 * arguments out of range.  svd_best_depth returns the k in 1..k_max with the largest
 * speedup (the shallower one on ties), or SVD_ERR_INVALID_ARG. */
double svd_expected_tokens_per_pass(double alpha, int k);
double svd_speedup(double alpha, int k, double draft_cost);
int svd_best_depth(double alpha, double draft_cost, int k_max);

/* Adaptive draft depth ("Decode is memory-bound ...", section "Two things the math says to
 * do": throttle the depth when the measured acceptance falls below 35 %).  The handle keeps
 * exponentially decayed counts of accepted drafts and of accept tests, fed with svd_accept's
 * outputs: a window that emitted n tokens at depth k accepted n - 1 drafts and, when
 * n - 1 < k, rejected one; windows with a non-zero status are skipped.  The decay halves a
 * window's weight after half_life_windows later windows.
 *   svd_spec_adapt_alpha: accepted / tests (NaN before the first test).
 *   svd_spec_adapt_depth: k_max before the first test; 1 while the estimate is below
 *   threshold (READING: the throttle drops to one draft, speculation stays on); otherwise
 *   svd_best_depth(estimate, draft_cost, k_max).
 * create returns NULL on bad arguments (k_max in 1..SVD_K_MAX, threshold in [0, 1],
 * half_life_windows > 0); observe returns SVD_OK or SVD_ERR_INVALID_ARG. */
typedef struct svd_spec_adapt svd_spec_adapt;
svd_spec_adapt *svd_spec_adapt_create(int k_max, double draft_cost, double threshold,
                                      double half_life_windows);
int svd_spec_adapt_observe(svd_spec_adapt *a, const int32_t *n_emitted, const int32_t *status,
                           int64_t n_windows, int k);
double svd_spec_adapt_alpha(const svd_spec_adapt *a);
int svd_spec_adapt_depth(const svd_spec_adapt *a);
void svd_spec_adapt_destroy(svd_spec_adapt *a);

/* n-gram drafter ("100 tokens per second ...", section "Lever 3: an n-gram overlay for
 * repetition"): an incremental hash map from every key of key_len consecutive tokens (1..64;
 * the page's sweep picked 6) to the position that followed its latest occurrence, over the
 * prompt and everything appended since.  svd_ngram_append adds tokens (host int32 array);
 * svd_ngram_propose looks up the last key_len tokens and, on a hit, writes up to k_max tokens
 * of the continuation that followed the key's latest earlier occurrence (the history up to its
 * end, at most) to out and returns how many; 0 on a miss or with fewer than key_len tokens.
 * Keys are compared token by token, so a hash collision never yields a wrong proposal.
 * create returns NULL on a bad key_len; the others return SVD_ERR_INVALID_ARG on null or
 * negative arguments.  svd_ngram_length returns the history length (-1 for NULL). */
typedef struct svd_ngram svd_ngram;
svd_ngram *svd_ngram_create(int key_len);
int svd_ngram_append(svd_ngram *g, const int32_t *tokens, int64_t n);
int svd_ngram_propose(const svd_ngram *g, int32_t *out, int k_max);
int64_t svd_ngram_length(const svd_ngram *g);
void svd_ngram_destroy(svd_ngram *g);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif
#endif /* SVD_H_ */
