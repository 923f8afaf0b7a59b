// api.cu -- the extern "C" surface of libsvd: argument checks, workspace queries, the lm_head
// composition and CUDA-graph capture of a whole verify pass.
#include <atomic>

#include "svd_common.cuh"

namespace svd {

size_t vl_workspace_bytes(int64_t in_f, int64_t out_f, int C);
int verify_linear(const svd_qweight *W, const void *X, int C, float *Y, void *ws, size_t ws_bytes,
                  int flags, cudaStream_t stream);
int native_sizes(int64_t in_f, int64_t out_f, size_t *cb, size_t *sb);
int kq_native_sizes(int64_t in_f, int64_t out_f, size_t *cb, size_t *hb);
int repack(const svd_qweight *src, void *dc, void *ds, cudaStream_t stream);
int unpack(const svd_qweight *src, void *dc, void *ds, cudaStream_t stream);
int verify_linear_noalloc(const svd_qweight *W, const void *X, int C, float *Y, int flags,
                          cudaStream_t stream);
size_t chain_workspace_bytes(const svd_linear_op *ops, int n_ops, int C);
int verify_chain(const svd_linear_op *ops, int n_ops, int C, void *ws, size_t ws_bytes, int flags,
                 cudaStream_t stream);
int verify_status(const void *ws, size_t ws_bytes, uint32_t *bits, cudaStream_t stream);
int verify_inject_stall(void *ws, size_t ws_bytes, uint32_t polls, cudaStream_t stream);
size_t sampler_ws_bytes(int rows, int64_t V);
int sampler_probs(const float *logits, int rows, int64_t V, const svd_sampler *s, float *probs,
                  int32_t *argmax, void *ws, size_t ws_bytes, cudaStream_t stream,
                  const float4 *stats = nullptr, int n_sb = 0, float *lse = nullptr);
int verify_linear_ex(const svd_qweight *W, const void *X, int C, float *Y, void *ws,
                     size_t ws_bytes, int flags, float4 *stats, float stat_k, bool *stats_done,
                     cudaStream_t stream);
int accept(const float *p, const int64_t *p_rows, const float *q, const int64_t *q_rows,
           const int32_t *tgt_am, const int32_t *draft, int64_t n, int k, int64_t V,
           uint64_t seed, uint64_t woff, const float *uniforms, int32_t *out_tokens,
           int32_t *n_emitted, int32_t *status, cudaStream_t stream);

static thread_local int g_last_cuda_error = 0;
void set_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace svd

struct svd_graph {
    cudaGraphExec_t exec;
};

extern "C" {

const char *svd_error_string(int code) {
    switch (code) {
        case SVD_OK: return "SVD_OK: success";
        case SVD_ERR_INVALID_ARG: return "SVD_ERR_INVALID_ARG: null, out-of-range or misaligned argument";
        case SVD_ERR_UNSUPPORTED: return "SVD_ERR_UNSUPPORTED: request not implemented by this build";
        case SVD_ERR_CUDA: return "SVD_ERR_CUDA: a CUDA call failed (see svd_last_cuda_error)";
        case SVD_ERR_WORKSPACE: return "SVD_ERR_WORKSPACE: workspace missing or too small";
        case SVD_ERR_TIMEOUT: return "SVD_ERR_TIMEOUT: a bounded wait of a kernel gave up";
        default: return "unknown svd error code";
    }
}

int svd_last_cuda_error(void) { return svd::g_last_cuda_error; }

int svd_device_sm_count(void) { return svd::sm_count(); }

int svd_native_sizes(int64_t in_f, int64_t out_f, size_t *cb, size_t *sb) {
    return svd::native_sizes(in_f, out_f, cb, sb);
}

int svd_q4k_native_sizes(int64_t in_f, int64_t out_f, size_t *cb, size_t *hb) {
    return svd::kq_native_sizes(in_f, out_f, cb, hb);
}

int svd_repack_weights(const svd_qweight *src, void *dc, void *ds, svd_stream_t stream) {
    return svd::repack(src, dc, ds, (cudaStream_t)stream);
}

int svd_unpack_weights(const svd_qweight *src, void *dc, void *ds, svd_stream_t stream) {
    return svd::unpack(src, dc, ds, (cudaStream_t)stream);
}

size_t svd_verify_linear_workspace_bytes(int64_t in_f, int64_t out_f, int C) {
    if (in_f <= 0 || out_f <= 0 || C < 1 || C > SVD_C_MAX || svd::sm_count() < 1) return 0;
    return svd::vl_workspace_bytes(in_f, out_f, C);
}

int svd_verify_linear(const svd_qweight *W, const void *X, int C, float *Y, void *ws,
                      size_t ws_bytes, int flags, svd_stream_t stream) {
    return svd::verify_linear(W, X, C, Y, ws, ws_bytes, flags, (cudaStream_t)stream);
}

int svd_verify_linear_noalloc(const svd_qweight *W, const void *X, int C, float *Y, int flags,
                              svd_stream_t stream) {
    return svd::verify_linear_noalloc(W, X, C, Y, flags, (cudaStream_t)stream);
}

size_t svd_verify_chain_workspace_bytes(const svd_linear_op *ops, int n_ops, int C) {
    if (!ops || n_ops < 1 || C < 1 || C > SVD_C_MAX || svd::sm_count() < 1) return 0;
    return svd::chain_workspace_bytes(ops, n_ops, C);
}

int svd_verify_chain(const svd_linear_op *ops, int n_ops, int C, void *ws, size_t ws_bytes,
                     int flags, svd_stream_t stream) {
    return svd::verify_chain(ops, n_ops, C, ws, ws_bytes, flags, (cudaStream_t)stream);
}

int svd_verify_status(const void *ws, size_t ws_bytes, uint32_t *bits, svd_stream_t stream) {
    return svd::verify_status(ws, ws_bytes, bits, (cudaStream_t)stream);
}

int svd_verify_inject_stall(void *ws, size_t ws_bytes, uint32_t polls, svd_stream_t stream) {
    return svd::verify_inject_stall(ws, ws_bytes, polls, (cudaStream_t)stream);
}

size_t svd_sampler_workspace_bytes(int rows, int64_t V) {
    if (rows < 1 || rows > SVD_C_MAX || V < 1) return 0;
    return svd::sampler_ws_bytes(rows, V);
}

int svd_sampler_probs(const float *logits, int rows, int64_t V, const svd_sampler *s, float *probs,
                      int32_t *argmax, void *ws, size_t ws_bytes, svd_stream_t stream) {
    return svd::sampler_probs(logits, rows, V, s, probs, argmax, ws, ws_bytes, (cudaStream_t)stream);
}

// lm_head workspace: [verify linear][the epilogue's block statistics: ceil(V / 64) x C float4]
// [sampler], each part 256-byte aligned.
static size_t lm_stats_bytes(int64_t vocab, int C) {
    return svd::align_up((size_t)((vocab + 63) / 64) * (size_t)C * 16, 256);
}

size_t svd_lm_head_workspace_bytes(int64_t hidden, int64_t vocab, int C) {
    if (hidden <= 0 || vocab <= 0 || C < 1 || C > SVD_C_MAX || svd::sm_count() < 1) return 0;
    return svd::align_up(svd::vl_workspace_bytes(hidden, vocab, C), 256) + lm_stats_bytes(vocab, C) +
           svd::sampler_ws_bytes(C, vocab);
}

int svd_lm_head_softmax(const svd_qweight *W, const void *H, int C, const svd_sampler *s,
                        float *logits, float *probs, int32_t *argmax, float *lse, void *ws,
                        size_t ws_bytes, svd_stream_t stream) {
    if (!W || !s || !logits || !probs) return SVD_ERR_INVALID_ARG;
    if (W->layout != SVD_LAYOUT_NATIVE) return SVD_ERR_INVALID_ARG;
    if (C < 1 || C > SVD_C_MAX || W->out_features > (1LL << 24)) return SVD_ERR_INVALID_ARG;
    const size_t need = svd_lm_head_workspace_bytes(W->in_features, W->out_features, C);
    if (!ws || need == 0 || ws_bytes < need) return SVD_ERR_WORKSPACE;
    const size_t vl = svd::align_up(svd::vl_workspace_bytes(W->in_features, W->out_features, C), 256);
    const size_t sb = lm_stats_bytes(W->out_features, C);
    float4 *stats = reinterpret_cast<float4 *>(reinterpret_cast<uint8_t *>(ws) + vl);
    const float stat_k = s->greedy ? 0.f : 1.4426950408889634f / s->temperature;
    bool fused = false;
    int rc = svd::verify_linear_ex(W, H, C, logits, ws, vl, 0, stats, stat_k, &fused, (cudaStream_t)stream);
    if (rc != SVD_OK) return rc;
    return svd::sampler_probs(logits, C, W->out_features, s, probs, argmax,
                              reinterpret_cast<uint8_t *>(ws) + vl + sb, ws_bytes - vl - sb,
                              (cudaStream_t)stream, fused ? stats : nullptr,
                              (int)((W->out_features + 63) / 64), lse);
}

int svd_accept(const float *p, const int64_t *p_rows, const float *q, const int64_t *q_rows,
               const int32_t *target_argmax, const int32_t *draft, int64_t n, int k, int64_t V,
               uint64_t seed, uint64_t woff, const float *uniforms, int32_t *out_tokens,
               int32_t *n_emitted, int32_t *status, svd_stream_t stream) {
    return svd::accept(p, p_rows, q, q_rows, target_argmax, draft, n, k, V, seed, woff, uniforms,
                       out_tokens, n_emitted, status, (cudaStream_t)stream);
}

int svd_graph_begin(svd_stream_t stream) {
    if (!stream) return SVD_ERR_INVALID_ARG;  // the legacy default stream cannot be captured
    SVD_CUDA_TRY(cudaStreamBeginCapture((cudaStream_t)stream, cudaStreamCaptureModeThreadLocal));
    return SVD_OK;
}

int svd_graph_end(svd_stream_t stream, svd_graph **out) {
    if (!stream || !out) return SVD_ERR_INVALID_ARG;
    cudaGraph_t graph = nullptr;
    SVD_CUDA_TRY(cudaStreamEndCapture((cudaStream_t)stream, &graph));
    cudaGraphExec_t exec = nullptr;
    cudaError_t e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    SVD_CUDA_TRY(e);
    svd_graph *g = new svd_graph;
    g->exec = exec;
    *out = g;
    return SVD_OK;
}

int svd_graph_launch(svd_graph *g, svd_stream_t stream) {
    if (!g) return SVD_ERR_INVALID_ARG;
    SVD_CUDA_TRY(cudaGraphLaunch(g->exec, (cudaStream_t)stream));
    return SVD_OK;
}

void svd_graph_destroy(svd_graph *g) {
    if (!g) return;
    cudaGraphExecDestroy(g->exec);
    delete g;
}

}  // extern "C"
