"""Thin ctypes binding of ``libsvd.so`` (declared in ``include/svd.h``).

Argument marshalling only: every function has the C entry point's name, turns torch tensors into
device pointers and streams into ``cudaStream_t`` handles, calls the library and raises
:class:`SvdError` on a non-zero return.  No arithmetic of the verify pass happens here, and
there is no fallback: when the library is missing or cannot be loaded, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsvd.so")

SVD_OK = 0
SVD_ERR_INVALID_ARG = -1
SVD_ERR_UNSUPPORTED = -2
SVD_ERR_CUDA = -3
SVD_ERR_WORKSPACE = -4
SVD_ERR_TIMEOUT = -5

SVD_ST_BAD_TOKEN = 1
SVD_ST_Q_ZERO = 2
SVD_ST_BAD_PROB = 4
SVD_ST_ZERO_RESIDUAL = 8
SVD_ST_EMPTY = 16

SVD_LAYOUT_CANONICAL = 0
SVD_LAYOUT_NATIVE = 1
SVD_LAYOUT_Q4K = 2
SVD_LAYOUT_Q4K_NATIVE = 3
SVD_F_PDL = 1
SVD_F_FRAGMENT_MMA = 2
SVD_POLL_DEFAULT = 0xFFFFFFFF
SVD_C_MAX = 32
SVD_K_MAX = 32
SVD_KV_HEAD_DIM = 128
SVD_KV_UNIT_POSITIONS = 16
SVD_KV_UNIT_BYTES = 3328

# Every symbol include/svd.h declares (checked by the CPU test suite).
EXPORTS = (
    "svd_error_string", "svd_last_cuda_error", "svd_native_sizes", "svd_q4k_native_sizes",
    "svd_repack_weights",
    "svd_unpack_weights", "svd_verify_linear_workspace_bytes", "svd_verify_linear",
    "svd_verify_linear_noalloc", "svd_verify_chain_workspace_bytes", "svd_verify_chain",
    "svd_verify_status", "svd_verify_inject_stall",
    "svd_sampler_workspace_bytes", "svd_sampler_probs", "svd_lm_head_workspace_bytes",
    "svd_lm_head_softmax", "svd_accept", "svd_graph_begin", "svd_graph_end", "svd_graph_launch",
    "svd_graph_destroy", "svd_device_sm_count",
    "svd_expected_tokens_per_pass", "svd_speedup", "svd_best_depth", "svd_spec_adapt_create",
    "svd_spec_adapt_observe", "svd_spec_adapt_alpha", "svd_spec_adapt_depth",
    "svd_spec_adapt_destroy", "svd_ngram_create", "svd_ngram_append", "svd_ngram_propose",
    "svd_ngram_length", "svd_ngram_destroy",
    "svd_kv_cache_bytes", "svd_kv_repack", "svd_kv_unpack", "svd_kv_append",
    "svd_kv_attention_workspace_bytes", "svd_kv_attention", "svd_kv_attention_append",
)


class SvdError(RuntimeError):
    def __init__(self, fn: str, code: int):
        detail = svd_error_string(code)
        if code == SVD_ERR_CUDA:
            detail += f" (cudaError {svd_last_cuda_error()})"
        super().__init__(f"{fn}: {detail}")
        self.code = code


class _QWeight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("in_features", ctypes.c_int64), ("out_features", ctypes.c_int64),
                ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class _Sampler(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_p", ctypes.c_float),
                ("min_p", ctypes.c_float), ("greedy", ctypes.c_int32)]


class QWeight:
    """A 4-bit matrix on the device: codes and scales tensors plus its shape and layout."""

    def __init__(self, codes, scales, in_features: int, out_features: int, layout: int):
        self.codes, self.scales = codes, scales
        self.in_features, self.out_features, self.layout = int(in_features), int(out_features), int(layout)

    def _c(self) -> _QWeight:
        return _QWeight(_ptr(self.codes), _ptr(self.scales), self.in_features, self.out_features,
                        self.layout, 0)


class _LinearOp(ctypes.Structure):
    _fields_ = [("W", _QWeight), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


class Sampler:
    def __init__(self, temperature=0.6, top_p=0.95, min_p=0.05, greedy=False):
        self.temperature, self.top_p, self.min_p, self.greedy = temperature, top_p, min_p, greedy

    def _c(self) -> _Sampler:
        return _Sampler(float(self.temperature), float(self.top_p), float(self.min_p),
                        int(bool(self.greedy)))


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Open libsvd.so (once).  Raises when it is missing: there is no fallback path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libsvd.so not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        P, i32, i64, u64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                                ctypes.c_size_t)
        sig = {
            "svd_error_string": (ctypes.c_char_p, [i32]),
            "svd_last_cuda_error": (i32, []),
            "svd_device_sm_count": (i32, []),
            "svd_native_sizes": (i32, [i64, i64, P, P]),
            "svd_q4k_native_sizes": (i32, [i64, i64, P, P]),
            "svd_repack_weights": (i32, [P, P, P, P]),
            "svd_unpack_weights": (i32, [P, P, P, P]),
            "svd_verify_linear_workspace_bytes": (sz, [i64, i64, i32]),
            "svd_verify_linear": (i32, [P, P, i32, P, P, sz, i32, P]),
            "svd_verify_linear_noalloc": (i32, [P, P, i32, P, i32, P]),
            "svd_verify_chain_workspace_bytes": (sz, [P, i32, i32]),
            "svd_verify_chain": (i32, [P, i32, i32, P, sz, i32, P]),
            "svd_verify_status": (i32, [P, sz, P, P]),
            "svd_verify_inject_stall": (i32, [P, sz, ctypes.c_uint32, P]),
            "svd_sampler_workspace_bytes": (sz, [i32, i64]),
            "svd_sampler_probs": (i32, [P, i32, i64, P, P, P, P, sz, P]),
            "svd_lm_head_workspace_bytes": (sz, [i64, i64, i32]),
            "svd_lm_head_softmax": (i32, [P, P, i32, P, P, P, P, P, P, sz, P]),
            "svd_accept": (i32, [P, P, P, P, P, P, i64, i32, i64, u64, u64, P, P, P, P, P]),
            "svd_graph_begin": (i32, [P]),
            "svd_graph_end": (i32, [P, P]),
            "svd_graph_launch": (i32, [P, P]),
            "svd_graph_destroy": (None, [P]),
            "svd_expected_tokens_per_pass": (ctypes.c_double, [ctypes.c_double, i32]),
            "svd_speedup": (ctypes.c_double, [ctypes.c_double, i32, ctypes.c_double]),
            "svd_best_depth": (i32, [ctypes.c_double, ctypes.c_double, i32]),
            "svd_spec_adapt_create": (P, [i32, ctypes.c_double, ctypes.c_double, ctypes.c_double]),
            "svd_spec_adapt_observe": (i32, [P, P, P, i64, i32]),
            "svd_spec_adapt_alpha": (ctypes.c_double, [P]),
            "svd_spec_adapt_depth": (i32, [P]),
            "svd_spec_adapt_destroy": (None, [P]),
            "svd_ngram_create": (P, [i32]),
            "svd_ngram_append": (i32, [P, P, i64]),
            "svd_ngram_propose": (i32, [P, P, i32]),
            "svd_ngram_length": (i64, [P]),
            "svd_ngram_destroy": (None, [P]),
            "svd_kv_cache_bytes": (sz, [i32, i32]),
            "svd_kv_repack": (i32, [P, P, P, P, i32, i32, i32, i32, P, i32, P]),
            "svd_kv_unpack": (i32, [P, i32, i32, i32, i32, P, P, P, P, i32, P]),
            "svd_kv_append": (i32, [P, P, i32, i32, i32, i32, P, i32, P]),
            "svd_kv_attention_workspace_bytes": (sz, [i32, i32, i32]),
            "svd_kv_attention_append": (i32, [P, P, P, i32, P, i32, i32, i32, i32, i32,
                                              ctypes.c_float, P, P, sz, P]),
            "svd_kv_attention": (i32, [P, P, i32, i32, i32, i32, i32, ctypes.c_float, P, P, sz,
                                       P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
        return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int):
    if rc != SVD_OK:
        raise SvdError(fn, rc)


def svd_error_string(code: int) -> str:
    return load().svd_error_string(int(code)).decode()


def svd_last_cuda_error() -> int:
    return int(load().svd_last_cuda_error())


def svd_device_sm_count() -> int:
    return int(load().svd_device_sm_count())


def svd_native_sizes(in_features: int, out_features: int):
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check("svd_native_sizes",
           load().svd_native_sizes(in_features, out_features, ctypes.byref(cb), ctypes.byref(sb)))
    return cb.value, sb.value


def svd_q4k_native_sizes(in_features: int, out_features: int):
    cb, hb = ctypes.c_size_t(), ctypes.c_size_t()
    _check("svd_q4k_native_sizes", load().svd_q4k_native_sizes(
        in_features, out_features, ctypes.byref(cb), ctypes.byref(hb)))
    return cb.value, hb.value


def svd_repack_weights(src: QWeight, dst_codes, dst_scales, stream=None):
    w = src._c()
    _check("svd_repack_weights", load().svd_repack_weights(
        ctypes.byref(w), _ptr(dst_codes), _ptr(dst_scales), _stream(stream)))


def svd_unpack_weights(src: QWeight, dst_codes, dst_scales, stream=None):
    w = src._c()
    _check("svd_unpack_weights", load().svd_unpack_weights(
        ctypes.byref(w), _ptr(dst_codes), _ptr(dst_scales), _stream(stream)))


def svd_verify_linear_workspace_bytes(in_features: int, out_features: int, C: int) -> int:
    return int(load().svd_verify_linear_workspace_bytes(in_features, out_features, C))


def svd_verify_linear(W: QWeight, X, C: int, Y, workspace=None, workspace_bytes: int = 0,
                      flags: int = 0, stream=None):
    w = W._c()
    if workspace is not None and not workspace_bytes and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("svd_verify_linear", load().svd_verify_linear(
        ctypes.byref(w), _ptr(X), int(C), _ptr(Y), _ptr(workspace), int(workspace_bytes),
        int(flags), _stream(stream)))


def svd_verify_linear_noalloc(W: QWeight, X, C: int, Y, flags: int = 0, stream=None):
    """svd_verify_linear without a workspace argument: the scratch lives in the library's own
    device memory (for callers that cannot allocate)."""
    w = W._c()
    _check("svd_verify_linear_noalloc", load().svd_verify_linear_noalloc(
        ctypes.byref(w), _ptr(X), int(C), _ptr(Y), int(flags), _stream(stream)))


def _ops_array(ops):
    """ops: sequence of (QWeight, X, Y) -> ctypes array of svd_linear_op."""
    arr = (_LinearOp * len(ops))()
    for i, (W, X, Y) in enumerate(ops):
        arr[i].W = W._c()
        arr[i].X = _ptr(X)
        arr[i].Y = _ptr(Y)
    return arr


def svd_verify_chain_workspace_bytes(ops, C: int) -> int:
    arr = _ops_array(ops)
    return int(load().svd_verify_chain_workspace_bytes(arr, len(ops), int(C)))


def svd_verify_chain(ops, C: int, workspace, workspace_bytes: int = 0, flags: int = 0,
                     stream=None):
    arr = _ops_array(ops)
    if not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("svd_verify_chain", load().svd_verify_chain(
        arr, len(ops), int(C), _ptr(workspace), int(workspace_bytes), int(flags), _stream(stream)))


def svd_verify_status(workspace, workspace_bytes: int = 0, stream=None):
    """Returns (rc, bits): rc is SVD_OK or SVD_ERR_TIMEOUT (a bounded wait gave up); the status
    word is cleared.  Other codes raise."""
    if not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    bits = ctypes.c_uint32(0)
    rc = int(load().svd_verify_status(_ptr(workspace), int(workspace_bytes), ctypes.byref(bits),
                                      _stream(stream)))
    if rc not in (SVD_OK, SVD_ERR_TIMEOUT):
        raise SvdError("svd_verify_status", rc)
    return rc, int(bits.value)


def svd_verify_inject_stall(workspace, polls, workspace_bytes: int = 0, stream=None):
    """Test hook: later kernels on this workspace issue no weight copy and give up a wait after
    `polls` polls; polls=None turns it off."""
    if polls is None:
        polls = SVD_POLL_DEFAULT
    if not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("svd_verify_inject_stall", load().svd_verify_inject_stall(
        _ptr(workspace), int(workspace_bytes), int(polls), _stream(stream)))


def svd_sampler_workspace_bytes(rows: int, V: int) -> int:
    return int(load().svd_sampler_workspace_bytes(rows, V))


def svd_sampler_probs(logits, rows: int, V: int, sampler: Sampler, probs, argmax, workspace,
                      workspace_bytes: int = 0, stream=None):
    s = sampler._c()
    if not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("svd_sampler_probs", load().svd_sampler_probs(
        _ptr(logits), int(rows), int(V), ctypes.byref(s), _ptr(probs), _ptr(argmax),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def svd_lm_head_workspace_bytes(hidden: int, vocab: int, C: int) -> int:
    return int(load().svd_lm_head_workspace_bytes(hidden, vocab, C))


def svd_lm_head_softmax(W: QWeight, H, C: int, sampler: Sampler, logits, probs, argmax,
                        workspace, workspace_bytes: int = 0, stream=None, lse=None):
    w = W._c()
    s = sampler._c()
    if not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("svd_lm_head_softmax", load().svd_lm_head_softmax(
        ctypes.byref(w), _ptr(H), int(C), ctypes.byref(s), _ptr(logits), _ptr(probs),
        _ptr(argmax), _ptr(lse), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def svd_accept(p, draft, n_windows: int, k: int, V: int, out_tokens, n_emitted, status,
               q=None, p_rows=None, q_rows=None, target_argmax=None, seed: int = 0,
               window_offset: int = 0, uniforms=None, stream=None):
    _check("svd_accept", load().svd_accept(
        _ptr(p), _ptr(p_rows), _ptr(q), _ptr(q_rows), _ptr(target_argmax), _ptr(draft),
        int(n_windows), int(k), int(V), int(seed) & (2**64 - 1),
        int(window_offset) & (2**64 - 1), _ptr(uniforms), _ptr(out_tokens), _ptr(n_emitted),
        _ptr(status), _stream(stream)))


class Graph:
    """An instantiated CUDA graph of library calls (svd_graph_*)."""

    def __init__(self, handle: int):
        self.handle = handle

    def launch(self, stream=None):
        _check("svd_graph_launch", load().svd_graph_launch(self.handle, _stream(stream)))

    def destroy(self):
        if self.handle:
            load().svd_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def svd_graph_begin(stream=None):
    _check("svd_graph_begin", load().svd_graph_begin(_stream(stream)))


def svd_graph_end(stream=None) -> Graph:
    h = ctypes.c_void_p()
    _check("svd_graph_end", load().svd_graph_end(_stream(stream), ctypes.byref(h)))
    return Graph(h.value)


# ---- host-side companions: depth policy and n-gram drafter ------------------------------
def _host_i32(a):
    """A contiguous host int32 array (numpy) for a host-pointer argument."""
    import numpy as np
    if hasattr(a, "detach"):  # a torch tensor: must live on the host
        if a.device.type != "cpu":
            raise ValueError("host array expected")
        a = a.detach().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def svd_expected_tokens_per_pass(alpha: float, k: int) -> float:
    return float(load().svd_expected_tokens_per_pass(float(alpha), int(k)))


def svd_speedup(alpha: float, k: int, draft_cost: float) -> float:
    return float(load().svd_speedup(float(alpha), int(k), float(draft_cost)))


def svd_best_depth(alpha: float, draft_cost: float, k_max: int) -> int:
    r = int(load().svd_best_depth(float(alpha), float(draft_cost), int(k_max)))
    _check("svd_best_depth", r if r < 0 else SVD_OK)
    return r


class SpecAdapt:
    """svd_spec_adapt: the draft depth throttled by the measured acceptance."""

    def __init__(self, k_max: int, draft_cost: float, threshold: float = 0.35,
                 half_life_windows: float = 256.0):
        self._h = load().svd_spec_adapt_create(int(k_max), float(draft_cost), float(threshold),
                                               float(half_life_windows))
        if not self._h:
            raise SvdError("svd_spec_adapt_create", SVD_ERR_INVALID_ARG)

    def observe(self, n_emitted, k: int, status=None):
        ne = _host_i32(n_emitted)
        st = None if status is None else _host_i32(status)
        _check("svd_spec_adapt_observe", load().svd_spec_adapt_observe(
            self._h, ne.ctypes.data, None if st is None else st.ctypes.data, ne.size, int(k)))

    @property
    def alpha(self) -> float:
        return float(load().svd_spec_adapt_alpha(self._h))

    @property
    def depth(self) -> int:
        return int(load().svd_spec_adapt_depth(self._h))

    def close(self):
        if getattr(self, "_h", None):
            load().svd_spec_adapt_destroy(self._h)
            self._h = None

    __del__ = close


class NgramDrafter:
    """svd_ngram: drafts from the continuation that followed the last key_len tokens before."""

    def __init__(self, key_len: int = 6):
        self._h = load().svd_ngram_create(int(key_len))
        if not self._h:
            raise SvdError("svd_ngram_create", SVD_ERR_INVALID_ARG)

    def append(self, tokens):
        t = _host_i32(tokens)
        _check("svd_ngram_append", load().svd_ngram_append(self._h, t.ctypes.data, t.size))

    def propose(self, k_max: int):
        import numpy as np
        out = np.empty(max(int(k_max), 1), dtype=np.int32)
        r = int(load().svd_ngram_propose(self._h, out.ctypes.data, int(k_max)))
        _check("svd_ngram_propose", r if r < 0 else SVD_OK)
        return out[:r].copy()

    def __len__(self) -> int:
        return int(load().svd_ngram_length(self._h))

    def close(self):
        if getattr(self, "_h", None):
            load().svd_ngram_destroy(self._h)
            self._h = None

    __del__ = close


def svd_kv_cache_bytes(n_kv_heads: int, capacity: int) -> int:
    return int(load().svd_kv_cache_bytes(int(n_kv_heads), int(capacity)))


def svd_kv_repack(k_codes, k_scales, v_codes, v_scales, n_kv_heads: int, ld: int,
                  pos_begin: int, pos_end: int, cache, capacity: int, stream=None):
    _check("svd_kv_repack", load().svd_kv_repack(
        _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), int(n_kv_heads), int(ld),
        int(pos_begin), int(pos_end), _ptr(cache), int(capacity), _stream(stream)))


def svd_kv_unpack(cache, capacity: int, n_kv_heads: int, pos_begin: int, pos_end: int,
                  k_codes, k_scales, v_codes, v_scales, ld: int, stream=None):
    _check("svd_kv_unpack", load().svd_kv_unpack(
        _ptr(cache), int(capacity), int(n_kv_heads), int(pos_begin), int(pos_end), _ptr(k_codes),
        _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), int(ld), _stream(stream)))


def svd_kv_append(k, v, ld: int, C: int, n_kv_heads: int, n_past: int, cache, capacity: int,
                  stream=None):
    _check("svd_kv_append", load().svd_kv_append(
        _ptr(k), _ptr(v), int(ld), int(C), int(n_kv_heads), int(n_past), _ptr(cache),
        int(capacity), _stream(stream)))


def svd_kv_attention_workspace_bytes(n_q_heads: int, n_kv_heads: int, C: int) -> int:
    return int(load().svd_kv_attention_workspace_bytes(int(n_q_heads), int(n_kv_heads), int(C)))


def svd_kv_attention(q, cache, capacity: int, n_q_heads: int, n_kv_heads: int, n_past: int,
                     C: int, scale: float, out, workspace, workspace_bytes: int = 0,
                     stream=None):
    if not workspace_bytes and workspace is not None and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("svd_kv_attention", load().svd_kv_attention(
        _ptr(q), _ptr(cache), int(capacity), int(n_q_heads), int(n_kv_heads), int(n_past), int(C),
        float(scale), _ptr(out), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def svd_kv_attention_append(q, k, v, ld: int, cache, capacity: int, n_q_heads: int,
                            n_kv_heads: int, n_past: int, C: int, scale: float, out, workspace,
                            workspace_bytes: int = 0, stream=None):
    if not workspace_bytes and workspace is not None and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("svd_kv_attention_append", load().svd_kv_attention_append(
        _ptr(q), _ptr(k), _ptr(v), int(ld), _ptr(cache), int(capacity), int(n_q_heads),
        int(n_kv_heads), int(n_past), int(C), float(scale), _ptr(out), _ptr(workspace),
        int(workspace_bytes), _stream(stream)))
