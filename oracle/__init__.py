"""The oracle: a plain, slow fp64 CPU restatement of the verify pass.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library never links it, and
the two share no source: the only common module is the seeded input generator, which holds none
of the method's arithmetic.

The arithmetic lives in ``orc.c`` (compiled with gcc, loaded with ctypes); the closed forms of
the pages live in :mod:`oracle.formulas`.  Every function cites the passage it follows.

Parity status: every function here is pinned by a ``-m "not gpu"`` test (see the test files
named ``test_oracle_*``), except where a docstring says "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orc.c")
_LIB = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``orc.c`` into ``liborc.so`` (plain gcc, -O2, OpenMP; no -march flags; no fused
    multiply-adds, so fp32 steps round as written on every host)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, u64, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_double
            L.orc_f16_to_f64.restype = dbl
            L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f64.restype = dbl
            L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.orc_verify_linear.restype = None
            L.orc_verify_linear.argtypes = [P, P, i64, i64, P, i64, P, P, i32]
            L.orc_sampler.restype = None
            L.orc_sampler.argtypes = [P, i64, i64, dbl, dbl, dbl, i32, P, P, P, P, i32]
            L.orc_philox4x32_10.restype = None
            L.orc_philox4x32_10.argtypes = [P, P, P]
            L.orc_uniforms.restype = None
            L.orc_uniforms.argtypes = [u64, u64, ctypes.c_uint32, P, P]
            L.orc_accept.restype = None
            L.orc_accept.argtypes = [P, P, P, P, P, P, i64, i32, i64, u64, u64, P, P, P, P, P, P,
                                     i32]
            L.orc_kv_attention.restype = None
            L.orc_kv_attention.argtypes = [P, P, P, P, P, i64, i64, i64, i64, i64, i64, dbl, P, P,
                                           i32]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_kv_quantize.restype = None
            L.orc_kv_quantize.argtypes = [P, P, i64, i64, P, P, P, P]
            L.orc_max_threads.restype = i32
            L.orc_max_threads.argtypes = []
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(lib().orc_max_threads())


def f16_to_f64(bits: int) -> float:
    """IEEE binary16 bit pattern -> value, decoded from the format's definition."""
    return float(lib().orc_f16_to_f64(int(bits) & 0xFFFF))


def bf16_to_f64(bits: int) -> float:
    """bfloat16 bit pattern -> value, decoded from the format's definition."""
    return float(lib().orc_bf16_to_f64(int(bits) & 0xFFFF))


def verify_linear(codes, scales, x_bf16, nthreads: int = 0):
    """y[c][j] = sum_i s[j][i/32] * (code[j][i]-8) * x[c][i] in fp64, and a = sum |terms|.

    codes: uint8 [out, in/2] (low nibble = even input); scales: uint16 fp16 bits [out, in/32];
    x_bf16: uint16 bf16 bits [C, in].  Returns (y, a), both float64 [C, out].
    Follows "100 tokens per second ..." ("How speculative decoding gets past a per-token
    wall": one weight read applied to a K-wide batch of activations).
    """
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    out_f, half_in = codes.shape
    in_f = 2 * half_in
    assert scales.shape == (out_f, in_f // 32) and in_f % 32 == 0
    C = x_bf16.shape[0]
    assert x_bf16.shape == (C, in_f)
    y = np.empty((C, out_f), np.float64)
    a = np.empty((C, out_f), np.float64)
    lib().orc_verify_linear(_p(codes), _p(scales), in_f, out_f, _p(x_bf16), C, _p(y), _p(a),
                            int(nthreads or max_threads()))
    return y, a


def sampler(logits, temperature=0.6, top_p=0.95, min_p=0.05, greedy=False, nthreads: int = 0):
    """Per-row temperature / min-p / top-p sampler distribution (fp64).

    logits: float32 [rows, V].  Returns (probs float64 [rows, V], argmax int32 [rows],
    n_kept int64 [rows], flags int32 [rows]).  Follows "Decode is memory-bound ..." ("Two
    things the math says to do": temperature 0.6, top-p 0.95, min-p 0.05); the order of
    the filters is a reading (both act on the same un-renormalised p).
    """
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    if logits.ndim == 1:
        logits = logits[None, :]
    rows, V = logits.shape
    probs = np.empty((rows, V), np.float64)
    am = np.empty(rows, np.int32)
    nk = np.empty(rows, np.int64)
    fl = np.empty(rows, np.int32)
    lib().orc_sampler(_p(logits), rows, V, float(temperature), float(top_p), float(min_p),
                      int(bool(greedy)), _p(probs), _p(am), _p(nk), _p(fl),
                      int(nthreads or max_threads()))
    return probs, am, nk, fl


def philox4x32_10(counter, key):
    """Philox4x32-10 (Salmon et al., SC'11) of a 4-word counter under a 2-word key."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniforms(seed: int, window: int, pos: int):
    """(u, u') of window `window`, position `pos`: words 0 and 1 of Philox, (w>>8)*2^-24."""
    u = ctypes.c_double()
    u2 = ctypes.c_double()
    lib().orc_uniforms(int(seed) & (2**64 - 1), int(window) & (2**64 - 1), int(pos),
                       ctypes.byref(u), ctypes.byref(u2))
    return u.value, u2.value


def accept(p, draft, q=None, target_argmax=None, seed=0, window_offset=0, uniforms=None,
           p_rows=None, q_rows=None, nthreads: int = 0, return_margin: bool = False):
    """Greedy (q None) or sampled acceptance of every window.

    p: float32 [P, V] rows (indexed by p_rows [n, k+1] when given, else [n*(k+1), V]);
    q: float32 rows likewise with q_rows [n, k]; draft: int32 [n, k].
    Returns (tokens int32 [n, k+1] padded with -1, n_emitted int32 [n], status int32 [n],
    near int32 [n]; with return_margin also margin float64 [n], the distance of each draw's
    u' to the nearer edge of its token's interval, +inf without a draw).  Follows "100 tokens per second ..." ("How speculative decoding gets past
    a per-token wall"), "Decode is memory-bound ..." ("Speculative decoding") and the HN
    thread's "D E F" example.
    """
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    n, k = draft.shape
    p = np.ascontiguousarray(p, dtype=np.float32)
    V = p.shape[-1]
    p = p.reshape(-1, V)
    if q is not None:
        q = np.ascontiguousarray(q, dtype=np.float32).reshape(-1, V)
    pr = None if p_rows is None else np.ascontiguousarray(p_rows, dtype=np.int64)
    qr = None if q_rows is None else np.ascontiguousarray(q_rows, dtype=np.int64)
    ta = None if target_argmax is None else np.ascontiguousarray(target_argmax, dtype=np.int32)
    un = None if uniforms is None else np.ascontiguousarray(uniforms, dtype=np.float32)
    tok = np.empty((n, k + 1), np.int32)
    ne = np.empty(n, np.int32)
    st = np.empty(n, np.int32)
    nr = np.empty(n, np.int32)
    mg = np.empty(n, np.float64)
    lib().orc_accept(_p(p), _p(pr), _p(q), _p(qr), _p(ta), _p(draft), n, k, V,
                     int(seed) & (2**64 - 1), int(window_offset) & (2**64 - 1), _p(un),
                     _p(tok), _p(ne), _p(st), _p(nr), _p(mg), int(nthreads or max_threads()))
    if return_margin:
        return tok, ne, st, nr, mg
    return tok, ne, st, nr


def kv_attention(q_bf16, k_codes, k_scales, v_codes, v_scales, n_past: int, scale=None,
                 nthreads: int = 0):
    """Attention of the C window queries over a q8_0-key / q4_0-value cache, in fp64.

    q_bf16: uint16 bf16 bits [C, Hq, D]; k_codes: int8 [Hkv, ld, D]; k_scales: uint16 fp16 bits
    [Hkv, ld, D/32]; v_codes: uint8 [Hkv, ld, D/2] (low nibble = even dimension); v_scales:
    uint16 fp16 bits [Hkv, ld, D/32].  The window occupies cache positions n_past .. n_past+C-1
    and position c attends to 0 .. n_past+c; query head h reads kv head h // (Hq // Hkv).
    scale defaults to 1/sqrt(D).  Returns (o, a), float64 [C, Hq, D]: the attention output and
    sum_j p_j |v_j| (the scale of the parity tolerance).  Follows "Decode is memory-bound ..."
    ("The ceiling": at long context the whole KV cache is read on every pass) and "100 tokens
    per second ..." ("The wall": a 32K context with the cache at q8_0/q4_0).
    """
    q_bf16 = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    k_codes = np.ascontiguousarray(k_codes, dtype=np.int8)
    k_scales = np.ascontiguousarray(k_scales, dtype=np.uint16)
    v_codes = np.ascontiguousarray(v_codes, dtype=np.uint8)
    v_scales = np.ascontiguousarray(v_scales, dtype=np.uint16)
    C, Hq, D = q_bf16.shape
    Hkv, ld, _ = k_codes.shape
    assert D % 32 == 0 and Hq % Hkv == 0 and k_codes.shape == (Hkv, ld, D)
    assert k_scales.shape == (Hkv, ld, D // 32) and v_scales.shape == (Hkv, ld, D // 32)
    assert v_codes.shape == (Hkv, ld, D // 2) and 0 <= n_past and n_past + C <= ld
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.empty((C, Hq, D), np.float64)
    a = np.empty((C, Hq, D), np.float64)
    lib().orc_kv_attention(_p(q_bf16), _p(k_codes), _p(k_scales), _p(v_codes), _p(v_scales),
                           Hq, Hkv, D, ld, int(n_past), C, float(scale), _p(o), _p(a),
                           int(nthreads or max_threads()))
    return o, a


def f32_to_f16_bits(x: float) -> int:
    """fp32 value -> IEEE binary16 bits, round to nearest even (from the formats' definitions)."""
    return int(lib().orc_f32_to_f16(ctypes.c_float(x)))


def kv_quantize(k, v):
    """q8_0 keys and q4_0 values of rows of fp32 keys and values (the cache's write side).

    k, v: float32 [rows, D], D % 32 == 0.  Returns (k_codes int8 [rows, D], k_scales uint16 fp16
    bits [rows, D/32], v_codes uint8 [rows, D/2] (low nibble = even dimension), v_scales uint16
    [rows, D/32]).  Follows "100 tokens per second ..." ("The wall": KV cache at q8_0/q4_0); the
    block definitions are a reading (those of the llama.cpp types of the same names).
    """
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    rows, D = k.shape
    assert v.shape == (rows, D) and D % 32 == 0
    kc = np.empty((rows, D), np.int8)
    ks = np.empty((rows, D // 32), np.uint16)
    vc = np.zeros((rows, D // 2), np.uint8)
    vs = np.empty((rows, D // 32), np.uint16)
    lib().orc_kv_quantize(_p(k), _p(v), rows, D, _p(kc), _p(ks), _p(vc), _p(vs))
    return kc, ks, vc, vs
