"""GPU parity of the KV-read attention (svd_kv_attention over a native cache written by
svd_kv_repack) against the fp64 oracle, element by element, and of the cache's write side
(svd_kv_append: codes and scales bit-exact against the oracle's quantiser).

Tolerance, from the arithmetic of the kernel: query-key products are exact (f16 codes and queries)
and summed in fp32; the only coarse rounding is P' = p * d_v to bfloat16 (relative 2^-9 per term)
in the value product, so |o_gpu - o| <= 2^-9 sum_j p_j |v_j| plus fp32 noise; the test allows
2^-8 * a, a = sum_j p_j |v_j| from the oracle."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, lib, to_dev

pytestmark = pytest.mark.gpu

D = synth.HEAD_DIM
TOL = 2.0 ** -8


def _native(kc, ks, vc, vs, capacity, fill=None, ranges=None):
    lib()
    Hkv, ld, _ = kc.shape
    cache = torch.empty(svd.svd_kv_cache_bytes(Hkv, capacity), dtype=torch.uint8, device=DEV)
    if fill is not None:
        cache.fill_(fill)
    dev = [to_dev(a) for a in (kc, ks, vc, vs)]
    for p0, p1 in ([(0, ld)] if ranges is None else ranges):
        svd.svd_kv_repack(*dev, Hkv, ld, p0, p1, cache, capacity)
    return cache


def _attend(q, cache, capacity, Hq, Hkv, n_past, scale=None, ws=None):
    C = q.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qd = to_dev(q)
    out = torch.full((C, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    if ws is None:
        ws = torch.zeros(svd.svd_kv_attention_workspace_bytes(Hq, Hkv, C), dtype=torch.uint8,
                         device=DEV)
    svd.svd_kv_attention(qd, cache, capacity, Hq, Hkv, n_past, C, scale, out, ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "a bounded wait gave up"
    return out.cpu().numpy().astype(np.float64)


def _check(o, o_ref, a_ref):
    err = np.abs(o - o_ref)
    bad = ~(err <= TOL * a_ref)
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outputs out of tolerance; worst "
                           f"{np.nanmax(err / np.maximum(a_ref, 1e-300)):.3e} of a")
    return float(np.max(err / np.maximum(a_ref, 1e-300)))


@pytest.mark.parametrize("Hkv,ld,capacity,ranges", [
    (1, 16, 16, None), (3, 50, 53, None), (8, 300, 320, [(0, 17), (17, 300)]),
    (2, 1000, 1000, [(0, 999), (999, 1000)]),
])
def test_repack_roundtrip_is_exact(Hkv, ld, capacity, ranges):
    kc, ks, vc, vs = synth.kv_cache(Hkv, ld, D, seed=ld)
    cache = _native(kc, ks, vc, vs, capacity, ranges=ranges)
    out = [torch.zeros_like(to_dev(a)) for a in (kc, ks, vc, vs)]
    svd.svd_kv_unpack(cache, capacity, Hkv, 0, ld, *out, ld)
    torch.cuda.synchronize()
    for got, want in zip(out, (kc, ks, vc, vs)):
        g = got.cpu().numpy()
        assert np.array_equal(g.view(want.dtype) if g.dtype != want.dtype else g, want)


@pytest.mark.parametrize("Hq,Hkv,n_past,C", [
    (1, 1, 0, 1),          # one position
    (8, 8, 0, 4),          # the window alone, G = 1
    (40, 8, 0, 4),         # the stack's grouping (G = 5), empty context
    (40, 8, 37, 4),        # ragged last unit
    (40, 8, 1000, 4),
    (40, 8, 4093, 4),      # the window crosses a 16-position unit boundary
    (40, 8, 2000, 1), (40, 8, 2000, 2), (40, 8, 2000, 6),
    (40, 8, 2000, 8),      # 40 rows: two row groups
    (4, 2, 100, 3), (6, 1, 500, 4), (7, 1, 300, 4), (16, 16, 3000, 4), (2, 1, 15, 1),
    (2, 1, 16, 1), (2, 1, 17, 2),
])
def test_matches_oracle(Hq, Hkv, n_past, C):
    L = n_past + C
    capacity = L + 21
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=L + 7 * Hq)
    q = synth.queries(C, Hq, D, seed=C + Hq)
    cache = _native(kc, ks, vc, vs, capacity)
    o = _attend(q, cache, capacity, Hq, Hkv, n_past)
    o_ref, a_ref = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    _check(o, o_ref, a_ref)


def test_bytes_past_the_window_are_never_used():
    # The cache is pre-filled with 0xFF (NaN scales, codes -1 / 15) and only positions
    # 0 .. n_past + C - 1 are written: the unit tail past the window must not leak in.
    Hq, Hkv, n_past, C = 40, 8, 90, 4
    L = n_past + C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=3)
    q = synth.queries(C, Hq, D, seed=4)
    cache = _native(kc, ks, vc, vs, L + 40, fill=0xFF)
    o = _attend(q, cache, L + 40, Hq, Hkv, n_past)
    assert np.isfinite(o).all()
    o_ref, a_ref = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    _check(o, o_ref, a_ref)


def test_explicit_scale_and_peaked_scores():
    # A large scale makes the softmax nearly one-hot: exercises the lazy running max (scores
    # jumping by far more than 8 in base 2 between units).
    Hq, Hkv, n_past, C = 8, 2, 700, 4
    L = n_past + C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=9)
    q = synth.queries(C, Hq, D, seed=10)
    cache = _native(kc, ks, vc, vs, L)
    for scale in (0.5, 2.0, 1e-3):
        o = _attend(q, cache, L, Hq, Hkv, n_past, scale=scale)
        o_ref, a_ref = oracle.kv_attention(q, kc, ks, vc, vs, n_past, scale=scale)
        _check(o, o_ref, a_ref)


def test_long_context_one_kv_head():
    Hq, Hkv, n_past, C = 5, 1, 131068, 4
    L = n_past + C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=11)
    q = synth.queries(C, Hq, D, seed=12)
    cache = _native(kc, ks, vc, vs, L)
    o = _attend(q, cache, L, Hq, Hkv, n_past)
    o_ref, a_ref = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    _check(o, o_ref, a_ref)


def test_full_size_32k_context_sampled_heads():
    # The benchmark's per-layer shape: 40 query heads over 8 kv heads, 32K positions (the window's
    # four at the end), the launch the benchmark times.  The oracle checks two kv heads (ten query
    # heads, all four window rows) on their own slices of the cache.
    Hq, Hkv, C = synth.N_Q_HEADS, synth.N_KV_HEADS, 4
    L = 32768
    n_past = L - C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=2024)
    q = synth.queries(C, Hq, D, seed=2025)
    cache = _native(kc, ks, vc, vs, L)
    o = _attend(q, cache, L, Hq, Hkv, n_past)
    G = Hq // Hkv
    for g in (0, 5):
        sl = slice(g, g + 1)
        o_ref, a_ref = oracle.kv_attention(q[:, g * G:(g + 1) * G], kc[sl], ks[sl], vc[sl], vs[sl],
                                           n_past)
        _check(o[:, g * G:(g + 1) * G], o_ref, a_ref)


def test_repeat_runs_are_bitwise_identical():
    Hq, Hkv, n_past, C = 40, 8, 5000, 4
    L = n_past + C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=13)
    q = synth.queries(C, Hq, D, seed=14)
    cache = _native(kc, ks, vc, vs, L)
    o1 = _attend(q, cache, L, Hq, Hkv, n_past)
    o2 = _attend(q, cache, L, Hq, Hkv, n_past)
    assert np.array_equal(o1, o2)


def test_bad_arguments_are_rejected():
    lib()
    Hq, Hkv, C, L = 8, 2, 4, 64
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=1)
    cache = _native(kc, ks, vc, vs, L)
    q = to_dev(synth.queries(C, Hq, D, seed=2))
    out = torch.empty((C, Hq, D), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_kv_attention_workspace_bytes(Hq, Hkv, C), dtype=torch.uint8, device=DEV)
    with pytest.raises(svd.SvdError):
        svd.svd_kv_attention(q, cache, L, Hq, 3, L - C, C, 0.1, out, ws)       # Hq % Hkv
    with pytest.raises(svd.SvdError):
        svd.svd_kv_attention(q, cache, L, Hq, Hkv, L - C + 1, C, 0.1, out, ws)  # past capacity
    with pytest.raises(svd.SvdError):
        svd.svd_kv_attention(q, cache, L, Hq, Hkv, L - C, C, -1.0, out, ws)    # scale
    with pytest.raises(svd.SvdError):
        svd.svd_kv_attention(q, cache, L, Hq, Hkv, L - C, C, 0.1, out, ws[:16])  # workspace
    with pytest.raises(svd.SvdError):
        svd.svd_kv_attention(q, cache[1:], L, Hq, Hkv, L - C, C, 0.1, out, ws)  # misaligned


def _window_kv(C, Hkv, ld, seed):
    """fp32 keys and values of a window, rows of ld floats (the kv heads' 128 values each at the
    front), with a zero block, a tie between the two largest value magnitudes and magnitudes
    from 1e-6 to 1e4."""
    g = np.random.default_rng(seed)
    k = np.zeros((C, ld), np.float32)
    v = np.zeros((C, ld), np.float32)
    for c in range(C):
        for h in range(Hkv):
            s = 10.0 ** g.uniform(-6, 4)
            k[c, h * D:(h + 1) * D] = g.normal(0, s, D)
            v[c, h * D:(h + 1) * D] = g.normal(0, s, D)
    k[0, 32:64] = 0.0
    v[0, 32:64] = 0.0
    v[-1, 5], v[-1, 9] = 3.0, -3.0
    v[-1, 0:32][np.abs(v[-1, 0:32]) > 2.5] = 0.5
    v[-1, 5], v[-1, 9] = 3.0, -3.0
    return k, v


@pytest.mark.parametrize("C,n_past,Hkv", [(4, 0, 8), (4, 29, 8), (1, 15, 2), (8, 100, 8),
                                          (3, 16, 1), (6, 8189, 8)])
def test_append_matches_the_oracle_quantiser(C, n_past, Hkv):
    lib()
    ld = Hkv * D + 64
    k, v = _window_kv(C, Hkv, ld, seed=C + n_past)
    capacity = n_past + C + 7
    # positions before the window hold an earlier cache, the rest a fill pattern
    kc0, ks0, vc0, vs0 = synth.kv_cache(Hkv, capacity, D, seed=3)
    cache = _native(kc0, ks0, vc0, vs0, capacity, ranges=[(0, n_past)] if n_past else [],
                    fill=0xA5)
    kd, vd = to_dev(k), to_dev(v)
    svd.svd_kv_append(kd, vd, ld, C, Hkv, n_past, cache, capacity)
    out = [torch.zeros_like(to_dev(a)) for a in (kc0, ks0, vc0, vs0)]
    svd.svd_kv_unpack(cache, capacity, Hkv, 0, n_past + C, *out, capacity)
    torch.cuda.synchronize()
    kc, ks, vc, vs = (o.cpu().numpy() for o in out)
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    rk = k[:, :Hkv * D].reshape(C * Hkv, D)
    rv = v[:, :Hkv * D].reshape(C * Hkv, D)
    qk, qks, qv, qvs = oracle.kv_quantize(rk, rv)
    for c in range(C):
        for h in range(Hkv):
            i, p = c * Hkv + h, n_past + c
            assert np.array_equal(kc[h, p], qk[i]) and np.array_equal(ks[h, p], qks[i])
            assert np.array_equal(vc[h, p], qv[i]) and np.array_equal(vs[h, p], qvs[i])
    # the positions before the window are untouched
    assert np.array_equal(kc[:, :n_past], kc0[:, :n_past])
    assert np.array_equal(vc[:, :n_past], vc0[:, :n_past])
    assert np.array_equal(vs[:, :n_past], vs0[:, :n_past])


def test_append_then_attend_matches_oracle():
    # The window's keys and values go in through svd_kv_append, then the window attends over the
    # whole cache: the oracle quantises the same rows and attends in fp64.
    lib()
    Hq, Hkv, n_past, C = 40, 8, 777, 4
    ld = Hkv * D
    L = n_past + C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=21)
    g = np.random.default_rng(22)
    k = g.normal(0, 3, (C, ld)).astype(np.float32)
    v = g.normal(0, 0.1, (C, ld)).astype(np.float32)
    cache = _native(kc, ks, vc, vs, L, ranges=[(0, n_past)])
    svd.svd_kv_append(to_dev(k), to_dev(v), ld, C, Hkv, n_past, cache, L)
    q = synth.queries(C, Hq, D, seed=23)
    o = _attend(q, cache, L, Hq, Hkv, n_past)
    qk, qks, qv, qvs = oracle.kv_quantize(k.reshape(C * Hkv, D), v.reshape(C * Hkv, D))
    for c in range(C):
        for h in range(Hkv):
            i = c * Hkv + h
            kc[h, n_past + c], ks[h, n_past + c] = qk[i], qks[i]
            vc[h, n_past + c], vs[h, n_past + c] = qv[i], qvs[i]
    o_ref, a_ref = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    _check(o, o_ref, a_ref)


def test_append_rejects_bad_arguments():
    lib()
    Hkv, C, L = 2, 4, 32
    cache = torch.zeros(svd.svd_kv_cache_bytes(Hkv, L), dtype=torch.uint8, device=DEV)
    k = torch.zeros((C, Hkv * D), dtype=torch.float32, device=DEV)
    with pytest.raises(svd.SvdError):
        svd.svd_kv_append(k, k, Hkv * D - 1, C, Hkv, 0, cache, L)     # ld too short
    with pytest.raises(svd.SvdError):
        svd.svd_kv_append(k, k, Hkv * D, C, Hkv, L - C + 1, cache, L)  # past capacity


@pytest.mark.parametrize("Hq,Hkv,n_past,C", [(40, 8, 1000, 4), (40, 8, 4093, 4), (10, 2, 14, 4),
                                             (40, 8, 2000, 8), (5, 1, 0, 3)])
def test_fused_append_equals_append_then_attend(Hq, Hkv, n_past, C):
    # svd_kv_attention_append (one kernel when the window's rows fit one row group, else the two
    # launches) leaves the same cache bytes as svd_kv_append followed by svd_kv_attention, and
    # the same output up to the summation order (the fused kernel splits the context slightly
    # differently), within 2^-16 of the values' scale; both match the oracle's tolerance.
    lib()
    L = n_past + C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=31)
    ld = Hkv * D + 32
    k, v = _window_kv(C, Hkv, ld, seed=32)
    q = synth.queries(C, Hq, D, seed=33)
    ranges = [(0, n_past)] if n_past else []
    c1 = _native(kc, ks, vc, vs, L, ranges=ranges, fill=0x5A)
    c2 = _native(kc, ks, vc, vs, L, ranges=ranges, fill=0x5A)
    kd, vd, qd = to_dev(k), to_dev(v), to_dev(q)
    ws = torch.zeros(svd.svd_kv_attention_workspace_bytes(Hq, Hkv, C), dtype=torch.uint8, device=DEV)
    o1 = torch.empty((C, Hq, D), dtype=torch.float32, device=DEV)
    o2 = torch.empty_like(o1)
    svd.svd_kv_append(kd, vd, ld, C, Hkv, n_past, c1, L)
    svd.svd_kv_attention(qd, c1, L, Hq, Hkv, n_past, C, 0.0884, o1, ws)
    svd.svd_kv_attention_append(qd, kd, vd, ld, c2, L, Hq, Hkv, n_past, C, 0.0884, o2, ws)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    scale = float(o1.abs().max())
    assert float((o1 - o2).abs().max()) <= 2.0 ** -16 * scale
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_full_size_262k_context_sampled_head():
    # The benchmark's longest context in its launch configuration (8 kv heads, 19 splits each):
    # the oracle checks kv head 3's five query heads at all four window rows.
    Hq, Hkv, C = synth.N_Q_HEADS, synth.N_KV_HEADS, 4
    L = 262144
    n_past = L - C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=262)
    q = synth.queries(C, Hq, D, seed=263)
    cache = _native(kc, ks, vc, vs, L)
    o = _attend(q, cache, L, Hq, Hkv, n_past)
    G, g = Hq // Hkv, 3
    sl = slice(g, g + 1)
    o_ref, a_ref = oracle.kv_attention(q[:, g * G:(g + 1) * G], kc[sl], ks[sl], vc[sl], vs[sl], n_past)
    _check(o[:, g * G:(g + 1) * G], o_ref, a_ref)


def test_full_size_fused_append_32k():
    # The pass's call at 32K: the window's keys and values quantised by the attention kernel
    # itself (shortened last split), 40 query heads over 8 kv heads; kv heads 0 and 7 against
    # the oracle over the oracle-quantised window.
    Hq, Hkv, C = synth.N_Q_HEADS, synth.N_KV_HEADS, 4
    L = 32768
    n_past = L - C
    kc, ks, vc, vs = synth.kv_cache(Hkv, L, D, seed=327)
    cache = _native(kc, ks, vc, vs, L, ranges=[(0, n_past)])
    ld = 7168
    g0 = np.random.default_rng(328)
    y = g0.normal(0, 4, (C, ld)).astype(np.float32)          # a q|k|v output row per position
    k, v = y[:, 5120:5120 + Hkv * D], y[:, 5120 + Hkv * D:5120 + 2 * Hkv * D]
    yd = to_dev(y)
    q = synth.queries(C, Hq, D, seed=329)
    out = torch.empty((C, Hq, D), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_kv_attention_workspace_bytes(Hq, Hkv, C), dtype=torch.uint8, device=DEV)
    base = yd.data_ptr()
    svd.svd_kv_attention_append(to_dev(q), base + 4 * 5120, base + 4 * (5120 + Hkv * D), ld, cache,
                                L, Hq, Hkv, n_past, C, 1.0 / np.sqrt(D), out, ws)
    torch.cuda.synchronize()
    o = out.cpu().numpy().astype(np.float64)
    qk, qks, qv, qvs = oracle.kv_quantize(np.ascontiguousarray(k).reshape(C * Hkv, D),
                                          np.ascontiguousarray(v).reshape(C * Hkv, D))
    for c in range(C):
        for h in range(Hkv):
            i = c * Hkv + h
            kc[h, n_past + c], ks[h, n_past + c] = qk[i], qks[i]
            vc[h, n_past + c], vs[h, n_past + c] = qv[i], qvs[i]
    G = Hq // Hkv
    for g in (0, 7):
        sl = slice(g, g + 1)
        o_ref, a_ref = oracle.kv_attention(q[:, g * G:(g + 1) * G], kc[sl], ks[sl], vc[sl], vs[sl],
                                           n_past)
        _check(o[:, g * G:(g + 1) * G], o_ref, a_ref)
