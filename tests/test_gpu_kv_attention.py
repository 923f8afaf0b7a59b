"""GPU parity of the KV-read attention (svd_kv_attention over a native cache written by
svd_kv_repack) against the fp64 oracle, element by element.

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
    for p0, p1 in (ranges or [(0, ld)]):
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
