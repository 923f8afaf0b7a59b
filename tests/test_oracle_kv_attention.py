"""Pins of the KV-read attention oracle against things other than itself: closed forms of the
uniform-attention average (which fixes the causal extent of every window row, the grouped-query
head mapping and the value decode), the two-position softmax (the logistic of the score gap, which
fixes the softmax scale, the key decode and the key-scale block index), the nibble order of the
value codes, and the invariants of attention (permutation of context positions, causality,
linearity in the values)."""
import math

import numpy as np
import pytest

import oracle
from speculative_decoding_verify_06_gb300 import synth


def _f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _bf16(x):
    return synth.bf16_bits(np.asarray(x, dtype=np.float32))


def _cache(Hkv, ld, D, seed=0):
    kc, ks, vc, vs = synth.kv_cache(Hkv, ld, D, seed)
    return kc.copy(), ks.copy(), vc.copy(), vs.copy()


@pytest.mark.parametrize("n_past,C", [(0, 1), (0, 4), (37, 4), (16, 3), (5, 8)])
def test_uniform_attention_is_the_mean_of_visible_positions(n_past, C):
    # q = 0 makes every score 0, so each row averages the values it may see.  Value codes 9
    # (value = scale) and scale = position + 512 * kv head (exact in fp16) give the closed form
    # o[c][h] = 512 * (h // G) + (n_past + c) / 2 in every dimension.
    Hq, Hkv, D = 6, 3, 64
    ld = n_past + C + 5
    kc, ks, vc, vs = _cache(Hkv, ld, D)
    vc[:] = 0x99
    for g in range(Hkv):
        for j in range(ld):
            vs[g, j, :] = _f16(j + 512 * g)
    q = np.zeros((C, Hq, D), np.uint16)
    o, a = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    G = Hq // Hkv
    for c in range(C):
        for h in range(Hq):
            want = 512 * (h // G) + (n_past + c) / 2
            assert np.allclose(o[c, h], want, rtol=0, atol=1e-9), (c, h)
            assert np.allclose(a[c, h], want, rtol=0, atol=1e-9)


@pytest.mark.parametrize("D,i0", [(32, 7), (64, 40), (128, 127)])
@pytest.mark.parametrize("scale", [None, 0.3])
def test_two_positions_follow_the_logistic_of_the_score_gap(D, i0, scale):
    # One window position (C = 1) after one context position: two visible keys.  A one-hot query
    # on dimension i0 reads k_j[i0] = s_j * code_j only; the output is
    # v_1 + (v_0 - v_1) * sigmoid(scale * (k_0[i0] - k_1[i0])).
    Hq = Hkv = 1
    kc, ks, vc, vs = _cache(Hkv, 2, D, seed=3)
    kc[0, 0, i0], kc[0, 1, i0] = 10, -20
    ks[0, 0, i0 // 32], ks[0, 1, i0 // 32] = _f16(0.5), _f16(0.25)
    q = np.zeros((1, Hq, D), np.float32)
    q[0, 0, i0] = 1.0
    o, _ = oracle.kv_attention(_bf16(q), kc, ks, vc, vs, n_past=1, scale=scale)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    gap = sc * (10 * 0.5 - (-20) * 0.25)
    sig = 1.0 / (1.0 + math.exp(-gap))

    def v(j):
        out = np.empty(D)
        for d in range(D):
            byte = int(vc[0, j, d // 2])
            code = (byte >> 4) if d & 1 else (byte & 15)
            out[d] = float(np.uint16(vs[0, j, d // 32]).view(np.float16)) * (code - 8)
        return out

    want = v(1) + (v(0) - v(1)) * sig
    assert np.allclose(o[0, 0], want, rtol=1e-13, atol=1e-15)


def test_value_codes_low_nibble_is_the_even_dimension():
    # A single visible position (n_past = 0, C = 1) is returned as is: byte 0x3C holds code 12
    # (value 4 s) for even dimensions and code 3 (value -5 s) for odd ones, s the scale of the
    # dimension's 32-block (0.125 for dimensions 0..31, 0.25 for 32..63).
    D = 64
    kc, ks, vc, vs = _cache(1, 1, D)
    vc[:] = 0x3C
    vs[0, 0, :] = _f16([0.125, 0.25])
    q = synth.queries(1, 1, D, seed=1)
    o, a = oracle.kv_attention(q, kc, ks, vc, vs, n_past=0)
    s = np.repeat([0.125, 0.25], 32)
    want = np.where(np.arange(D) % 2 == 0, 4.0, -5.0) * s
    assert np.array_equal(o[0, 0], want)
    assert np.array_equal(a[0, 0], np.abs(want))


def test_key_codes_are_signed_bytes():
    # Code -128 must read as -128 (not 128): with scale 1 and a query of 1 on that dimension the
    # two keys -128 and +127 score -128/sqrt(D) and 127/sqrt(D).
    D = 32
    kc, ks, vc, vs = _cache(1, 2, D)
    kc[0, :, :] = 0
    kc[0, 0, 5], kc[0, 1, 5] = -128, 127
    ks[:] = _f16(1.0)
    vc[:] = 0x88
    vc[0, 0, :] = 0x99   # position 0: value +1 everywhere; position 1: value 0
    vs[:] = _f16(1.0)
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 5] = 1.0
    o, _ = oracle.kv_attention(_bf16(q), kc, ks, vc, vs, n_past=1)
    w0 = 1.0 / (1.0 + math.exp((127 + 128) / math.sqrt(D)))
    assert np.allclose(o[0, 0], w0, rtol=1e-12, atol=0)


def test_context_positions_are_a_set():
    # Attention over positions 0 .. n_past-1 is invariant under any permutation of them (keys,
    # values and scales moved together); the window's own positions stay in place.
    Hq, Hkv, D, n_past, C = 4, 2, 64, 23, 3
    kc, ks, vc, vs = _cache(Hkv, n_past + C, D, seed=7)
    q = synth.queries(C, Hq, D, seed=8)
    o, _ = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    perm = np.concatenate([np.random.default_rng(1).permutation(n_past), np.arange(n_past, n_past + C)])
    o2, _ = oracle.kv_attention(q, kc[:, perm], ks[:, perm], vc[:, perm], vs[:, perm], n_past)
    assert np.allclose(o, o2, rtol=0, atol=1e-14)


def test_window_rows_are_causal():
    # Row c may not see positions after n_past + c: changing positions n_past + 2 onwards leaves
    # rows 0 and 1 unchanged and does change the last row.
    Hq, Hkv, D, n_past, C = 2, 1, 32, 10, 4
    kc, ks, vc, vs = _cache(Hkv, n_past + C, D, seed=11)
    q = synth.queries(C, Hq, D, seed=12)
    o, _ = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, n_past + 2:] = -kc2[:, n_past + 2:] // 2
    vc2[:, n_past + 2:] ^= 0x55
    o2, _ = oracle.kv_attention(q, kc2, ks, vc2, vs, n_past)
    assert np.array_equal(o[:2], o2[:2])
    assert not np.allclose(o[C - 1], o2[C - 1])


def test_output_is_linear_in_the_value_scales():
    Hq, Hkv, D, n_past, C = 4, 1, 64, 9, 2
    kc, ks, vc, vs = _cache(Hkv, n_past + C, D, seed=5)
    q = synth.queries(C, Hq, D, seed=6)
    o, a = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    vs2 = _f16(2.0 * vs.view(np.float16).astype(np.float64))
    o2, a2 = oracle.kv_attention(q, kc, ks, vc, vs2, n_past)
    assert np.allclose(o2, 2 * o, rtol=1e-14, atol=0)
    assert np.all(a >= np.abs(o) - 1e-15)


def test_single_query_head_per_kv_head_matches_grouped_layout():
    # With G = Hq / Hkv query heads per kv head, head h reads kv head h // G: a cache holding one
    # kv head per query head (each repeated G times) gives the same output.
    Hq, Hkv, D, n_past, C = 6, 2, 32, 12, 2
    kc, ks, vc, vs = _cache(Hkv, n_past + C, D, seed=21)
    q = synth.queries(C, Hq, D, seed=22)
    o, _ = oracle.kv_attention(q, kc, ks, vc, vs, n_past)
    rep = np.repeat(np.arange(Hkv), Hq // Hkv)
    o2, _ = oracle.kv_attention(q, kc[rep], ks[rep], vc[rep], vs[rep], n_past)
    assert np.array_equal(o, o2)
