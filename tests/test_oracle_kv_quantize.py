"""Pins of the oracle's cache quantiser (q8_0 keys, q4_0 values) and of its fp32 -> fp16 rounding
against things other than itself: numpy's float16 conversion, and the properties the block
definitions fix -- code ranges, the extreme element's code, signs and order, the reconstruction
bound, the zero block and the tie rule for the value block's extreme."""
import numpy as np
import pytest

import oracle


def test_f32_to_f16_matches_numpy():
    g = np.random.default_rng(0)
    vals = np.concatenate([
        g.normal(0, 1, 20000), g.normal(0, 1e-5, 5000), g.normal(0, 3e4, 5000),
        np.ldexp(1.0, np.arange(-30, 17)), [0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e6, -1e6,
                                             2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 6.1e-5],
    ]).astype(np.float32)
    # halfway cases between neighbouring fp16 values, both parities
    h = np.arange(0x0400, 0x7bff, 97, dtype=np.uint16).view(np.float16).astype(np.float32)
    h2 = np.nextafter(h.astype(np.float16), np.float16(np.inf)).astype(np.float32)
    vals = np.concatenate([vals, (h + h2) / 2, -(h + h2) / 2]).astype(np.float32)
    got = np.array([oracle.f32_to_f16_bits(float(x)) for x in vals], dtype=np.uint16)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def _f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _blocks(seed, rows=64, D=128):
    g = np.random.default_rng(seed)
    k = (g.normal(0, 1, (rows, D)) * g.uniform(0.01, 50, (rows, 1))).astype(np.float32)
    v = (g.normal(0, 1, (rows, D)) * g.uniform(0.01, 50, (rows, 1))).astype(np.float32)
    return k, v


def _v_codes(vc):
    out = np.empty((vc.shape[0], 2 * vc.shape[1]), np.int64)
    out[:, 0::2] = vc & 15
    out[:, 1::2] = vc >> 4
    return out


def test_key_blocks_q8_0_properties():
    k, v = _blocks(1)
    kc, ks, _, _ = oracle.kv_quantize(k, v)
    rows, D = k.shape
    kb = k.reshape(rows, D // 32, 32).astype(np.float64)
    qb = kc.reshape(rows, D // 32, 32).astype(np.int64)
    amax = np.abs(kb).max(axis=2)
    d32 = amax / 127.0
    # the block's extreme element gets code +-127, with its sign; every code within range
    idx = np.abs(kb).argmax(axis=2)
    ext = np.take_along_axis(qb, idx[..., None], axis=2)[..., 0]
    assert np.array_equal(np.abs(ext), np.full_like(ext, 127))
    assert np.all(np.sign(qb) * np.sign(kb) >= 0) and np.abs(qb).max() <= 127
    # monotone within a block, and rounding to the nearest code of step d
    for r in range(rows):
        for b in range(D // 32):
            o = np.argsort(kb[r, b], kind="stable")
            assert np.all(np.diff(qb[r, b][o]) >= 0)
    assert np.all(np.abs(kb - d32[..., None] * qb) <= d32[..., None] * (0.5 + 1e-5))
    # the stored scale is the fp32 d = max|x| / 127 rounded to fp16 (numpy's conversion)
    d_f32 = np.abs(k.reshape(rows, D // 32, 32)).max(axis=2) / np.float32(127.0)
    assert np.array_equal(ks, d_f32.astype(np.float32).astype(np.float16).view(np.uint16))


def test_value_blocks_q4_0_properties():
    k, v = _blocks(2)
    _, _, vc, vs = oracle.kv_quantize(k, v)
    rows, D = v.shape
    vb = v.reshape(rows, D // 32, 32).astype(np.float64)
    cb = _v_codes(vc).reshape(rows, D // 32, 32)
    assert cb.min() >= 0 and cb.max() <= 15
    idx = np.abs(vb).argmax(axis=2)
    m = np.take_along_axis(vb, idx[..., None], axis=2)[..., 0]
    d = m / -8.0
    # the extreme value maps to code 0, i.e. to d * (0 - 8) = m
    assert np.all(np.take_along_axis(cb, idx[..., None], axis=2)[..., 0] == 0)
    # reconstruction: within |d| / 2 except where the top code clamps (within |d| there)
    err = np.abs(vb - d[..., None] * (cb - 8))
    assert np.all(err <= np.abs(d)[..., None] * (1.0 + 1e-5))
    unclamped = cb < 15
    assert np.all(err[unclamped] <= (np.abs(d)[..., None] * (0.5 + 1e-5) * np.ones_like(err))[unclamped])
    # codes decrease as values increase when the extreme is positive (d < 0), and vice versa
    for r in range(rows):
        for b in range(D // 32):
            o = np.argsort(vb[r, b], kind="stable")
            step = np.diff(cb[r, b][o])
            assert np.all(step <= 0) if d[r, b] < 0 else np.all(step >= 0)
    m32 = np.take_along_axis(v.reshape(rows, D // 32, 32), idx[..., None], axis=2)[..., 0]
    assert np.array_equal(vs, (m32 / np.float32(-8.0)).astype(np.float32).astype(np.float16).view(np.uint16))


def test_zero_block_and_tie_rule():
    D = 32
    k = np.zeros((2, D), np.float32)
    v = np.zeros((2, D), np.float32)
    v[1, 3], v[1, 7] = -2.0, 2.0          # two values of the largest magnitude: the first wins
    v[1, 10] = 1.0
    kc, ks, vc, vs = oracle.kv_quantize(k, v)
    assert np.all(kc == 0) and np.all(ks == 0)
    codes = _v_codes(vc)
    assert np.all(codes[0] == 8) and _f16(vs[0, 0]) == 0.0   # d = 0 / -8 (a signed zero)
    # m = -2 -> d = 0.25: -2 -> code 0, +2 -> trunc(8 + 8.5) clamped to 15, 1 -> 12, 0 -> 8
    assert _f16(vs[1, 0]) == 0.25
    assert codes[1, 3] == 0 and codes[1, 7] == 15 and codes[1, 10] == 12 and codes[1, 0] == 8


@pytest.mark.parametrize("x,code", [(0.49, 0), (0.5, 1), (-0.5, -1), (1.5, 2), (-2.5, -3)])
def test_key_rounding_is_half_away_from_zero(x, code):
    # One block whose extreme is 127 (d = 1, 1/d = 1 exactly): codes are round-half-away(x).
    k = np.zeros((1, 32), np.float32)
    k[0, 0] = 127.0
    k[0, 5] = x
    kc, ks, _, _ = oracle.kv_quantize(k, np.zeros_like(k))
    assert kc[0, 5] == code and kc[0, 0] == 127 and _f16(ks[0, 0]) == 1.0
