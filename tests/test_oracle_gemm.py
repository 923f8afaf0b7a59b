"""Pins of the oracle's number formats and dequant GEMM against things other than itself:
numpy/torch format conversions, a dense numpy matmul written independently, exact rational
arithmetic and closed-form special cases."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import synth


def test_f16_decode_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_bf16_decode_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def _dense_reference(codes, scales, x_bf16):
    """Independent dequantise-to-dense then numpy matmul in float64."""
    out_f, half = codes.shape
    lo = (codes & 0x0F).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    q = np.empty((out_f, 2 * half), np.int64)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    s = scales.view(np.float16).astype(np.float64)
    w = (q - 8).astype(np.float64) * np.repeat(s, 32, axis=1)
    x = torch.from_numpy(x_bf16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return x @ w.T, np.abs(x)[:, None, :] * np.abs(w)[None, :, :]


@pytest.mark.parametrize("out_f,in_f,C", [(1, 32, 1), (3, 64, 4), (17, 96, 3), (64, 64, 8),
                                          (40, 160, 5), (33, 32, 2)])
def test_gemm_brute_force_tiny(out_f, in_f, C):
    codes, scales = synth.qweight(out_f, in_f, seed=out_f * 1000 + in_f)
    x = synth.activations(C, in_f, seed=C + 7)
    y, a = oracle.verify_linear(codes, scales, x, nthreads=2)
    ref, absterms = _dense_reference(codes, scales, x)
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * np.abs(absterms).sum(-1).max())
    assert np.allclose(a, absterms.sum(-1), rtol=1e-13)


def test_gemm_all_codes_eight_is_exactly_zero():
    out_f, in_f, C = 20, 128, 4
    codes = np.full((out_f, in_f // 2), 0x88, np.uint8)
    _, scales = synth.qweight(out_f, in_f, seed=1)
    x = synth.activations(C, in_f, seed=2)
    y, a = oracle.verify_linear(codes, scales, x)
    assert np.all(y == 0.0) and np.all(a == 0.0)


@pytest.mark.parametrize("j,i", [(0, 0), (0, 1), (5, 31), (5, 32), (9, 63), (13, 94), (13, 95)])
def test_gemm_single_code_selects_one_input(j, i):
    """code 9 (value +1) at (j, i) with scale 1 on its block: y[c][j] = x[c][i], others 0.
    Pins the nibble order (even input in the low nibble) and the block indexing."""
    out_f, in_f, C = 16, 96, 3
    codes = np.full((out_f, in_f // 2), 0x88, np.uint8)
    b = codes[j, i // 2]
    codes[j, i // 2] = (b & 0xF0) | 9 if i % 2 == 0 else (b & 0x0F) | (9 << 4)
    scales = np.zeros((out_f, in_f // 32), np.uint16)
    scales[j, i // 32] = synth.f16_bits(1.0)
    x = synth.activations(C, in_f, seed=3)
    y, _ = oracle.verify_linear(codes, scales, x)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    expect = np.zeros((C, out_f))
    expect[:, j] = xv[:, i]
    assert np.array_equal(y, expect)


def test_gemm_power_of_two_scales_is_exact():
    """With scales 2^-e and bf16 inputs every product and every partial sum of a short row is
    exactly representable; compare with exact rational arithmetic."""
    out_f, in_f, C = 6, 64, 2
    g = synth.rng(11)
    codes = g.integers(0, 256, size=(out_f, in_f // 2), dtype=np.uint8)
    exps = g.integers(4, 9, size=(out_f, in_f // 32))
    scales = synth.f16_bits(np.ldexp(1.0, -exps))
    xf = np.ldexp(g.integers(-64, 64, size=(C, in_f)).astype(np.float64), -3)
    x = synth.bf16_bits(xf.astype(np.float32))
    y, _ = oracle.verify_linear(codes, scales, x)
    for c in range(C):
        for jj in range(out_f):
            acc = Fraction(0)
            for ii in range(in_f):
                byte = int(codes[jj, ii // 2])
                code = (byte >> 4) if ii % 2 else (byte & 15)
                acc += Fraction(2) ** (-int(exps[jj, ii // 32])) * (code - 8) * Fraction(xf[c, ii])
            assert y[c, jj] == float(acc)
