"""Pins of the K-quant (Q4_K) oracle: scale and code unpacking against hand-worked bytes, the
dequantisation against the symmetric format's oracle through an exact special case, closed
forms, and the product against a brute-force loop."""
import numpy as np

import oracle
from oracle import kquant
from speculative_decoding_verify_06_gb300 import synth

F16 = np.float16


def _block(d, dmin, scales12, qs128):
    b = np.zeros(kquant.BLOCK_BYTES, np.uint8)
    b[0:2] = np.array([d], F16).view(np.uint8)
    b[2:4] = np.array([dmin], F16).view(np.uint8)
    b[4:16] = scales12
    b[16:144] = qs128
    return b


def test_scale_unpacking_hand_worked():
    # bytes s0..s11; by the layout: j < 4: sc = s[j] & 63, m = s[j+4] & 63; j >= 4: sc = (s[j+4]
    # & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4.  Worked by hand:
    # j=4: sc = 0xA | 1<<4 = 26, m = 0x9 | 0<<4 = 9;   j=5: sc = 0xC | 2<<4 = 44, m = 0xB | 1<<4 = 27
    # j=6: sc = 0xE | 0<<4 = 14, m = 0xD | 2<<4 = 45;  j=7: sc = 0x1 | 3<<4 = 49, m = 0xF | 3<<4 = 63
    s = np.array([0x41, 0x82, 0x03, 0xC4, 0x05, 0x46, 0x87, 0xC8, 0x9A, 0xBC, 0xDE, 0xF1], np.uint8)
    sc, m = kquant.unpack_scales(s)
    assert sc.tolist() == [1, 2, 3, 4, 26, 44, 14, 49]
    assert m.tolist() == [5, 6, 7, 8, 9, 27, 45, 63]


def test_code_unpacking_hand_placed():
    qs = np.zeros(128, np.uint8)
    qs[0] = 0x21     # weight 0 <- 1, weight 32 <- 2
    qs[31] = 0x65    # weight 31 <- 5, weight 63 <- 6
    qs[32] = 0x43    # weight 64 <- 3, weight 96 <- 4
    qs[127] = 0xF7   # weight 223 <- 7, weight 255 <- 15
    q = kquant.unpack_codes(qs)
    expect = np.zeros(256, np.int64)
    expect[[0, 32, 31, 63, 64, 96, 223, 255]] = [1, 2, 5, 6, 3, 4, 7, 15]
    assert np.array_equal(q, expect)


def test_closed_forms():
    g = np.random.default_rng(1)
    qs = g.integers(0, 256, 128, dtype=np.uint8)
    q = kquant.unpack_codes(qs)
    # d = 1, dmin = 0, every sc = 1 (bytes 0..3 = 1, bytes 8..11 low nibbles 1): the codes
    s = np.array([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], np.uint8)
    w = kquant.dequant(_block(1.0, 0.0, s, qs)[None, :], 256)[0]
    assert np.array_equal(w, q.astype(np.float64))
    # d = 0: every weight of sub-block j is -dmin * m[j], whatever the codes
    s2 = np.array([0, 0, 0, 0, 3, 5, 7, 9, 0x20, 0x40, 0x60, 0x80], np.uint8)
    _, m = kquant.unpack_scales(s2)
    w = kquant.dequant(_block(0.0, 0.5, s2, qs)[None, :], 256)[0]
    assert np.array_equal(w, np.repeat(-0.5 * m.astype(np.float64), 32))


def _pack_symmetric_case(out_f, in_f, seed):
    """A Q4_K matrix with m[j] = sc[j] and dmin = 8 d, so that every weight is d sc[j] (q - 8):
    the symmetric 4.5-bit format with scale d sc[j] per 32 inputs (exact in fp16 for d = 2^-10,
    sc < 64).  Returns (Q4_K bytes, canonical codes [out][in/2], fp16 scale bits [out][in/32])."""
    g = np.random.default_rng(seed)
    nsb = in_f // 256
    d = 2.0 ** -10
    sc = g.integers(1, 64, size=(out_f, nsb, 8))
    q = g.integers(0, 16, size=(out_f, nsb, 256))
    blocks = np.zeros((out_f, nsb, 144), np.uint8)
    blocks[..., 0:2] = np.array([d], F16).view(np.uint8)
    blocks[..., 2:4] = np.array([8 * d], F16).view(np.uint8)
    s = np.zeros((out_f, nsb, 12), np.int64)
    for j in range(8):  # the packing of the layout, written field by field
        if j < 4:
            s[..., j] |= sc[..., j] & 63
            s[..., j + 4] |= sc[..., j] & 63          # m[j] = sc[j]
        else:
            s[..., j + 4] |= (sc[..., j] & 15) | ((sc[..., j] & 15) << 4)
            s[..., j - 4] |= (sc[..., j] >> 4) << 6
            s[..., j] |= (sc[..., j] >> 4) << 6
    blocks[..., 4:16] = s.astype(np.uint8)
    for gq in range(4):
        lo = q[..., 64 * gq:64 * gq + 32]
        hi = q[..., 64 * gq + 32:64 * gq + 64]
        blocks[..., 16 + 32 * gq:16 + 32 * gq + 32] = (lo | (hi << 4)).astype(np.uint8)
    # the same weights in the canonical symmetric layout
    qq = q.reshape(out_f, in_f)
    codes = (qq[:, 0::2] | (qq[:, 1::2] << 4)).astype(np.uint8)
    scales = np.array(d * sc.reshape(out_f, nsb * 8), F16).view(np.uint16)
    return blocks.reshape(out_f, nsb * 144), codes, scales


def test_symmetric_special_case_equals_the_symmetric_oracle():
    out_f, in_f, C = 37, 768, 3
    blocks, codes, scales = _pack_symmetric_case(out_f, in_f, seed=4)
    x = synth.activations(C, in_f, seed=5)
    y_k, a_k = kquant.verify_linear(blocks, in_f, x)
    y_s, a_s = oracle.verify_linear(codes, scales, x)
    assert np.allclose(y_k, y_s, rtol=1e-12, atol=1e-12)
    assert np.allclose(a_k, a_s, rtol=1e-12, atol=1e-12)


def test_product_brute_force():
    g = np.random.default_rng(9)
    blocks = g.integers(0, 256, size=(2, 2 * 144), dtype=np.uint8)
    for r in range(2):
        for sb in range(2):  # finite d, dmin
            blocks[r, sb * 144:sb * 144 + 4] = np.array([0.03, 0.01], F16).view(np.uint8)
    x = synth.activations(2, 512, seed=3)
    y, a = kquant.verify_linear(blocks, 512, x)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for r in range(2):
        for c in range(2):
            acc = absacc = 0.0
            for sb in range(2):
                blk = blocks[r, sb * 144:(sb + 1) * 144]
                d = float(blk[0:2].view(F16)[0])
                dmin = float(blk[2:4].view(F16)[0])
                sc, m = kquant.unpack_scales(blk[4:16])
                q = kquant.unpack_codes(blk[16:144])
                for i in range(256):
                    w = d * sc[i // 32] * q[i] - dmin * m[i // 32]
                    acc += w * xf[c, 256 * sb + i]
                    absacc += abs(w * xf[c, 256 * sb + i])
            assert abs(acc - y[c, r]) <= 1e-12 * absacc
            assert abs(absacc - a[c, r]) <= 1e-12 * absacc
