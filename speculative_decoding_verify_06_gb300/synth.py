"""Seeded synthetic inputs shared by the CUDA path, the oracle and the benchmark.

Only random draws and number-format conversions live here -- none of the verify pass's
arithmetic -- so both sides of every parity test can take their inputs from this module.
Recipes (the pages measure real models on real prompts, which are not available; these stand in
for them):

* 4-bit weights: codes uniform on 0..15 (a uniform byte holds two uniform nibbles), fp16 scales
  drawn U(0.005, 0.02) and rounded to nearest fp16, one per 32 inputs of a row.
* activations: N(0, 1) rounded to nearest-even bfloat16, [C][in] token-major.
* window logits: N(0, std^2) fp32; a drafter that "shares" a fraction f of the target's logit
  variance draws l_q = sqrt(f) l_p + sqrt(1 - f) l', l' independent N(0, std^2).
* Zipf-ranked logits: l(v) = -s ln(rank(v)) under a uniformly random ranking.
* KV cache (keys q8_0-style, values q4_0-style): key codes uniform on -128..127 with fp16 scales
  U(0.01, 0.04) per 32 dimensions (scores of N(0, 1) queries then spread with a standard
  deviation near 2 after the 1/sqrt(128) scale); value codes uniform on 0..15 with the weights'
  scale recipe; queries N(0, 1) bfloat16, [C][Hq][128].
"""
from __future__ import annotations

import numpy as np

# The 27B-shaped dense stack: 64 layers, hidden 5120, FFN 17408; per layer the fused q|k|v
# projection (5120 -> 5120 + 1024 + 1024), o (5120 -> 5120), fused gate|up (5120 -> 2 x 17408)
# and down (17408 -> 5120); the lm_head 5120 -> 151936.
LAYERS = 64
HIDDEN = 5120
FFN = 17408
VOCAB = 151936
LAYER_GEMMS = ((HIDDEN, HIDDEN + 1024 + 1024), (HIDDEN, HIDDEN), (HIDDEN, 2 * FFN), (FFN, HIDDEN))
LAYER_GEMM_NAMES = ("qkv", "o", "gate_up", "down")

SCALE_LO, SCALE_HI = 0.005, 0.02

# Attention geometry of the same stack: the fused q|k|v output (5120 + 1024 + 1024) read as 40
# query heads and 8 kv heads of dimension 128.
N_Q_HEADS, N_KV_HEADS, HEAD_DIM = 40, 8, 128
K_SCALE_LO, K_SCALE_HI = 0.01, 0.04


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(x) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def f16_bits(x) -> np.ndarray:
    """fp32/fp64 -> IEEE binary16 bit patterns (numpy rounds to nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def qweight(out_f: int, in_f: int, seed: int):
    """Canonical 4-bit matrix: (codes uint8 [out, in/2], scales uint16 fp16 bits [out, in/32])."""
    assert in_f % 32 == 0
    g = rng(seed)
    codes = g.integers(0, 256, size=(out_f, in_f // 2), dtype=np.uint8)
    scales = f16_bits(g.uniform(SCALE_LO, SCALE_HI, size=(out_f, in_f // 32)))
    return codes, scales


def activations(C: int, in_f: int, seed: int, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns [C, in] drawn N(0, std^2)."""
    return bf16_bits(rng(seed).normal(0.0, std, size=(C, in_f)).astype(np.float32))


def qweight_torch(out_f: int, in_f: int, seed: int, device):
    """The same recipe drawn on a device with torch's generator (for shapes too large to draw
    on the host); returns (codes uint8, scales int16 holding fp16 bits)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    codes = torch.randint(0, 256, (out_f, in_f // 2), dtype=torch.uint8, device=device, generator=g)
    s = torch.empty((out_f, in_f // 32), dtype=torch.float32, device=device)
    s.uniform_(SCALE_LO, SCALE_HI, generator=g)
    return codes, s.to(torch.float16).view(torch.int16)


# Q4_K super-block fields: d and dmin drawn U(Q4K_D_LO, Q4K_D_HI) and rounded to fp16 (6-bit
# sub-block scales up to 63 then give per-weight steps up to ~0.13, like the symmetric recipe's
# 8 x 0.02); scale and code bytes uniform.
Q4K_D_LO, Q4K_D_HI = 5e-4, 2e-3


def q4k_blocks(out_f: int, in_f: int, seed: int) -> np.ndarray:
    """Q4_K matrix: uint8 [out, in / 256 * 144], super-blocks of (fp16 d, fp16 dmin, 12 scale
    bytes, 128 code bytes) with uniform bytes and d, dmin from the recipe above."""
    assert in_f % 256 == 0
    g = rng(seed)
    nsb = in_f // 256
    b = g.integers(0, 256, size=(out_f, nsb, 144), dtype=np.uint8)
    dd = f16_bits(g.uniform(Q4K_D_LO, Q4K_D_HI, size=(out_f, nsb, 2)))
    b[..., 0:4] = dd.view(np.uint8).reshape(out_f, nsb, 4)
    return b.reshape(out_f, nsb * 144)


def q4k_blocks_torch(out_f: int, in_f: int, seed: int, device):
    """The same recipe drawn on a device with torch's generator."""
    import torch
    assert in_f % 256 == 0
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    nsb = in_f // 256
    b = torch.randint(0, 256, (out_f, nsb, 144), dtype=torch.uint8, device=device, generator=g)
    dd = torch.empty((out_f, nsb, 2), dtype=torch.float32, device=device)
    dd.uniform_(Q4K_D_LO, Q4K_D_HI, generator=g)
    b[..., 0:4] = dd.to(torch.float16).view(torch.uint8).reshape(out_f, nsb, 4)
    return b.reshape(out_f, nsb * 144)


def activations_torch(C: int, in_f: int, seed: int, device, std: float = 1.0):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.empty((C, in_f), dtype=torch.float32, device=device)
    x.normal_(0.0, std, generator=g)
    return x.to(torch.bfloat16)


def normal_logits(rows: int, V: int, seed: int, std: float = 2.0) -> np.ndarray:
    return rng(seed).normal(0.0, std, size=(rows, V)).astype(np.float32)


def shared_logits(lp: np.ndarray, share: float, seed: int, std: float = 2.0) -> np.ndarray:
    """l_q = sqrt(share) l_p + sqrt(1 - share) l' with l' ~ N(0, std^2) independent."""
    lo = rng(seed).normal(0.0, std, size=lp.shape)
    return (np.sqrt(share) * lp.astype(np.float64) + np.sqrt(1.0 - share) * lo).astype(np.float32)


def zipf_logits(V: int, seed: int, s: float = 1.1) -> np.ndarray:
    """l(v) = -s ln(rank(v)), ranks 1..V assigned by a uniformly random permutation."""
    rank = rng(seed).permutation(V) + 1
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


def perturb(l: np.ndarray, sigma: float, seed: int) -> np.ndarray:
    """l + N(0, sigma^2) noise (the drafter of a window in the lm_head workload)."""
    return (l.astype(np.float64) + rng(seed).normal(0.0, sigma, size=l.shape)).astype(np.float32)


def draw_from(probs: np.ndarray, seed: int) -> np.ndarray:
    """One categorical draw per row (the harness's drafter sampling; inverse CDF on numpy's
    generator)."""
    probs = np.asarray(probs, dtype=np.float64)
    u = rng(seed).random(probs.shape[0])
    cdf = np.cumsum(probs, axis=1)
    cdf /= cdf[:, -1:]
    idx = (cdf <= u[:, None]).sum(axis=1)
    return np.minimum(idx, probs.shape[1] - 1).astype(np.int32)


def kv_cache(Hkv: int, ld: int, D: int, seed: int):
    """Canonical cache of ld positions: (k_codes int8 [Hkv, ld, D], k_scales fp16 bits
    [Hkv, ld, D/32], v_codes uint8 [Hkv, ld, D/2] (low nibble = even dimension), v_scales fp16
    bits [Hkv, ld, D/32])."""
    assert D % 32 == 0
    g = rng(seed)
    kc = g.integers(-128, 128, size=(Hkv, ld, D), dtype=np.int8)
    ks = f16_bits(g.uniform(K_SCALE_LO, K_SCALE_HI, size=(Hkv, ld, D // 32)))
    vc = g.integers(0, 256, size=(Hkv, ld, D // 2), dtype=np.uint8)
    vs = f16_bits(g.uniform(SCALE_LO, SCALE_HI, size=(Hkv, ld, D // 32)))
    return kc, ks, vc, vs


def queries(C: int, Hq: int, D: int, seed: int, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns [C, Hq, D] drawn N(0, std^2)."""
    return bf16_bits(rng(seed).normal(0.0, std, size=(C, Hq, D)).astype(np.float32))


def kv_cache_torch(Hkv: int, ld: int, D: int, seed: int, device):
    """The kv_cache recipe drawn on a device with torch's generator (for long contexts); returns
    (k_codes int8, k_scales int16, v_codes uint8, v_scales int16), scales holding fp16 bits."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    kc = torch.randint(-128, 128, (Hkv, ld, D), dtype=torch.int8, device=device, generator=g)
    ks = torch.empty((Hkv, ld, D // 32), dtype=torch.float32, device=device)
    ks.uniform_(K_SCALE_LO, K_SCALE_HI, generator=g)
    vc = torch.randint(0, 256, (Hkv, ld, D // 2), dtype=torch.uint8, device=device, generator=g)
    vs = torch.empty((Hkv, ld, D // 32), dtype=torch.float32, device=device)
    vs.uniform_(SCALE_LO, SCALE_HI, generator=g)
    return kc, ks.to(torch.float16).view(torch.int16), vc, vs.to(torch.float16).view(torch.int16)
