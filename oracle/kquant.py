"""Oracle for the K-quant 4-bit super-block format (Q4_K), in fp64 numpy.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see the package docstring): only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it.

"100 tokens per second from a 27B model on a 24 GB AMD card", section "The wall", and "Decode is
memory-bound ...", section "The ceiling", run 27B checkpoints in UD-Q4_K_XL and Q4_K_M, mixes
whose 4-bit tensors are Q4_K super-blocks; the pages do not give the layout, so this module
follows the format's public specification (the llama.cpp/ggml quantisation types):

* a super-block holds 256 consecutive weights of one row in 144 bytes: fp16 ``d``, fp16
  ``dmin``, 12 bytes of packed 6-bit sub-block scales ``sc[j]`` and mins ``m[j]`` (j = 0..7, one
  pair per 32 weights), then 128 bytes of 4-bit codes ``q``;
* weight ``i`` of sub-block ``j`` is ``d * sc[j] * q - dmin * m[j]``;
* scale packing: for j < 4, ``sc[j]`` and ``m[j]`` are the low 6 bits of bytes j and j + 4; for
  j >= 4 their low 4 bits are the low and high nibbles of byte j + 4 and their high 2 bits are
  the top 2 bits of bytes j - 4 (for ``sc``) and j (for ``m``);
* code packing: the 256 codes form four groups of 64; byte ``32 g + l`` of the code area holds
  weight ``64 g + l`` in its low nibble and weight ``64 g + 32 + l`` in its high nibble.

Each function below states the step it implements; pins are in ``tests/test_oracle_kquant.py``.
"""
from __future__ import annotations

import numpy as np

QK_K = 256            # weights per super-block
BLOCK_BYTES = 144     # bytes per super-block
SUB = 32              # weights per sub-block


def unpack_scales(scales12: np.ndarray):
    """(sc, m): uint8 arrays [..., 8] from the 12 packed scale bytes [..., 12]."""
    s = np.asarray(scales12, dtype=np.uint8).astype(np.int64)
    sc = np.empty(s.shape[:-1] + (8,), np.int64)
    m = np.empty_like(sc)
    for j in range(8):
        if j < 4:
            sc[..., j] = s[..., j] & 63
            m[..., j] = s[..., j + 4] & 63
        else:
            sc[..., j] = (s[..., j + 4] & 15) | ((s[..., j - 4] >> 6) << 4)
            m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    return sc, m


def unpack_codes(qs128: np.ndarray) -> np.ndarray:
    """The 256 codes of each super-block, in weight order, from its 128 code bytes."""
    b = np.asarray(qs128, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (QK_K,), np.int64)
    for g in range(4):
        chunk = b[..., 32 * g:32 * g + 32].astype(np.int64)
        out[..., 64 * g:64 * g + 32] = chunk & 15
        out[..., 64 * g + 32:64 * g + 64] = chunk >> 4
    return out


def split_blocks(blocks: np.ndarray, in_f: int):
    """A row-major Q4_K matrix (uint8 [out][in / 256 * 144]) as its fields: d, dmin (fp64
    [out][nsb]), scale bytes [out][nsb][12], code bytes [out][nsb][128]."""
    out_f = blocks.shape[0]
    nsb = in_f // QK_K
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(out_f, nsb, BLOCK_BYTES)
    d = b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = b[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    return d, dmin, b[..., 4:16], b[..., 16:144]


def dequant(blocks: np.ndarray, in_f: int) -> np.ndarray:
    """fp64 weights [out][in]: d * sc[j] * q - dmin * m[j] for every weight."""
    if in_f % QK_K:
        raise ValueError("in_features must be a multiple of 256")
    d, dmin, scb, qsb = split_blocks(blocks, in_f)
    sc, m = unpack_scales(scb)                      # [out][nsb][8]
    q = unpack_codes(qsb).astype(np.float64)        # [out][nsb][256]
    a = (d[..., None] * sc)[..., :, None]           # [out][nsb][8][1]
    b = (dmin[..., None] * m)[..., :, None]
    w = a * q.reshape(q.shape[:-1] + (8, SUB)) - b  # [out][nsb][8][32]
    return w.reshape(blocks.shape[0], in_f)


def verify_linear(blocks: np.ndarray, in_f: int, x_bf16: np.ndarray):
    """(Y, A): Y[c][j] = sum_i w[j][i] x[c][i] in fp64 and A[c][j] = sum_i |w[j][i] x[c][i]| (the
    tolerance scale), for bf16 activations given as uint16 bit patterns [C][in]."""
    x = (np.asarray(x_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = dequant(blocks, in_f)
    return x @ w.T, np.abs(x) @ np.abs(w).T
