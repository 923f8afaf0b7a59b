"""A seeded sweep of random matrix shapes and window widths through every verify path, each
output compared with the oracle: the symmetric format on the warp-level kernel (C <= 16) and the
tcgen05 kernel (17..32), the Q4_K native layout on the stream kernel (C <= 16) and the Q4_K bytes
as stored (C <= 8).  Shapes are drawn ragged in both dimensions (rows not a multiple of 64,
inputs a multiple of 32 -- of 256 for Q4_K -- but not of 64), small enough for the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kquant
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, native_weight, to_dev

pytestmark = pytest.mark.gpu

_rng = np.random.default_rng(20261203)
SYM = [(int(_rng.integers(1, 700)), 32 * int(_rng.integers(1, 90)), int(_rng.integers(1, 33)))
       for _ in range(24)]
Q4K = [(int(_rng.integers(1, 700)), 256 * int(_rng.integers(1, 12)), int(_rng.integers(1, 17)))
       for _ in range(16)]


@pytest.mark.parametrize("out_f,in_f,C", SYM)
def test_symmetric_random_shapes(out_f, in_f, C):
    lib()
    codes, scales = synth.qweight(out_f, in_f, seed=out_f * 131 + in_f + C)
    x = synth.activations(C, in_f, seed=C + out_f)
    W, _ = native_weight(codes, scales)
    Y = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_linear(W, to_dev(x), C, Y, ws)
    torch.cuda.synchronize()
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)
    y_ref, a_ref = oracle.verify_linear(codes, scales, x)
    # tcgen05 above 16 columns: fp16 operands, held to 2^-10 of sum |w x| (the 1e-3 bound)
    assert_gemm_parity(Y.cpu().numpy(), y_ref, a_ref, tol=2.0 ** -10 if C > 16 else 1e-3)


@pytest.mark.parametrize("out_f,in_f,C", Q4K)
def test_q4k_random_shapes(out_f, in_f, C):
    lib()
    blocks = synth.q4k_blocks(out_f, in_f, seed=out_f * 17 + in_f + C)
    x = synth.activations(C, in_f, seed=C + 3 * out_f)
    y_ref, a_ref = kquant.verify_linear(blocks, in_f, x)
    bd = to_dev(blocks)
    cb, hb = svd.svd_q4k_native_sizes(in_f, out_f)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    hdr = torch.empty(hb, dtype=torch.uint8, device=DEV)
    svd.svd_repack_weights(svd.QWeight(bd, None, in_f, out_f, svd.SVD_LAYOUT_Q4K), codes, hdr)
    W = svd.QWeight(codes, hdr, in_f, out_f, svd.SVD_LAYOUT_Q4K_NATIVE)
    Y = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_linear(W, to_dev(x), C, Y, ws)
    torch.cuda.synchronize()
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)
    assert_gemm_parity(Y.cpu().numpy(), y_ref, a_ref)
    if C <= 8:  # the bytes as stored, on the CUDA-core kernel
        Y2 = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
        svd.svd_verify_linear(svd.QWeight(bd, None, in_f, out_f, svd.SVD_LAYOUT_Q4K), to_dev(x), C, Y2, None)
        torch.cuda.synchronize()
        assert_gemm_parity(Y2.cpu().numpy(), y_ref, a_ref)
