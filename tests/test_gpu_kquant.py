"""GPU parity of the verify GEMM on K-quant (Q4_K) super-block weights (SVD_LAYOUT_Q4K) against
the Q4_K oracle: max |delta| <= 1e-3 * sum |w x| per output, element by element on small and
ragged shapes for every C the kernel takes, and on sampled rows of full 27B-shaped matrices."""
import numpy as np
import pytest
import torch

from oracle import kquant
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, to_dev

pytestmark = pytest.mark.gpu


def run(blocks_dev, in_f, out_f, x, flags=0):
    C = x.shape[0]
    W = svd.QWeight(blocks_dev, None, in_f, out_f, svd.SVD_LAYOUT_Q4K)
    Y = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
    svd.svd_verify_linear(W, to_dev(x), C, Y, None, flags=flags)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


@pytest.mark.parametrize("out_f,in_f,C", [
    (37, 768, 1), (37, 768, 4), (64, 256, 8), (300, 5120, 3), (33, 2304, 5), (131, 4096, 2),
    (8, 2048, 6), (1, 256, 7),
])
def test_q4k_matches_oracle(out_f, in_f, C):
    lib()
    blocks = synth.q4k_blocks(out_f, in_f, seed=out_f + in_f + C)
    x = synth.activations(C, in_f, seed=C)
    y = run(to_dev(blocks), in_f, out_f, x, flags=svd.SVD_F_PDL if C % 2 else 0)
    y_ref, a_ref = kquant.verify_linear(blocks, in_f, x)
    assert_gemm_parity(y, y_ref, a_ref)


@pytest.mark.parametrize("out_f,in_f", [(7168, 5120), (5120, 17408)])
def test_q4k_full_size_sampled_rows(out_f, in_f):
    lib()
    C = 4
    b = synth.q4k_blocks_torch(out_f, in_f, seed=3, device=DEV)
    x = synth.activations(C, in_f, seed=4)
    y = run(b, in_f, out_f, x)
    rows = np.unique(np.r_[synth.rng(5).choice(out_f, 40, replace=False), 0, 31, 32, out_f - 1])
    host = b[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    y_ref, a_ref = kquant.verify_linear(host, in_f, x)
    assert_gemm_parity(y[:, rows], y_ref, a_ref)


def test_q4k_argument_errors():
    lib()
    b = to_dev(synth.q4k_blocks(16, 512, seed=1))
    X = to_dev(synth.activations(4, 512, seed=2))
    Y = torch.empty((9, 16), dtype=torch.float32, device=DEV)
    bad = [
        (svd.QWeight(b, b, 512, 16, svd.SVD_LAYOUT_Q4K), 4, svd.SVD_ERR_INVALID_ARG),   # scales given
        (svd.QWeight(b, None, 480, 16, svd.SVD_LAYOUT_Q4K), 4, svd.SVD_ERR_INVALID_ARG),  # in % 256
        (svd.QWeight(b, None, 512, 16, svd.SVD_LAYOUT_Q4K), 9, svd.SVD_ERR_UNSUPPORTED),  # C > 8
    ]
    for W, C, code in bad:
        with pytest.raises(svd.SvdError) as e:
            svd.svd_verify_linear(W, X, C, Y, None)
        assert e.value.code == code
    # chains take the native layout only
    W = svd.QWeight(b, None, 512, 16, svd.SVD_LAYOUT_Q4K)
    with pytest.raises(svd.SvdError) as e:
        svd.svd_verify_chain([(W, X, Y)], 4, torch.zeros(1 << 20, dtype=torch.uint8, device=DEV))
    assert e.value.code == svd.SVD_ERR_INVALID_ARG
