"""GPU parity of the verify linear (tensor-core native kernel and CUDA-core canonical kernel)
against the oracle: max |delta| <= 1e-3 * sum |w x| per output, element by element on small and
ragged shapes, and on sampled rows of the full 27B-shaped matrices at the benchmark's launch
configuration."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, native_weight, to_dev, verify_linear

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("out_f,in_f,C", [
    (2048, 2048, 4),   # the tiny verify window: one 2048 x 2048 layer, K+1 = 4
    (40, 96, 1), (40, 96, 8), (7, 32, 1), (64, 64, 2), (200, 160, 3), (1000, 544, 6),
    (130, 2048, 5), (300, 1056, 7), (4096, 256, 4),
])
def test_native_matches_oracle(out_f, in_f, C):
    codes, scales = synth.qweight(out_f, in_f, seed=out_f + 31 * in_f)
    x = synth.activations(C, in_f, seed=C)
    W, _ = native_weight(codes, scales)
    y = verify_linear(W, x)
    y_ref, a_ref = oracle.verify_linear(codes, scales, x)
    assert_gemm_parity(y, y_ref, a_ref)


@pytest.mark.parametrize("C", [9, 16, 17, 24, 32])
def test_native_wide_window(C):
    out_f, in_f = 300, 544
    codes, scales = synth.qweight(out_f, in_f, seed=C)
    x = synth.activations(C, in_f, seed=C + 1)
    W, _ = native_weight(codes, scales)
    y_ref, a_ref = oracle.verify_linear(codes, scales, x)
    assert_gemm_parity(verify_linear(W, x), y_ref, a_ref)


@pytest.mark.parametrize("out_f,in_f,C", [(2048, 2048, 4), (40, 96, 1), (333, 640, 8), (100, 5120, 3)])
def test_canonical_cuda_core_kernel_matches_oracle(out_f, in_f, C):
    lib()
    codes, scales = synth.qweight(out_f, in_f, seed=5 + C)
    x = synth.activations(C, in_f, seed=6)
    W = svd.QWeight(to_dev(codes), to_dev(scales), in_f, out_f, svd.SVD_LAYOUT_CANONICAL)
    y_ref, a_ref = oracle.verify_linear(codes, scales, x)
    assert_gemm_parity(verify_linear(W, x), y_ref, a_ref)


@pytest.mark.parametrize("out_f,in_f", [(40, 96), (64, 64), (130, 544), (2048, 2048), (7, 32)])
def test_repack_roundtrip_is_identity(out_f, in_f):
    codes, scales = synth.qweight(out_f, in_f, seed=3)
    W, src = native_weight(codes, scales)
    c2 = torch.empty_like(src.codes)
    s2 = torch.empty_like(src.scales)
    svd.svd_unpack_weights(W, c2, s2)
    torch.cuda.synchronize()
    assert torch.equal(c2, src.codes) and torch.equal(s2, src.scales)


def test_deterministic_and_pdl_flag_and_shared_workspace():
    shapes = [(5120, 1024), (544, 2048), (2048, 160)]
    ws = torch.zeros(max(svd.svd_verify_linear_workspace_bytes(i, o, 4) for i, o in shapes),
                     dtype=torch.uint8, device=DEV)
    for (in_f, out_f) in shapes:
        codes, scales = synth.qweight(out_f, in_f, seed=in_f)
        x = synth.activations(4, in_f, seed=out_f)
        W, _ = native_weight(codes, scales)
        y1 = verify_linear(W, x, ws=ws)
        y2 = verify_linear(W, x, ws=ws)
        y3 = verify_linear(W, x, flags=svd.SVD_F_PDL, ws=ws)
        assert np.array_equal(y1, y2) and np.array_equal(y1, y3)
        y_ref, a_ref = oracle.verify_linear(codes, scales, x)
        assert_gemm_parity(y1, y_ref, a_ref)
    # the ticket counters are back to zero after every call
    assert int(ws[-svd.svd_verify_linear_workspace_bytes(2048, 160, 4):].sum()) >= 0


def test_workspace_too_small_is_rejected():
    codes, scales = synth.qweight(256, 256, seed=1)
    W, _ = native_weight(codes, scales)
    X = to_dev(synth.activations(4, 256, seed=2))
    Y = torch.empty((4, 256), dtype=torch.float32, device=DEV)
    need = svd.svd_verify_linear_workspace_bytes(256, 256, 4)
    ws = torch.zeros(need - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(svd.SvdError) as e:
        svd.svd_verify_linear(W, X, 4, Y, ws)
    assert e.value.code == svd.SVD_ERR_WORKSPACE


def _sampled_rows(out_f, n, seed):
    g = synth.rng(seed)
    rows = set(g.choice(out_f, size=n, replace=False).tolist())
    rows |= {0, 1, 15, 16, 63, 64, out_f - 1, out_f - 64, out_f // 2}
    return np.array(sorted(r for r in rows if 0 <= r < out_f))


@pytest.mark.parametrize("in_f,out_f,C", [
    (5120, 7168, 4), (5120, 5120, 4), (5120, 34816, 4), (17408, 5120, 4),
    (5120, 7168, 1), (17408, 5120, 8), (5120, 5120, 32),
])
def test_full_size_27b_matrices_sampled_rows(in_f, out_f, C):
    """The 27B-shaped matrices at full size, launched exactly as the benchmark does (PDL flag,
    shared workspace); 80 sampled rows of each checked against the oracle."""
    lib()
    codes, scales = synth.qweight_torch(out_f, in_f, seed=in_f + out_f + C, device=DEV)
    cb, sb = svd.svd_native_sizes(in_f, out_f)
    nc = torch.empty(cb, dtype=torch.uint8, device=DEV)
    ns = torch.empty(sb, dtype=torch.uint8, device=DEV)
    svd.svd_repack_weights(svd.QWeight(codes, scales, in_f, out_f, svd.SVD_LAYOUT_CANONICAL), nc, ns)
    W = svd.QWeight(nc, ns, in_f, out_f, svd.SVD_LAYOUT_NATIVE)
    X = synth.activations_torch(C, in_f, seed=11, device=DEV)
    Y = torch.empty((C, out_f), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_linear(W, X, C, Y, ws, flags=svd.SVD_F_PDL)
    torch.cuda.synchronize()
    rows = _sampled_rows(out_f, 80, seed=C)
    c_h = codes[rows].cpu().numpy()
    s_h = scales[rows].cpu().numpy().view(np.uint16)
    x_h = X.view(torch.int16).cpu().numpy().view(np.uint16)
    y_ref, a_ref = oracle.verify_linear(c_h, s_h, x_h)
    assert_gemm_parity(Y.cpu().numpy()[:, rows], y_ref, a_ref)
    assert torch.isfinite(Y).all()
