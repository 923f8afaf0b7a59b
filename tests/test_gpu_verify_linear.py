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


def _ops_for(shapes, C, seed):
    mats, ops = [], []
    for n, (in_f, out_f) in enumerate(shapes):
        codes, scales = synth.qweight(out_f, in_f, seed=seed + n)
        x = synth.activations(C, in_f, seed=seed + 100 + n)
        W, _ = native_weight(codes, scales)
        X = to_dev(x)
        Y = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
        mats.append((codes, scales, x))
        ops.append((W, X, Y))
    return mats, ops


@pytest.mark.parametrize("C", [1, 4, 6, 8, 16, 32])
def test_chain_equals_single_launches_and_oracle(C):
    """A chain mixing large, small and ragged matrices (some with fewer units than CTAs) equals
    one svd_verify_linear per op bit for bit, and matches the oracle."""
    shapes = [(5120, 1024), (96, 40), (544, 2048), (2048, 160), (64, 64), (1024, 3000), (32, 7)]
    mats, ops = _ops_for(shapes, C, seed=C)
    ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_chain(ops, C, ws)
    torch.cuda.synchronize()
    chained = [Y.clone() for _, _, Y in ops]
    for (W, X, Y), ref in zip(ops, chained):
        Y.fill_(float("nan"))
        svd.svd_verify_linear(W, X, C, Y, ws)
        torch.cuda.synchronize()
        assert torch.equal(Y, ref)
    for (codes, scales, x), y in zip(mats, chained):
        y_ref, a_ref = oracle.verify_linear(codes, scales, x)
        assert_gemm_parity(y.cpu().numpy(), y_ref, a_ref)


def test_chain_reads_what_the_previous_op_wrote():
    """Op 1 reads, as its bf16 activations, the bytes op 0 writes as fp32 outputs.  The chain
    must give the same bits as two launches ordered by the stream; reading op 1's input before
    op 0 finished would see the zeros it starts from."""
    C = 4
    in_f, out_f = 256, 128
    codes, scales = synth.qweight(out_f, in_f, seed=1)
    W, _ = native_weight(codes, scales)
    X = to_dev(synth.activations(C, in_f, seed=2))

    def run(chained: bool):
        Y0 = torch.zeros((C, out_f), dtype=torch.float32, device=DEV)
        X1 = Y0.view(torch.int16)  # [C][256] bf16 bit patterns
        Y1 = torch.zeros((C, out_f), dtype=torch.float32, device=DEV)
        ops = [(W, X, Y0), (W, X1, Y1)]
        ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8,
                         device=DEV)
        if chained:
            svd.svd_verify_chain(ops, C, ws)
        else:
            for Wi, Xi, Yi in ops:
                svd.svd_verify_linear(Wi, Xi, C, Yi, ws)
        torch.cuda.synchronize()
        return Y1.view(torch.int32).clone()

    a, b = run(True), run(False)
    assert torch.equal(a, b)
    assert (a != 0).any()


def test_long_chain_splits_into_launches():
    C = 2
    shapes = [(64, 64), (96, 128)] * 150  # 300 ops: two launches of the chain kernel
    mats, ops = _ops_for(shapes, C, seed=7)
    ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_chain(ops, C, ws)
    torch.cuda.synchronize()
    for i in (0, 1, 255, 256, 299):
        codes, scales, x = mats[i]
        y_ref, a_ref = oracle.verify_linear(codes, scales, x)
        assert_gemm_parity(ops[i][2].cpu().numpy(), y_ref, a_ref)
