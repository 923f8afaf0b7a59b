"""GPU parity of the batched verify GEMM on the tcgen05 tensor cores (17..32 activation columns)
against the oracle: max |delta| <= 1e-3 * sum |w x| per output, and -- the kernel's own
arithmetic, fp16 weights s * (c - 8) rounded once and activations rounded from bf16 to fp16 --
within 2^-10 * sum |w x|.  Shapes cover one row block (the second of the 128-row MMA unit
missing), a 32-input tail chunk, ragged row counts, ranges that split row groups between CTAs
and pipes, and a full 27B-shaped matrix; C covers the padded token columns.  Results are
deterministic and a chain equals its single launches bit for bit; the warp-level kernel
(SVD_F_FRAGMENT_MMA) agrees within the bound; a stalled launch reports SVD_ERR_TIMEOUT and the
context stays usable."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, native_weight, to_dev, verify_linear

pytestmark = pytest.mark.gpu

FP16_BOUND = 2.0 ** -10  # 2^-11 per weight rounding, doubled for fp32 accumulation and slack


@pytest.mark.parametrize("out_f,in_f,C", [
    (64, 64, 17),      # one native row block: rows 64..127 of the MMA unit do not exist
    (200, 160, 20),    # in % 64 == 32: the last chunk has one scale block
    (130, 2048, 25),   # ragged rows
    (7, 32, 32),
    (1000, 5120, 32),  # 8 row groups x 80 chunks over the grid: split row groups, owner waits
    (4096, 256, 18),   # many short row groups: several segments per CTA
    (5120, 5120, 32),
])
def test_tensor_core_path_matches_oracle(out_f, in_f, C):
    codes, scales = synth.qweight(out_f, in_f, seed=out_f + 7 * in_f + C)
    x = synth.activations(C, in_f, seed=C + 3)
    W, _ = native_weight(codes, scales)
    y = verify_linear(W, x)
    y_ref, a_ref = oracle.verify_linear(codes, scales, x)
    worst = assert_gemm_parity(y, y_ref, a_ref)
    assert worst <= FP16_BOUND, worst


def test_deterministic_and_fragment_kernel_agrees():
    out_f, in_f, C = 2048, 3072, 32
    codes, scales = synth.qweight(out_f, in_f, seed=11)
    x = synth.activations(C, in_f, seed=12)
    W, _ = native_weight(codes, scales)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8,
                     device=DEV)
    y1 = verify_linear(W, x, ws=ws)
    y2 = verify_linear(W, x, ws=ws)
    y3 = verify_linear(W, x, flags=svd.SVD_F_PDL, ws=ws)
    assert np.array_equal(y1, y2) and np.array_equal(y1, y3)
    yf = verify_linear(W, x, flags=svd.SVD_F_FRAGMENT_MMA, ws=ws)
    y_ref, a_ref = oracle.verify_linear(codes, scales, x)
    assert assert_gemm_parity(y1, y_ref, a_ref) <= FP16_BOUND
    assert_gemm_parity(yf, y_ref, a_ref)
    # the fragment kernel is exact up to fp32 sums: the two differ by the fp16 rounding only
    assert np.all(np.abs(y1.astype(np.float64) - yf) <= FP16_BOUND * a_ref)


def test_chain_equals_single_launches():
    lib()
    C = 32
    shapes = [(1024, 2048), (2048, 1024), (1024, 3072), (3072, 640)]
    ops, mats = [], []
    for i, (in_f, out_f) in enumerate(shapes):
        codes, scales = synth.qweight(out_f, in_f, seed=70 + i)
        x = synth.activations(C, in_f, seed=80 + i)
        W, _ = native_weight(codes, scales)
        mats.append((codes, scales, x))
        ops.append((W, to_dev(x), torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)))
    ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_chain(ops, C, ws)
    torch.cuda.synchronize()
    for (W, X, Y), (codes, scales, x) in zip(ops, mats):
        single = verify_linear(W, x)
        assert np.array_equal(Y.cpu().numpy(), single)
        y_ref, a_ref = oracle.verify_linear(codes, scales, x)
        assert assert_gemm_parity(single, y_ref, a_ref) <= FP16_BOUND


def test_chain_reads_what_the_previous_op_wrote():
    """Op 1 reads, as its bf16 activations, the bytes op 0 writes as fp32 outputs: the chain
    gives the same bits as two launches ordered by the stream."""
    C, in_f, out_f = 32, 256, 128
    codes, scales = synth.qweight(out_f, in_f, seed=1)
    W, _ = native_weight(codes, scales)
    X = to_dev(synth.activations(C, in_f, seed=2))

    def run(chained):
        Y0 = torch.zeros((C, out_f), dtype=torch.float32, device=DEV)
        Y1 = torch.zeros((C, out_f), dtype=torch.float32, device=DEV)
        ops = [(W, X, Y0), (W, Y0.view(torch.int16), Y1)]
        ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8, device=DEV)
        if chained:
            svd.svd_verify_chain(ops, C, ws)
        else:
            for Wi, Xi, Yi in ops:
                svd.svd_verify_linear(Wi, Xi, C, Yi, ws)
        torch.cuda.synchronize()
        return Y1.view(torch.int32).clone()

    a, b = run(True), run(False)
    assert torch.equal(a, b) and (a != 0).any()


def test_stalled_launch_reports_timeout_and_recovers():
    lib()
    C, in_f, out_f = 32, 5120, 5120
    codes, scales = synth.qweight(out_f, in_f, seed=91)
    x = synth.activations(C, in_f, seed=92)
    W, _ = native_weight(codes, scales)
    X = to_dev(x)
    Y = torch.empty((C, out_f), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8,
                     device=DEV)
    svd.svd_verify_inject_stall(ws, 0)
    svd.svd_verify_linear(W, X, C, Y, ws)
    rc, bits = svd.svd_verify_status(ws)
    assert rc == svd.SVD_ERR_TIMEOUT and bits != 0 and bits & ~7 == 0
    svd.svd_verify_inject_stall(ws, None)
    Y.fill_(float("nan"))
    svd.svd_verify_linear(W, X, C, Y, ws)
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)
    rows = np.r_[0:128, 2500:2628, out_f - 128:out_f]
    y_ref, a_ref = oracle.verify_linear(codes[rows], scales[rows], x)
    assert assert_gemm_parity(Y.cpu().numpy()[:, rows], y_ref, a_ref) <= FP16_BOUND
