"""The verify-linear entry point that allocates nothing (svd_verify_linear_noalloc).

Some callers cannot allocate device memory where they run the verify pass -- the allocator is
owned by someone else, or allocating is not allowed in that context -- so this entry point
keeps the kernel's scratch in the library's own device memory instead of a caller workspace.
The test calls it through the C ABI twice in a row.  Each result must equal, bit for bit, that of
svd_verify_linear on the same inputs (both run the same deterministic kernel and summation
order; the scratch only holds the tagged partial sums of row blocks split between CTAs and the
counters), and must match the oracle within the GEMM tolerance the other tests use
(|delta| <= 1e-3 * sum |w x| per output).  The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, native_weight, to_dev

pytestmark = pytest.mark.gpu


def _compare(out_f, in_f, C, seed):
    codes, scales = synth.qweight(out_f, in_f, seed=seed)
    x = synth.activations(C, in_f, seed=seed + 1)
    W, _ = native_weight(codes, scales)
    X = to_dev(x)
    y_ws = torch.empty((C, out_f), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8,
                     device=DEV)
    svd.svd_verify_linear(W, X, C, y_ws, ws)
    y = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
    svd.svd_verify_linear_noalloc(W, X, C, y)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y_ws.view(torch.int32))
    y_ref, a_ref = oracle.verify_linear(codes, scales, x)
    assert_gemm_parity(y.cpu().numpy(), y_ref, a_ref)


def test_noalloc_matches_verify_linear_on_two_calls_in_a_row():
    lib()
    # 2048 x 2048 at K+1 = 4: row blocks are split between CTAs, so owners read tagged partials
    # from the scratch
    _compare(2048, 2048, 4, seed=11)
    # the next call reuses whatever the first one left in the shared scratch
    _compare(1000, 544, 6, seed=12)


def test_noalloc_rejects_too_many_rows():
    lib()
    out_f = 262144 + 64  # above the scratch's row limit: rejected before any launch
    W = svd.QWeight(torch.zeros(16, dtype=torch.uint8, device=DEV),
                    torch.zeros(16, dtype=torch.uint8, device=DEV), 64, out_f,
                    svd.SVD_LAYOUT_NATIVE)
    X = torch.zeros((1, 64), dtype=torch.bfloat16, device=DEV)
    Y = torch.zeros((1, 16), dtype=torch.float32, device=DEV)
    with pytest.raises(svd.SvdError) as e:
        svd.svd_verify_linear_noalloc(W, X, 1, Y)
    assert e.value.code == svd.SVD_ERR_UNSUPPORTED
