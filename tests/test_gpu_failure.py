"""Failure detection of the verify kernels and the KV-read attention, tested without a GPU fault.

Every spin-wait of these kernels is bounded.  A test hook in the workspace injects a stall: the
verify kernels issue no weight copy, as if the copy engine had stopped, and give up a wait after
a few polls, so their first ring wait really runs out; the KV attention's hook makes its ring
waits give up at once.  The kernel must then record
the give-up in the workspace, stop, let its own copies land and return -- no hang, no fault --
and the context must stay usable: the next call with the default limit gives the oracle's
result.  The partial-sum tags are also checked across the wrap of their launch epoch."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, native_weight, to_dev

pytestmark = pytest.mark.gpu


def _linear(out_f, in_f, C, seed):
    codes, scales = synth.qweight(out_f, in_f, seed=seed)
    x = synth.activations(C, in_f, seed=seed + 1)
    W, _ = native_weight(codes, scales)
    return codes, scales, x, W


def test_verify_linear_wait_runs_out_and_is_reported():
    lib()
    C, in_f, out_f = 4, 5120, 17408
    codes, scales, x, W = _linear(out_f, in_f, C, seed=41)
    X = to_dev(x)
    Y = torch.empty((C, out_f), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8,
                     device=DEV)
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)
    svd.svd_verify_inject_stall(ws, 0)
    svd.svd_verify_linear(W, X, C, Y, ws)
    rc, bits = svd.svd_verify_status(ws)
    assert rc == svd.SVD_ERR_TIMEOUT and bits != 0 and bits & ~7 == 0
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)  # the query cleared it
    # the stall injection off: the same workspace and context give the oracle's result
    svd.svd_verify_inject_stall(ws, None)
    Y.fill_(float("nan"))
    svd.svd_verify_linear(W, X, C, Y, ws)
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)
    rows = np.r_[0:64, out_f - 64:out_f, 8000:8064]
    y_ref, a_ref = oracle.verify_linear(codes[rows], scales[rows], x)
    assert_gemm_parity(Y.cpu().numpy()[:, rows], y_ref, a_ref)


def test_chain_wait_runs_out_and_is_reported():
    lib()
    C = 4
    mats, ops = [], []
    for i, (in_f, out_f) in enumerate([(512, 2048), (2048, 1024), (1024, 3000), (3000 // 32 * 32, 640)]):
        codes, scales, x, W = _linear(out_f, in_f, C, seed=50 + i)
        mats.append((codes, scales, x))
        ops.append((W, to_dev(x), torch.empty((C, out_f), dtype=torch.float32, device=DEV)))
    ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_inject_stall(ws, 0)
    svd.svd_verify_chain(ops, C, ws)
    rc, bits = svd.svd_verify_status(ws)
    assert rc == svd.SVD_ERR_TIMEOUT and bits != 0
    svd.svd_verify_inject_stall(ws, None)
    svd.svd_verify_chain(ops, C, ws)
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)
    for (codes, scales, x), (_, _, Y) in zip(mats, ops):
        y_ref, a_ref = oracle.verify_linear(codes, scales, x)
        assert_gemm_parity(Y.cpu().numpy(), y_ref, a_ref)


def test_partial_tags_across_the_epoch_wrap():
    """The launch epoch sits in the workspace's last word; partial tags repeat every 2^24 - 1
    launches.  Stale entries carrying the first tag of the next cycle are planted in every
    partial slot just before the wrap: the launch at the wrap clears them, so the launches after
    it still give exactly the bits of an ordinary launch."""
    lib()
    C, in_f, out_f = 4, 2048, 2048  # row blocks split between CTAs: owners read partials
    codes, scales, x, W = _linear(out_f, in_f, C, seed=61)
    X = to_dev(x)
    nbytes = svd.svd_verify_linear_workspace_bytes(in_f, out_f, C)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    ref = torch.empty((C, out_f), dtype=torch.float32, device=DEV)
    svd.svd_verify_linear(W, X, C, ref, ws)
    words = ws.view(torch.int32)
    part = ws[:nbytes - 256].view(torch.int64)
    stale = (1 << 8) << 32 | int(np.float32(1e30).view(np.uint32))  # tag of (e24 = 1, op 0)
    part.fill_(stale)
    words[-1] = 0xFFFFFF - 2  # three launches before the epoch's e24 comes back to 1
    torch.cuda.synchronize()
    for i in range(6):
        Y = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
        svd.svd_verify_linear(W, X, C, Y, ws)
        torch.cuda.synchronize()
        assert torch.equal(Y, ref), f"launch {i} across the wrap differs"
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)


def test_kv_attention_wait_runs_out_and_is_reported():
    """The hook word set to 1 makes every ring wait of the split pass give up at once (the
    kernel is compute-bound, so its copies have usually landed before it waits).  The give-up
    sets bit 0 of the workspace's first word and the kernel lets its copies in flight land and
    returns; the next call with the default limit gives the bits of a call made before."""
    lib()
    Hq, Hkv, D, C = 40, 8, synth.HEAD_DIM, 4
    L = 32_768
    n_past = L - C
    kc, ks, vc, vs = synth.kv_cache_torch(Hkv, L, D, 73, DEV)
    cache = torch.empty(svd.svd_kv_cache_bytes(Hkv, L), dtype=torch.uint8, device=DEV)
    svd.svd_kv_repack(kc, ks, vc, vs, Hkv, L, 0, L, cache, L)
    del kc, ks, vc, vs
    qd = to_dev(synth.queries(C, Hq, D, seed=74))
    ws = torch.zeros(svd.svd_kv_attention_workspace_bytes(Hq, Hkv, C), dtype=torch.uint8, device=DEV)
    words = ws[:8].view(torch.int32)

    def run():
        out = torch.full((C, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
        svd.svd_kv_attention(qd, cache, L, Hq, Hkv, n_past, C, 1.0 / np.sqrt(D), out, ws)
        torch.cuda.synchronize()
        return out

    before = run()
    assert int(words[0].item()) == 0
    words[1] = 1  # every ring wait gives up at once
    run()
    assert int(words[0].item()) & 1 == 1
    words[0] = 0
    words[1] = 0
    after = run()
    assert int(words[0].item()) == 0
    assert torch.equal(after.view(torch.int32), before.view(torch.int32))
