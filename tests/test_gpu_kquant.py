"""GPU parity of the verify GEMM on K-quant (Q4_K) super-block weights (SVD_LAYOUT_Q4K) against
the Q4_K oracle: max |delta| <= 1e-3 * sum |w x| per output, element by element on small and
ragged shapes for every C the kernel takes, and on sampled rows of full 27B-shaped matrices."""
import numpy as np
import pytest
import torch

from oracle import kquant
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, native_weight, to_dev

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


# ---- the Q4_K native layout: repacked super-blocks streamed by the tensor-core kernel ----------

def q4k_native(blocks_dev, in_f, out_f):
    cb, hb = svd.svd_q4k_native_sizes(in_f, out_f)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    hdr = torch.empty(hb, dtype=torch.uint8, device=DEV)
    svd.svd_repack_weights(svd.QWeight(blocks_dev, None, in_f, out_f, svd.SVD_LAYOUT_Q4K), codes, hdr)
    return svd.QWeight(codes, hdr, in_f, out_f, svd.SVD_LAYOUT_Q4K_NATIVE), (codes, hdr)


def run_native(W, x, out_f, ws=None, flags=0):
    C = x.shape[0]
    if ws is None:
        ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(W.in_features, out_f, C),
                         dtype=torch.uint8, device=DEV)
    Y = torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)
    svd.svd_verify_linear(W, to_dev(x), C, Y, ws, flags=flags)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


@pytest.mark.parametrize("out_f,in_f", [(37, 768), (130, 512), (64, 256), (1, 2048)])
def test_q4k_native_repack_round_trip(out_f, in_f):
    lib()
    blocks = synth.q4k_blocks(out_f, in_f, seed=out_f * 7 + in_f)
    W, _ = q4k_native(to_dev(blocks), in_f, out_f)
    back = torch.empty((out_f, in_f // 256 * 144), dtype=torch.uint8, device=DEV)
    svd.svd_unpack_weights(W, back, None)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), blocks)


@pytest.mark.parametrize("out_f,in_f,C", [
    (37, 768, 1), (37, 768, 4), (64, 256, 8), (300, 5120, 3), (33, 2304, 5), (131, 4096, 2),
    (8, 2048, 6), (1, 256, 7), (200, 17408, 4), (1100, 1280, 8),
    (37, 768, 9), (300, 5120, 12), (131, 4096, 16), (1100, 1280, 13), (1, 256, 10),
])
def test_q4k_native_matches_oracle(out_f, in_f, C):
    lib()
    blocks = synth.q4k_blocks(out_f, in_f, seed=out_f + 3 * in_f + C)
    x = synth.activations(C, in_f, seed=C + 11)
    W, _ = q4k_native(to_dev(blocks), in_f, out_f)
    y = run_native(W, x, out_f, flags=svd.SVD_F_PDL if C % 2 else 0)
    y_ref, a_ref = kquant.verify_linear(blocks, in_f, x)
    assert_gemm_parity(y, y_ref, a_ref)


def test_q4k_native_edge_values():
    """Zero and extreme scale fields: d = 0 rows, dmin = 0 rows, all sc and m at 63, codes all 0
    or all 15, large activations."""
    lib()
    out_f, in_f, C = 64, 512, 4
    blocks = synth.q4k_blocks(out_f, in_f, seed=5).reshape(out_f, 2, 144)
    blocks[0:8, :, 0:2] = 0                                  # d = 0: only the mins remain
    blocks[8:16, :, 2:4] = 0                                 # dmin = 0: no mins
    blocks[16:24, :, 4:16] = 0xFF                            # every sc, m = 63
    blocks[24:32, :, 16:] = 0x00                             # codes 0
    blocks[32:40, :, 16:] = 0xFF                             # codes 15
    blocks = blocks.reshape(out_f, 2 * 144)
    x = synth.activations(C, in_f, seed=6, std=30.0)
    W, _ = q4k_native(to_dev(blocks), in_f, out_f)
    y = run_native(W, x, out_f)
    y_ref, a_ref = kquant.verify_linear(blocks, in_f, x)
    assert_gemm_parity(y, y_ref, a_ref)


@pytest.mark.parametrize("out_f,in_f", [(7168, 5120), (5120, 17408), (34816, 5120)])
def test_q4k_native_full_size_sampled_rows(out_f, in_f):
    lib()
    C = 4
    b = synth.q4k_blocks_torch(out_f, in_f, seed=13, device=DEV)
    W, keep = q4k_native(b, in_f, out_f)
    x = synth.activations(C, in_f, seed=14)
    y = run_native(W, x, out_f)
    rows = np.unique(np.r_[synth.rng(15).choice(out_f, 40, replace=False), 0, 63, 64, out_f - 1])
    host = b[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    y_ref, a_ref = kquant.verify_linear(host, in_f, x)
    assert_gemm_parity(y[:, rows], y_ref, a_ref)


@pytest.mark.parametrize("C", [1, 4, 8, 12, 16])
def test_q4k_native_chain_equals_single_launches_and_oracle(C):
    lib()
    shapes = [(5120, 1024), (96, 256), (544, 2048), (2048, 160), (64, 512), (1024, 3000)]
    mats, ops, keep = [], [], []
    for i, (in_f, out_f) in enumerate(shapes):
        in_f = (in_f + 255) // 256 * 256
        blocks = synth.q4k_blocks(out_f, in_f, seed=100 + i + C)
        x = synth.activations(C, in_f, seed=200 + i)
        W, k = q4k_native(to_dev(blocks), in_f, out_f)
        keep.append(k)
        mats.append((blocks, in_f, x))
        ops.append((W, to_dev(x), torch.full((C, out_f), float("nan"), dtype=torch.float32, device=DEV)))
    ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_chain(ops, C, ws)
    torch.cuda.synchronize()
    chained = [Y.clone() for _, _, Y in ops]
    for (W, X, Y), ref in zip(ops, chained):
        Y.fill_(float("nan"))
        svd.svd_verify_linear(W, X, C, Y, ws)
        torch.cuda.synchronize()
        assert torch.equal(Y, ref)
    for (blocks, in_f, x), y in zip(mats, chained):
        y_ref, a_ref = kquant.verify_linear(blocks, in_f, x)
        assert_gemm_parity(y.cpu().numpy(), y_ref, a_ref)


def test_q4k_native_chain_reads_what_the_previous_op_wrote():
    lib()
    C, in_f, out_f = 4, 256, 128
    blocks = synth.q4k_blocks(out_f, in_f, seed=21)
    W, keep = q4k_native(to_dev(blocks), in_f, out_f)
    X = to_dev(synth.activations(C, in_f, seed=22))

    def run(chained):
        Y0 = torch.zeros((C, out_f), dtype=torch.float32, device=DEV)
        X1 = Y0.view(torch.int16)  # [C][256] bf16 bit patterns
        Y1 = torch.zeros((C, out_f), dtype=torch.float32, device=DEV)
        ops = [(W, X, Y0), (W, X1, Y1)]
        ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, C), dtype=torch.uint8, device=DEV)
        if chained:
            svd.svd_verify_chain(ops, C, ws)
        else:
            for Wi, Xi, Yi in ops:
                svd.svd_verify_linear(Wi, Xi, C, Yi, ws)
        torch.cuda.synchronize()
        return Y1.view(torch.int32).clone()

    a, b = run(True), run(False)
    assert torch.equal(a, b)
    assert torch.count_nonzero(a) > 0


def test_q4k_native_argument_errors():
    lib()
    blocks = to_dev(synth.q4k_blocks(16, 512, seed=1))
    W, keep = q4k_native(blocks, 512, 16)
    X = to_dev(synth.activations(17, 512, seed=2))
    Y = torch.empty((17, 16), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(512, 16, 17), dtype=torch.uint8, device=DEV)
    with pytest.raises(svd.SvdError) as e:                       # C > 16
        svd.svd_verify_linear(W, X, 17, Y, ws)
    assert e.value.code == svd.SVD_ERR_UNSUPPORTED
    with pytest.raises(svd.SvdError) as e:                       # no workspace
        svd.svd_verify_linear(W, X, 4, Y, None)
    assert e.value.code == svd.SVD_ERR_WORKSPACE
    with pytest.raises(svd.SvdError) as e:                       # in % 256
        svd.svd_verify_linear(svd.QWeight(W.codes, W.scales, 480, 16, svd.SVD_LAYOUT_Q4K_NATIVE), X, 4, Y, ws)
    assert e.value.code == svd.SVD_ERR_INVALID_ARG
    with pytest.raises(svd.SvdError) as e:                       # unpack wants dst_scales NULL
        svd.svd_unpack_weights(W, torch.empty(16 * 288, dtype=torch.uint8, device=DEV), ws)
    assert e.value.code == svd.SVD_ERR_INVALID_ARG
    # a chain takes one layout
    codes, scales = synth.qweight(16, 512, seed=3)
    Wn, _ = native_weight(codes, scales)
    ops = [(W, X, Y), (Wn, X, Y)]
    cws = torch.zeros(svd.svd_verify_chain_workspace_bytes(ops, 4), dtype=torch.uint8, device=DEV)
    with pytest.raises(svd.SvdError) as e:
        svd.svd_verify_chain(ops, 4, cws)
    assert e.value.code == svd.SVD_ERR_INVALID_ARG


def test_q4k_stack_graph_matches_oracle():
    """stack.Q4kStack (the bench's Q4_K stack, one chain launch replayed from a CUDA graph) on a
    small two-layer stack: every product matches the oracle on the weights read back from the
    native layout, and no wait gave up."""
    from speculative_decoding_verify_06_gb300 import stack
    lib()
    qs = stack.Q4kStack(layers=2, C=4, seed=3, device=DEV, gemms=((512, 768), (768, 256))).capture()
    for Y in (op[2] for op in qs.ops):
        Y.fill_(float("nan"))
    qs.launch()
    torch.cuda.synchronize()
    assert svd.svd_verify_status(qs.ws) == (svd.SVD_OK, 0)
    for W, X, Y in qs.ops:
        raw = torch.empty((W.out_features, W.in_features // 256 * 144), dtype=torch.uint8, device=DEV)
        svd.svd_unpack_weights(W, raw, None)
        x = X.view(torch.int16).cpu().numpy().view(np.uint16)
        y_ref, a_ref = kquant.verify_linear(raw.cpu().numpy(), W.in_features, x)
        assert_gemm_parity(Y.cpu().numpy(), y_ref, a_ref)


@pytest.mark.parametrize("C", [4, 12])
def test_q4k_native_wait_runs_out_and_is_reported(C):
    """The stall hook on a Q4_K launch: no weight copy is issued, the first ring wait runs out,
    the status word reports it, and the same workspace then gives the oracle's result."""
    lib()
    out_f, in_f = 7168, 5120
    b = synth.q4k_blocks_torch(out_f, in_f, seed=31, device=DEV)
    W, keep = q4k_native(b, in_f, out_f)
    x = synth.activations(C, in_f, seed=32)
    X = to_dev(x)
    Y = torch.empty((C, out_f), dtype=torch.float32, device=DEV)
    ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(in_f, out_f, C), dtype=torch.uint8, device=DEV)
    svd.svd_verify_inject_stall(ws, 0)
    svd.svd_verify_linear(W, X, C, Y, ws)
    rc, bits = svd.svd_verify_status(ws)
    assert rc == svd.SVD_ERR_TIMEOUT and bits != 0 and bits & ~7 == 0
    svd.svd_verify_inject_stall(ws, None)
    Y.fill_(float("nan"))
    svd.svd_verify_linear(W, X, C, Y, ws)
    assert svd.svd_verify_status(ws) == (svd.SVD_OK, 0)
    rows = np.r_[0:64, out_f - 64:out_f]
    host = b[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    y_ref, a_ref = kquant.verify_linear(host, in_f, x)
    assert_gemm_parity(Y.cpu().numpy()[:, rows], y_ref, a_ref)
