"""Helpers for the GPU parity tests: move seeded inputs to the device and call the C ABI."""
import numpy as np
import torch

from speculative_decoding_verify_06_gb300 import build, svd

DEV = torch.device("cuda:0")
_built = False


def lib():
    global _built
    if not _built:
        build.build_library()
        _built = True
    return svd.load()


def to_dev(a: np.ndarray):
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def native_weight(codes: np.ndarray, scales: np.ndarray):
    """Canonical host arrays -> NATIVE device QWeight (through svd_repack_weights)."""
    lib()
    out_f, half = codes.shape
    in_f = 2 * half
    cb, sb = svd.svd_native_sizes(in_f, out_f)
    nc = torch.empty(cb, dtype=torch.uint8, device=DEV)
    ns = torch.empty(sb, dtype=torch.uint8, device=DEV)
    src = svd.QWeight(to_dev(codes), to_dev(scales), in_f, out_f, svd.SVD_LAYOUT_CANONICAL)
    svd.svd_repack_weights(src, nc, ns)
    return svd.QWeight(nc, ns, in_f, out_f, svd.SVD_LAYOUT_NATIVE), src


def verify_linear(W, x_bf16: np.ndarray, flags: int = 0, ws=None):
    C = x_bf16.shape[0]
    X = to_dev(x_bf16)
    Y = torch.full((C, W.out_features), float("nan"), dtype=torch.float32, device=DEV)
    if ws is None and W.layout == svd.SVD_LAYOUT_NATIVE:
        ws = torch.zeros(svd.svd_verify_linear_workspace_bytes(W.in_features, W.out_features, C),
                         dtype=torch.uint8, device=DEV)
    svd.svd_verify_linear(W, X, C, Y, ws, flags=flags)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


def assert_gemm_parity(y, y_ref, a_ref, tol=1e-3):
    """max |delta| <= tol * sum |w x| per output."""
    err = np.abs(y.astype(np.float64) - y_ref)
    bound = tol * a_ref
    bad = ~(err <= bound)
    assert not bad.any(), (f"{bad.sum()} outputs out of tolerance; worst ratio "
                           f"{np.nanmax(err / np.maximum(a_ref, 1e-300)):.3e}")
    return float(np.max(err / np.maximum(a_ref, 1e-300)))


def sampler(logits: np.ndarray, smp):
    """svd_sampler_probs over the rows, SVD_C_MAX rows (one call's limit) at a time."""
    rows, V = logits.shape
    L = to_dev(logits.astype(np.float32))
    P = torch.empty_like(L)
    am = torch.empty(rows, dtype=torch.int32, device=DEV)
    step = min(rows, svd.SVD_C_MAX)
    ws = torch.zeros(svd.svd_sampler_workspace_bytes(step, V), dtype=torch.uint8, device=DEV)
    for r0 in range(0, rows, step):
        n = min(step, rows - r0)
        svd.svd_sampler_probs(L[r0:r0 + n], n, V, smp, P[r0:r0 + n], am[r0:r0 + n], ws)
    torch.cuda.synchronize()
    return P.cpu().numpy(), am.cpu().numpy()


def accept(p, draft, q=None, p_rows=None, q_rows=None, target_argmax=None, seed=0, woff=0,
           uniforms=None, V=None):
    n, k = draft.shape
    V = V or p.shape[-1]
    args = {}
    tp = to_dev(np.ascontiguousarray(p, np.float32))
    tq = None if q is None else to_dev(np.ascontiguousarray(q, np.float32))
    tok = torch.full((n, k + 1), -7, dtype=torch.int32, device=DEV)
    ne = torch.full((n,), -7, dtype=torch.int32, device=DEV)
    st = torch.full((n,), -7, dtype=torch.int32, device=DEV)
    svd.svd_accept(tp, to_dev(draft.astype(np.int32)), n, k, V, tok, ne, st, q=tq,
                   p_rows=None if p_rows is None else to_dev(p_rows.astype(np.int64)),
                   q_rows=None if q_rows is None else to_dev(q_rows.astype(np.int64)),
                   target_argmax=None if target_argmax is None else to_dev(target_argmax.astype(np.int32)),
                   seed=seed, window_offset=woff,
                   uniforms=None if uniforms is None else to_dev(uniforms.astype(np.float32)))
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ne.cpu().numpy(), st.cpu().numpy()
