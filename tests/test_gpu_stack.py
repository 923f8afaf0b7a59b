"""The whole verify pass: layer stack + lm_head + sampler + acceptance recorded into CUDA graphs
with programmatic dependent launch; replays must equal eager launches bit for bit and sampled
outputs must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import stack, svd, synth
from gpu_helpers import assert_gemm_parity, lib

pytestmark = pytest.mark.gpu


def test_graph_replay_equals_eager_and_oracle():
    lib()
    vp = stack.VerifyPass(layers=2, C=4, seed=3, keep_canonical=True)
    vp.enqueue_stack()
    vp.enqueue_tail()
    torch.cuda.synchronize()
    eager = [lin.Y.clone() for lin in vp.linears] + [vp.lm.Y.clone(), vp.probs.clone(),
                                                     vp.tokens.clone(), vp.n_emitted.clone()]
    for lin in vp.linears + [vp.lm]:
        lin.Y.fill_(float("nan"))
    vp.capture()
    for _ in range(3):
        vp.launch()
    torch.cuda.synchronize()
    replay = [lin.Y for lin in vp.linears] + [vp.lm.Y, vp.probs, vp.tokens, vp.n_emitted]
    for a, b in zip(eager, replay):
        assert torch.equal(a, b)
    assert int(vp.status.item()) == 0 and 1 <= int(vp.n_emitted.item()) <= vp.k + 1
    # sampled rows of every linear against the oracle
    g = synth.rng(0)
    for lin in vp.linears:
        rows = np.unique(np.r_[g.choice(lin.out_f, 24, replace=False), 0, lin.out_f - 1])
        codes, scales = lin.canonical
        y_ref, a_ref = oracle.verify_linear(codes[rows].cpu().numpy(),
                                            scales[rows].cpu().numpy().view(np.uint16),
                                            lin.X.view(torch.int16).cpu().numpy().view(np.uint16))
        assert_gemm_parity(lin.Y.cpu().numpy()[:, rows], y_ref, a_ref)
    # the acceptance of the window against the oracle on the same p, q and drafts
    tok_r, ne_r, st_r, near = oracle.accept(vp.probs.cpu().numpy(), vp.draft.cpu().numpy(),
                                            q=vp.q.cpu().numpy(), seed=vp.seed)
    if near[0] == 0:
        assert np.array_equal(vp.tokens.cpu().numpy(), tok_r)
        assert int(vp.n_emitted.item()) == ne_r[0] and int(vp.status.item()) == st_r[0]


def test_chain_pdl_and_plain_launches_agree():
    lib()
    a = stack.VerifyPass(layers=2, C=4, seed=5, head=False, chain=True)
    b = stack.VerifyPass(layers=2, C=4, seed=5, head=False, chain=False, pdl=True)
    c = stack.VerifyPass(layers=2, C=4, seed=5, head=False, chain=False, pdl=False)
    for v in (a, b, c):
        v.capture()
        v.launch()
    torch.cuda.synchronize()
    for x, y, z in zip(a.linears, b.linears, c.linears):
        assert torch.equal(x.Y, y.Y) and torch.equal(x.Y, z.Y)


def test_pass_with_kv_attention_matches_eager_and_oracle():
    # Two layers of the stack with each layer's KV-read attention in its place (between its
    # q|k|v and o products, the matrices in between as chain launches), recorded into one graph:
    # replays equal the eager run, the attention output matches the oracle and the last linear's
    # output equals the plain stack's.
    lib()
    vp = stack.VerifyPass(layers=2, C=4, seed=5, head=False)
    vp.enqueue_stack()
    torch.cuda.synchronize()
    y_plain = vp.linears[-1].Y.clone()
    ctx = 300
    kp = stack.KvPass(vp, ctx, seed=9)
    kp.enqueue()
    torch.cuda.synchronize()
    o_eager = kp.o.clone()
    assert torch.equal(vp.linears[-1].Y, y_plain)
    kp.o.fill_(float("nan"))
    kp.capture()
    for _ in range(2):
        kp.launch()
    torch.cuda.synchronize()
    assert torch.equal(kp.o, o_eager)
    # the oracle on host copies of the same cache bytes (every layer's cache holds this draw)
    kc, ks, vc, vs = synth.kv_cache_torch(kp.Hkv, ctx, kp.D, 9, torch.device("cuda:0"))
    q = kp.q.view(torch.int16).cpu().numpy().view(np.uint16)
    o_ref, a_ref = oracle.kv_attention(q, kc.cpu().numpy(), ks.cpu().numpy().view(np.uint16),
                                       vc.cpu().numpy(), vs.cpu().numpy().view(np.uint16), ctx - 4)
    err = np.abs(o_eager.cpu().numpy().astype(np.float64) - o_ref)
    assert np.all(err <= 2.0 ** -8 * a_ref)
