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
    # Two layers of the stack with each layer's KV cache in its place (the window's keys and
    # values appended from the q|k|v output, then attention, between the q|k|v and o products;
    # the matrices in between as chain launches), recorded into one graph: replays equal the
    # eager run, the last attention output matches the oracle over the oracle-quantised window
    # and the last linear's output equals the plain stack's.
    lib()
    vp = stack.VerifyPass(layers=2, C=4, seed=5, head=False)
    vp.enqueue_stack()
    torch.cuda.synchronize()
    y_plain = vp.linears[-1].Y.clone()
    ctx, C = 300, 4
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
    # the oracle: the cache's draw, with the window's positions quantised from the last layer's
    # q|k|v output (columns 5120.. for keys, 6144.. for values)
    Hkv, D = kp.Hkv, kp.D
    kc, ks, vc, vs = (a.cpu().numpy() for a in synth.kv_cache_torch(Hkv, ctx, D, 9,
                                                                  torch.device("cuda:0")))
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    y = vp.linears[len(vp.gemms)].Y.cpu().numpy()
    kw = y[:, synth.HIDDEN:synth.HIDDEN + Hkv * D].reshape(C * Hkv, D)
    vw = y[:, synth.HIDDEN + Hkv * D:synth.HIDDEN + 2 * Hkv * D].reshape(C * Hkv, D)
    qk, qks, qv, qvs = oracle.kv_quantize(kw, vw)
    for c in range(C):
        for h in range(Hkv):
            i, p = c * Hkv + h, ctx - C + c
            kc[h, p], ks[h, p], vc[h, p], vs[h, p] = qk[i], qks[i], qv[i], qvs[i]
    q = kp.q.view(torch.int16).cpu().numpy().view(np.uint16)
    o_ref, a_ref = oracle.kv_attention(q, kc, ks, vc, vs, ctx - C)
    err = np.abs(o_eager.cpu().numpy().astype(np.float64) - o_ref)
    assert np.all(err <= 2.0 ** -8 * a_ref)
