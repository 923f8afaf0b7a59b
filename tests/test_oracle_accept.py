"""Pins of the oracle's acceptance rule: the greedy worked example of the HN thread, Monte-Carlo
exactness of the sampled output distribution on a vocabulary of 8, the acceptance rate
sum(min(p, q)), the expected tokens per pass under i.i.d. acceptance, and the invariants."""
import json
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import formulas
from speculative_decoding_verify_06_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _onehot_rows(ids, V):
    p = np.zeros((len(ids), V), np.float32)
    p[np.arange(len(ids)), ids] = 1.0
    return p


def test_greedy_worked_example():
    g = json.load(open(os.path.join(GOLD, "greedy_example.json")))
    alpha = g["alphabet"]
    V = len(alpha)
    drafts = np.array([[alpha.index(c) for c in g["drafts"]]], np.int32)
    k = drafts.shape[1]
    for case in g["cases"]:
        tgt = [alpha.index(c) for c in case["target"]]
        bonus = alpha.index("A")  # the target's token after the last draft (unused here)
        p = _onehot_rows(tgt + [bonus], V)
        tok, ne, st, _ = oracle.accept(p, drafts)
        want = [alpha.index(c) for c in case["emitted"]]
        assert ne[0] == len(want) and list(tok[0, : ne[0]]) == want and st[0] == 0
        assert np.all(tok[0, ne[0]:] == -1)
        # the same decisions from an explicit target argmax
        tok2, ne2, _, _ = oracle.accept(p, drafts, target_argmax=np.array([tgt + [bonus]], np.int32))
        assert np.array_equal(tok, tok2) and np.array_equal(ne, ne2)
    # all drafts match: k + 1 tokens, the last the target's own
    p = _onehot_rows(list(drafts[0]) + [alpha.index("G")], V)
    tok, ne, _, _ = oracle.accept(p, drafts)
    assert ne[0] == k + 1 and list(tok[0]) == list(drafts[0]) + [alpha.index("G")]


def _pq_with_overlap(alpha, V=8):
    """p on tokens 0..3, q = alpha p + (1 - alpha) r with r on tokens 4..7: sum min(p,q) = alpha."""
    p = np.array([0.4, 0.3, 0.2, 0.1, 0, 0, 0, 0], np.float64)
    r = np.array([0, 0, 0, 0, 0.1, 0.2, 0.3, 0.4], np.float64)
    q = alpha * p + (1 - alpha) * r
    return p.astype(np.float32), q.astype(np.float32)


def _run_windows(p_pos, q_pos, n, seed, drafter="stochastic"):
    """Windows whose position i uses (p_pos[i], q_pos[i]); drafts drawn by the harness."""
    k = len(q_pos)
    V = p_pos[0].shape[0]
    P = np.stack(p_pos).astype(np.float32)
    Q = np.stack(q_pos).astype(np.float32)
    p_rows = np.tile(np.arange(k + 1, dtype=np.int64), (n, 1))
    q_rows = np.tile(np.arange(k, dtype=np.int64), (n, 1))
    draft = np.empty((n, k), np.int32)
    for i in range(k):
        if drafter == "greedy":
            draft[:, i] = int(np.argmax(Q[i]))
        else:
            draft[:, i] = synth.draw_from(np.repeat(Q[i][None], n, 0), seed * 131 + i)
    return oracle.accept(P, draft, q=Q, seed=seed, p_rows=p_rows, q_rows=q_rows), draft


@pytest.mark.parametrize("case", ["mixed", "disjoint", "equal", "general"])
def test_sampled_output_distribution_is_exactly_p(case):
    V, k, n = 8, 3, 400_000
    g = synth.rng(42)
    if case == "mixed":
        p_pos = [_pq_with_overlap(0.6)[0]] * (k + 1)
        q_pos = [_pq_with_overlap(0.6)[1]] * k
    elif case == "disjoint":
        p_pos = [_pq_with_overlap(0.0)[0]] * (k + 1)
        q_pos = [_pq_with_overlap(0.0)[1]] * k
    elif case == "equal":
        pp = g.dirichlet(np.ones(V)).astype(np.float32)
        p_pos = [pp] * (k + 1)
        q_pos = [pp] * k
    else:
        p_pos = [g.dirichlet(np.ones(V)).astype(np.float32) for _ in range(k + 1)]
        q_pos = [g.dirichlet(np.ones(V) * 0.5).astype(np.float32) for _ in range(k)]
    (tok, ne, st, _), _ = _run_windows(p_pos, q_pos, n, seed=7)
    assert np.all(st == 0)
    assert np.all((ne >= 1) & (ne <= k + 1))
    for i in range(k + 1):
        reached = ne > i
        obs = np.bincount(tok[reached, i], minlength=V)
        exp = p_pos[i].astype(np.float64) / p_pos[i].sum() * reached.sum()
        support = exp > 0
        assert obs[~support].sum() == 0
        if support.sum() > 1:
            e = exp[support] * (obs[support].sum() / exp[support].sum())
            pval = stats.chisquare(obs[support], e).pvalue
            assert pval > 1e-4, (case, i, obs, exp)


@pytest.mark.parametrize("alpha", [0.35, 0.6, 0.9])
def test_first_position_acceptance_is_sum_min(alpha):
    p, q = _pq_with_overlap(alpha)
    n = 200_000
    (tok, ne, st, _), draft = _run_windows([p, p], [q], n, seed=3)
    acc = (ne >= 2).mean()
    a_true = formulas.acceptance_rate(p, q)
    assert abs(a_true - alpha) < 1e-6
    assert abs(acc - a_true) < 5 * np.sqrt(a_true * (1 - a_true) / n)


def test_greedy_drafter_acceptance_is_p_of_argmax_q():
    g = synth.rng(5)
    p = g.dirichlet(np.ones(8)).astype(np.float32)
    q = g.dirichlet(np.ones(8)).astype(np.float32)
    n = 200_000
    # a greedy drafter's own distribution is the one-hot at argmax q
    q1 = np.zeros_like(q)
    q1[int(np.argmax(q))] = 1.0
    (tok, ne, st, _), draft = _run_windows([p, p], [q1], n, seed=4, drafter="greedy")
    assert np.all(draft == int(np.argmax(q)))
    acc = (ne >= 2).mean()
    a_true = formulas.greedy_drafter_acceptance(p, q)
    assert abs(acc - a_true) < 5 * np.sqrt(a_true * (1 - a_true) / n)


@pytest.mark.parametrize("alpha,k", [(0.35, 1), (0.5, 3), (0.7, 5), (0.8, 3), (0.9, 5)])
def test_mean_tokens_per_pass_matches_closed_form(alpha, k):
    p, q = _pq_with_overlap(alpha)
    n = 200_000
    (tok, ne, st, _), _ = _run_windows([p] * (k + 1), [q] * k, n, seed=11)
    m, se = ne.mean(), ne.std() / np.sqrt(n)
    assert abs(m - formulas.expected_tokens_per_pass(alpha, k)) < 4 * se


def test_status_and_edge_cases():
    V, k = 8, 2
    p = np.full((1, k + 1, V), 1.0 / V, np.float32)
    q = np.full((1, k, V), 1.0 / V, np.float32)
    # a draft id outside the vocabulary is rejected and flagged
    tok, ne, st, _ = oracle.accept(p, np.array([[V + 3, 0]], np.int32), q=q, seed=1)
    assert st[0] & 1 and ne[0] == 1 and 0 <= tok[0, 0] < V
    # p == q: every draft is accepted, the window emits k + 1 tokens
    tok, ne, st, _ = oracle.accept(p, np.array([[1, 2]], np.int32), q=q, seed=1)
    assert st[0] == 0 and ne[0] == k + 1 and list(tok[0, :2]) == [1, 2]
    # q(x) = 0 for a drafted token is flagged; the test u*q < p still decides (accepts)
    q0 = q.copy()
    q0[0, 0, 5] = 0.0
    tok, ne, st, _ = oracle.accept(p, np.array([[5, 2]], np.int32), q=q0, seed=1)
    assert st[0] & 2 and tok[0, 0] == 5
    # a NaN probability in a row that is read (the bonus row: p == q accepts both drafts) is
    # flagged; rows that are never scanned are not
    pn = p.copy()
    pn[0, k, 3] = np.nan
    _, _, st, _ = oracle.accept(pn, np.array([[1, 2]], np.int32), q=q, seed=1)
    assert st[0] & 4
    # zero residual mass (p <= q everywhere at the rejected position) falls back to p
    p2 = p.copy()
    p2[0, 0] = 0.0
    p2[0, 0, 7] = 1.0
    q2 = q.copy()
    q2[0, 0] = 0.0
    q2[0, 0, 7] = 1.0
    uni = np.zeros((1, k + 1, 2), np.float32)
    uni[0, 0, 0] = 0.5
    # draft 3 has q = 0 and p = 0: rejected; (p - q)+ = 0 -> draw from p -> token 7
    tok, ne, st, _ = oracle.accept(p2, np.array([[3, 2]], np.int32), q=q2, uniforms=uni)
    assert st[0] & 8 and tok[0, 0] == 7 and ne[0] == 1


def test_uniform_hook_reproduces_philox_stream():
    V, k, n = 16, 3, 500
    g = synth.rng(8)
    p = g.dirichlet(np.ones(V), size=n * (k + 1)).astype(np.float32)
    q = g.dirichlet(np.ones(V), size=n * k).astype(np.float32)
    draft = g.integers(0, V, size=(n, k)).astype(np.int32)
    seed, woff = 1234567, 99
    uni = np.array([[oracle.uniforms(seed, woff + w, i) for i in range(k + 1)] for w in range(n)],
                   np.float32)
    a = oracle.accept(p, draft, q=q, seed=seed, window_offset=woff)
    b = oracle.accept(p, draft, q=q, uniforms=uni)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x, y)
