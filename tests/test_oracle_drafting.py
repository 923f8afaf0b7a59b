"""Pins of the oracle's host-side drafting functions (oracle/drafting.py) against hand-worked
cases and closed forms, then the library's native versions (svd_ngram_*, svd_spec_adapt_*,
svd_speedup, svd_best_depth) against the oracle.  No GPU."""
import math

import numpy as np
import pytest

from oracle import drafting, formulas
from speculative_decoding_verify_06_gb300 import svd


# ---- pins of the oracle ---------------------------------------------------------------------
def test_ngram_hand_worked_cases():
    # "a b c d e a b c": the key "a b c" last occurred at 0..2, followed by "d e a b c"
    h = [1, 2, 3, 4, 5, 1, 2, 3]
    assert drafting.ngram_propose(h, 3, 4) == [4, 5, 1, 2]
    assert drafting.ngram_propose(h, 3, 9) == [4, 5, 1, 2, 3]   # up to the history's end
    assert drafting.ngram_propose(h, 4, 4) == []                # "5 1 2 3" never seen before
    assert drafting.ngram_propose(h[:3], 3, 4) == []            # the key alone: no earlier copy
    assert drafting.ngram_propose(h[:2], 3, 4) == []            # shorter than the key
    # the latest earlier occurrence wins: "7 8" was followed by 1, later by 2
    assert drafting.ngram_propose([7, 8, 1, 7, 8, 2, 7, 8], 2, 1) == [2]
    # a key overlapping its own continuation (runs of one token)
    assert drafting.ngram_propose([5, 5, 5, 5], 2, 3) == [5]


def test_ngram_periodic_and_distinct_sequences():
    # period P >= key_len: the proposal is the next tokens of the period
    P = 7
    seq = [(i * 3) % P + 10 for i in range(40)]
    for L in (1, 3, 6):
        prop = drafting.ngram_propose(seq, L, 5)
        assert prop == [seq[(40 + i) - P] for i in range(5)]
    # all tokens distinct: never a hit
    assert drafting.ngram_propose(list(range(100)), 1, 3) == []


def test_best_depth_special_cases():
    # free drafts (c = 0) and any acceptance > 0: deeper is always better
    for a in (0.1, 0.5, 0.9):
        assert drafting.best_depth(a, 0.0, 8) == 8
    # nothing accepted: every draft only costs
    assert drafting.best_depth(0.0, 0.1, 8) == 1
    # at alpha = 0.35 and c = 0.05 the table's flat rows pay for two drafts at most
    k = drafting.best_depth(0.35, 0.05, 8)
    assert all(formulas.speedup(0.35, k, 0.05) >= formulas.speedup(0.35, j, 0.05)
               for j in range(1, 9))


def test_spec_adapt_oracle_rules():
    # alpha measured exactly: 3 windows at k = 3 emitting 2 (1 accepted, 1 rejected) -> 1/2
    out = drafting.spec_adapt([([2, 2, 2], 3, None)], k_max=5, draft_cost=0.0,
                              half_life_windows=1e12)
    assert abs(out[0][0] - 0.5) < 1e-9 and out[0][1] == 5
    # all accepted at k = 3 (emit 4): acceptance 1, no rejection counted
    out = drafting.spec_adapt([([4, 4], 3, None)], k_max=5, draft_cost=0.3, half_life_windows=1e12)
    assert out[0][0] == 1.0
    # below the threshold: one draft
    out = drafting.spec_adapt([([1] * 10, 3, None)], k_max=5, draft_cost=0.0)
    assert out[0] == (0.0, 1)
    # nothing measured yet, and skipped windows
    assert drafting.spec_adapt([([], 3, None)], 6, 0.1) == [(None, 6)]
    assert drafting.spec_adapt([([1, 1], 3, [1, 2])], 6, 0.1) == [(None, 6)]


# ---- the library against the oracle -------------------------------------------------------
def test_speedup_and_depth_match_the_oracle():
    for a in np.linspace(0.0, 1.0, 21):
        for k in range(0, 9):
            assert math.isclose(svd.svd_expected_tokens_per_pass(a, k),
                                formulas.expected_tokens_per_pass(a, k), rel_tol=1e-12)
            for c in (0.0, 0.02, 0.1, 0.5):
                assert math.isclose(svd.svd_speedup(a, k, c), formulas.speedup(a, k, c),
                                    rel_tol=1e-12)
        for c in (0.0, 0.02, 0.1, 0.5):
            for kmax in (1, 3, 8):
                assert svd.svd_best_depth(a, c, kmax) == drafting.best_depth(a, c, kmax)
    assert math.isnan(svd.svd_speedup(1.5, 3, 0.1)) and math.isnan(svd.svd_speedup(0.5, 3, -1))
    with pytest.raises(svd.SvdError):
        svd.svd_best_depth(0.5, 0.1, 0)


def test_spec_adapt_matches_the_oracle_on_iid_windows():
    g = np.random.default_rng(5)
    batches = []
    for alpha, k in [(0.9, 5), (0.9, 5), (0.2, 3), (0.2, 3), (0.2, 1), (0.7, 4), (0.7, 4)]:
        acc = g.random((500, k)) < alpha
        ne = np.where(acc.all(1), k + 1, acc.argmin(1) + 1).astype(np.int32)  # first rejection
        st = (g.random(500) < 0.02).astype(np.int32) * 4                      # a few bad windows
        batches.append((ne, k, st))
    ref = drafting.spec_adapt([(list(b[0]), b[1], list(b[2])) for b in batches], k_max=6,
                              draft_cost=0.05, half_life_windows=300)
    a = svd.SpecAdapt(6, 0.05, 0.35, 300)
    assert a.depth == 6 and math.isnan(a.alpha)
    for (ne, k, st), (alpha_ref, depth_ref) in zip(batches, ref):
        a.observe(ne, k, st)
        assert math.isclose(a.alpha, alpha_ref, rel_tol=1e-12) and a.depth == depth_ref
    depths = [d for _, d in ref]
    assert depths[:2] == [6, 6] and depths[4] == 1 and depths[6] > 1  # throttled, then back
    a.close()


def test_ngram_drafter_matches_the_oracle():
    g = np.random.default_rng(11)
    for key_len in (1, 2, 6, 12):
        d = svd.NgramDrafter(key_len)
        hist = []
        # a token stream with planted repeats of earlier spans, appended in uneven pieces
        while len(hist) < 3000:
            if hist and g.random() < 0.4:
                s = int(g.integers(0, len(hist)))
                piece = hist[s:s + int(g.integers(1, 40))]
            else:
                piece = [int(x) for x in g.integers(0, 50, int(g.integers(1, 12)))]
            d.append(np.array(piece, dtype=np.int32))
            hist += piece
            for k in (1, 3, 8):
                assert list(d.propose(k)) == drafting.ngram_propose(hist, key_len, k)
        assert len(d) == len(hist)
        d.close()
    with pytest.raises(svd.SvdError):
        svd.NgramDrafter(0)
