"""Pins of the oracle's sampler: the plain softmax special case, hand-computed examples of each
filter, tie handling and invariants."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from speculative_decoding_verify_06_gb300 import synth


def test_no_filters_is_plain_softmax():
    l = synth.normal_logits(3, 1000, seed=5)
    probs, am, nk, fl = oracle.sampler(l, temperature=1.0, top_p=1.0, min_p=0.0)
    ref = softmax(l.astype(np.float64), axis=1)
    assert np.allclose(probs, ref, rtol=1e-13, atol=0)
    assert np.array_equal(am, np.argmax(l, axis=1))
    assert np.all(nk == 1000)


def test_temperature_only():
    l = synth.normal_logits(2, 300, seed=6)
    probs, *_ = oracle.sampler(l, temperature=0.6, top_p=1.0, min_p=0.0)
    assert np.allclose(probs, softmax(l.astype(np.float64) / 0.6, axis=1), rtol=1e-12)


P5 = np.array([0.5, 0.25, 0.15, 0.07, 0.03])


def _logits_for(p):
    return np.log(p).astype(np.float32)[None, :]


def _expected(keep):
    p = P5 * keep
    return p / p.sum()


def test_min_p_hand_example():
    # max p = 0.5; min_p = 0.2 keeps p >= 0.1: tokens 0, 1, 2
    probs, *_ = oracle.sampler(_logits_for(P5), temperature=1.0, top_p=1.0, min_p=0.2)
    assert np.allclose(probs[0], _expected(np.array([1, 1, 1, 0, 0])), rtol=1e-6)


def test_top_p_hand_example_crossing_token_is_kept():
    # cumulative 0.5, 0.75, 0.90, 0.97, 1.0: top_p 0.8 first reached by token 2 (kept)
    probs, *_ = oracle.sampler(_logits_for(P5), temperature=1.0, top_p=0.8, min_p=0.0)
    assert np.allclose(probs[0], _expected(np.array([1, 1, 1, 0, 0])), rtol=1e-6)
    # top_p 0.6 is reached by token 1
    probs, *_ = oracle.sampler(_logits_for(P5), temperature=1.0, top_p=0.6, min_p=0.0)
    assert np.allclose(probs[0], _expected(np.array([1, 1, 0, 0, 0])), rtol=1e-6)
    # top_p 0.4: the argmax alone
    probs, *_ = oracle.sampler(_logits_for(P5), temperature=1.0, top_p=0.4, min_p=0.0)
    assert np.allclose(probs[0], [1, 0, 0, 0, 0])


def test_filters_intersect_on_the_same_unrenormalised_p():
    # min_p 0.1 alone keeps p >= 0.05 (tokens 0-3); top_p 0.8 alone keeps tokens 0-2
    probs, *_ = oracle.sampler(_logits_for(P5), temperature=1.0, top_p=0.8, min_p=0.1)
    assert np.allclose(probs[0], _expected(np.array([1, 1, 1, 0, 0])), rtol=1e-6)
    # min_p 0.4 keeps p >= 0.2 (tokens 0-1); top_p 0.95 keeps 0-3
    probs, *_ = oracle.sampler(_logits_for(P5), temperature=1.0, top_p=0.95, min_p=0.4)
    assert np.allclose(probs[0], _expected(np.array([1, 1, 0, 0, 0])), rtol=1e-6)


def test_temperature_then_min_p_hand_example():
    # T = 2: p ~ sqrt(P5); ratio to the max is sqrt(p / 0.5)
    probs, *_ = oracle.sampler(_logits_for(P5), temperature=2.0, top_p=1.0, min_p=0.4)
    r = np.sqrt(P5 / 0.5)
    keep = r >= 0.4  # tokens 0..2 (0.3742 < 0.4 for token 3)
    e = np.sqrt(P5) * keep
    assert np.array_equal(keep, [True, True, True, False, False])
    assert np.allclose(probs[0], e / e.sum(), rtol=1e-6)


def test_top_p_ties_keep_lowest_ids():
    p = np.array([0.1, 0.3, 0.3, 0.3])
    probs, *_ = oracle.sampler(np.log(p).astype(np.float32)[None], temperature=1.0, top_p=0.5,
                               min_p=0.0)
    # order: ids 1, 2, 3 (equal p, ascending id), then 0: mass 0.3 < 0.5, 0.6 >= 0.5
    assert np.allclose(probs[0], [0, 0.5, 0.5, 0], rtol=1e-6)


def test_greedy_one_hot_lowest_id_on_ties():
    l = np.array([[0.0, 3.0, 3.0, 1.0]], np.float32)
    probs, am, *_ = oracle.sampler(l, greedy=True)
    assert am[0] == 1 and np.array_equal(probs[0], [0, 1, 0, 0])


def test_invariants_random_rows():
    l = synth.normal_logits(16, 5000, seed=9, std=4.0)
    probs, am, nk, fl = oracle.sampler(l, 0.6, 0.95, 0.05)
    assert np.allclose(probs.sum(1), 1.0, rtol=1e-12)
    for r in range(16):
        assert probs[r, am[r]] > 0
        order = np.lexsort((np.arange(5000), -l[r].astype(np.float64)))
        kept = probs[r, order] > 0
        n = kept.sum()
        assert n == nk[r] and kept[:n].all() and not kept[n:].any()  # a rank prefix
