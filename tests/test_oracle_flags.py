"""Pins of the oracle's boundary flags, which decide which outputs the GPU parity tests may excuse.

The sampler flags a row (bit 0) when some probability lies within a relative 1e-6 of the min-p
threshold min_p * max p, and (bit 1) when the top-p crossing leaves the cumulative mass, before or
after the crossing token, within 1e-5 of top_p ("Decode is memory-bound ...", "Two things the math
says to do": T 0.6, top-p 0.95, min-p 0.05).  The acceptance reports, for every window with a
draw, the distance (margin) of the resampling uniform u' to the nearer edge of the emitted token's
interval [C_{v-1}/R, C_v/R), and flags it (near) when that distance is below 1e-6.  The rows and
draws below are built so that the expected flags, kept sets, tokens and margins follow from exact
arithmetic by hand: exact binary fractions for the draws, logits whose ratios sit a known
distance from the thresholds for the sampler."""
import math

import numpy as np

import oracle

F32 = np.float32


def _row(ratios):
    """fp32 logits whose softmax at T = 1 has the given ratios to the first entry."""
    return np.array([math.log(r) for r in ratios], dtype=F32)


def _ratio_in_f64(logits, v, ref=0):
    return math.exp(float(logits[v]) - float(logits[ref]))


def test_min_p_flag_set_exactly_at_the_threshold():
    # token 1 sits at min_p * max p (up to the fp32 rounding of its logit, ~3e-7 relative)
    lg = _row([1.0, 0.05, 0.3, 0.01])
    rel = abs(_ratio_in_f64(lg, 1) - 0.05) / 0.05
    assert rel < 5e-7  # the premise: inside the 1e-6 band
    _, _, _, fl = oracle.sampler(lg[None, :], F32(1.0), F32(1.0), F32(0.05))
    assert fl[0] & 1 == 1


def test_min_p_flag_clear_outside_the_band():
    for ratio, kept in ((0.05 * (1 + 1e-4), True), (0.05 * (1 - 1e-4), False)):
        lg = _row([1.0, ratio, 0.3, 0.01])
        p, _, nk, fl = oracle.sampler(lg[None, :], F32(1.0), F32(1.0), F32(0.05))
        assert fl[0] & 1 == 0
        assert (p[0, 1] > 0) == kept
        assert p[0, 3] == 0.0  # 0.01 < 0.05: dropped
        assert nk[0] == (3 if kept else 2)


def test_min_p_flag_needs_min_p():
    # min_p = 0 disables the filter, and with it the flag, even for a tiny probability
    lg = _row([1.0, 1e-12, 0.5])
    _, _, nk, fl = oracle.sampler(lg[None, :], F32(1.0), F32(1.0), F32(0.0))
    assert fl[0] == 0 and nk[0] == 3


def test_top_p_flag_when_the_crossing_lands_on_top_p():
    # sorted mass 0.5, 0.45, 0.05: the cumulative mass reaches 0.95 exactly at the second token
    lg = _row([0.5 / 0.5, 0.45 / 0.5, 0.05 / 0.5])
    _, _, _, fl = oracle.sampler(lg[None, :], F32(1.0), F32(0.95), F32(0.0))
    assert fl[0] & 2 == 2
    assert fl[0] & 1 == 0


def test_top_p_flag_when_the_mass_before_the_crossing_is_at_top_p():
    # 0.949995 before the second token, 1 - 0.949995 in the other two: |before - 0.95| = 5e-6
    a = 0.949995
    lg = _row([1.0, 0.04 / a, (1 - a - 0.04) / a])
    p, _, nk, fl = oracle.sampler(lg[None, :], F32(1.0), F32(0.95), F32(0.0))
    assert fl[0] & 2 == 2
    assert nk[0] == 2  # the crossing token (the second) is kept


def test_top_p_flag_clear_far_from_the_crossing():
    cases = (([0.6, 0.3, 0.1], 3),            # 0.9 before, 1.0 after: both 0.05 away
             ([0.95 + 2e-5, 0.03, 0.02 - 2e-5], 1))  # crosses at the first token, 2e-5 above
    for masses, kept in cases:
        lg = _row([m / masses[0] for m in masses])
        p, _, nk, fl = oracle.sampler(lg[None, :], F32(1.0), F32(0.95), F32(0.0))
        assert fl[0] == 0, masses
        assert nk[0] == kept, masses
        assert abs(p[0].sum() - 1.0) < 1e-12


def _draw(p_rows, q_rows, draft, u2, u=0.5):
    """One window with k = len(draft) drafts and the given uniforms (u for the accept tests,
    u2 for every position's draw), through the oracle's uniforms hook."""
    k = len(draft)
    un = np.zeros((1, k + 1, 2), F32)
    un[0, :, 0] = u
    un[0, :, 1] = u2
    return oracle.accept(np.array(p_rows, F32), np.array([draft], np.int32),
                         q=None if q_rows is None else np.array(q_rows, F32), uniforms=un,
                         return_margin=True)


# Residual after rejecting token 3 (q puts all its mass there, p none): (p - q)+ = p =
# (0.25, 0.25, 0.5, 0), R = 1, interval edges 0.25, 0.5, 1.0.
P_REJ = [[0.25, 0.25, 0.5, 0.0], [0.1, 0.2, 0.3, 0.4]]
Q_REJ = [[0.0, 0.0, 0.0, 1.0]]
E24 = 2.0 ** -24


def test_margin_and_near_on_a_rejection_draw():
    cases = (  # u', emitted token, exact margin
        (0.5 + E24, 2, E24), (0.5 - E24, 1, E24), (0.75, 2, 0.25), (0.125, 0, 0.125),
        (0.25, 1, 0.0), (1.0 - E24, 2, E24),
    )
    for u2, tok, m in cases:
        t, ne, st, near, margin = _draw(P_REJ, Q_REJ, [3], u2)
        assert st[0] == 0 and ne[0] == 1 and t[0, 0] == tok, (u2, t[0])
        assert margin[0] == m, (u2, margin[0], m)
        assert near[0] == (1 if m < 1e-6 else 0)


def test_near_switches_at_one_millionth():
    # 16 * 2^-24 = 9.54e-7 < 1e-6 <= 17 * 2^-24 = 1.013e-6
    for steps, flagged in ((16, 1), (17, 0)):
        _, _, _, near, margin = _draw(P_REJ, Q_REJ, [3], 0.5 + steps * E24)
        assert margin[0] == steps * E24 and near[0] == flagged


def test_margin_on_the_capping_draw_after_all_accepted():
    # the draft (token 0, q = p) is accepted whatever u < 1; the capping draw uses p_1 =
    # (0.1, 0.2, 0.3, 0.4): edges 0.1, 0.3, 0.6, 1.0 (as fp32 sums of fp32 masses)
    p = [[1.0, 0.0, 0.0, 0.0], [0.1, 0.2, 0.3, 0.4]]
    q = [[1.0, 0.0, 0.0, 0.0]]
    e = np.cumsum(np.array(p[1], F32).astype(np.float64))
    for u2 in (0.35, 0.9, 0.05):
        u2 = round(u2 * 2 ** 24) * E24  # uniforms are multiples of 2^-24
        t, ne, st, near, margin = _draw(p, q, [0], u2)
        v = int(np.searchsorted(e, u2 * e[-1], side="right"))
        lo = e[v - 1] / e[-1] if v > 0 else 0.0
        assert ne[0] == 2 and t[0, 0] == 0 and t[0, 1] == v
        assert abs(margin[0] - min(u2 - lo, e[v] / e[-1] - u2)) < 1e-15
        assert near[0] == 0


def test_no_draw_no_margin():
    # greedy windows draw nothing: margin +inf, never near
    p = np.array([[0.1, 0.7, 0.2], [0.3, 0.3, 0.4]], F32)
    t, ne, st, near, margin = oracle.accept(p, np.array([[1]], np.int32), return_margin=True)
    assert np.isinf(margin[0]) and near[0] == 0 and ne[0] == 2 and t[0, 1] == 2


def test_margin_is_in_units_of_the_uniform_when_the_residual_mass_is_not_one():
    # (p - q)+ = (0, 0.25, 0.25, 0): R = 0.5, edges at u' = 0.5 and 1.0; rejecting token 3
    # (q 0.5 > p 0)
    p = [[0.25, 0.25, 0.5, 0.0], [0.25, 0.25, 0.25, 0.25]]
    q = [[0.25, 0.0, 0.25, 0.5]]
    for u2, tok, m in ((0.5 + E24, 2, E24), (0.5 - 3 * E24, 1, 3 * E24), (0.125, 1, 0.125)):
        t, ne, st, near, margin = _draw(p, q, [3], u2)
        assert st[0] == 0 and ne[0] == 1 and t[0, 0] == tok, (u2, t[0])
        assert margin[0] == m, (u2, margin[0])
