"""Closed forms the pages state, written out in double precision.

TEST INFRASTRUCTURE (part of the oracle).  Each function cites its passage.
"""
from __future__ import annotations

import numpy as np


def expected_tokens_per_pass(alpha: float, k: int) -> float:
    """E[tokens per pass] = (1 - alpha^(k+1)) / (1 - alpha) for i.i.d. acceptance.

    "Decode is memory-bound ..." (trefon.com), section "Speculative decoding", the
    E[tokens per pass] formula (attributed there to Leviathan et al., 2023).  At alpha = 1
    every draft is accepted and the pass yields k + 1 tokens (the limit of the formula).
    """
    if alpha == 1.0:
        return float(k + 1)
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


def alpha_from_tokens_per_pass(tokens: float, k: int) -> float:
    """Invert E[tokens per pass] in alpha by bisection (it is increasing in alpha on [0, 1]).

    Used for the consistency check in "Decode is memory-bound ...", section "A consistency
    check on my own numbers" (1.8 - 2 tokens per pass at three drafts).
    """
    lo, hi = 0.0, 1.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if expected_tokens_per_pass(mid, k) < tokens:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def speedup(alpha: float, k: int, c: float) -> float:
    """speedup = (1 - alpha^(k+1)) / ((1 - alpha) * (k*c + 1)), c = one draft step's cost
    relative to a target pass.  "Decode is memory-bound ...", section "Speculative decoding".
    """
    return expected_tokens_per_pass(alpha, k) / (k * c + 1.0)


def acceptance_rate(p, q) -> float:
    """Expected acceptance alpha = sum_x min(p(x), q(x)).

    "Decode is memory-bound ...", section "Two things the math says to do".
    """
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    return float(np.minimum(p, q).sum())


def greedy_drafter_acceptance(p, q) -> float:
    """A greedy drafter puts all its mass on argmax q, so alpha = p(argmax q).

    "Decode is memory-bound ...", section "Two things the math says to do".
    """
    q = np.asarray(q)
    return float(np.asarray(p, dtype=np.float64)[int(np.argmax(q))])


def passes_ceiling(bandwidth_gb_s: float, bytes_per_pass_gb: float) -> float:
    """The bandwidth ceiling: passes (or tokens) per second <= bandwidth / bytes per pass.

    "100 tokens per second ..." (curriculo.me), section "The wall"; "Decode is memory-bound
    ...", section "The ceiling".
    """
    return bandwidth_gb_s / bytes_per_pass_gb
