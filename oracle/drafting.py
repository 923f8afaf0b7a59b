"""Host-side drafting and depth policy, written out plainly (slow, obviously correct).

TEST INFRASTRUCTURE (part of the oracle).  Each function cites its passage; pinned by
``tests/test_oracle_drafting.py``.
"""
from __future__ import annotations

from . import formulas


def ngram_propose(history, key_len: int, k_max: int):
    """The n-gram overlay's proposal for the next tokens.

    "100 tokens per second ..." (curriculo.me), section "Lever 3: an n-gram overlay for
    repetition": a map from k-token keys to whatever continuation followed them last time, over
    the prompt and everything generated; when the most recent tokens hit the map, the stored
    continuation is proposed.  Written as a search: the key is the last ``key_len`` tokens; find
    the latest earlier position p (key_len <= p < len) whose preceding ``key_len`` tokens equal
    the key; propose history[p : p + k_max] (what followed it, up to the end of the history).
    No earlier occurrence, or a history shorter than the key: no proposal.
    """
    h = list(history)
    n = len(h)
    if n < key_len or k_max <= 0:
        return []
    key = h[n - key_len:]
    for p in range(n - 1, key_len - 1, -1):  # p = n would be the key itself
        if h[p - key_len:p] == key:
            return h[p:p + k_max]
    return []


def best_depth(alpha: float, draft_cost: float, k_max: int) -> int:
    """The depth in 1..k_max with the largest speedup (the shallower one on ties).

    "Decode is memory-bound ..." (trefon.com), section "Speculative decoding": the speedup
    counts the drafter's cost, (1 - a^(k+1)) / ((1 - a)(k c + 1)).
    """
    best, sb = 1, formulas.speedup(alpha, 1, draft_cost)
    for k in range(2, k_max + 1):
        s = formulas.speedup(alpha, k, draft_cost)
        if s > sb:
            best, sb = k, s
    return best


def spec_adapt(batches, k_max: int, draft_cost: float, threshold: float = 0.35,
               half_life_windows: float = 256.0):
    """Depth chosen after each batch of verified windows.

    "Decode is memory-bound ...", section "Two things the math says to do": throttle the draft
    depth when the measured acceptance falls below 35 %.  Reading: acceptance is measured as
    accepted drafts / accept tests over recent windows (each weight halved after
    ``half_life_windows`` later windows); a window that emitted n tokens at depth k accepted
    n - 1 drafts and rejected one if n - 1 < k; windows with a non-zero status are skipped.
    Below the threshold the depth drops to one draft; otherwise it is the best depth for the
    measured acceptance.  ``batches`` is a list of (n_emitted list, k, status list or None);
    returns [(alpha or None, depth)] after each batch.
    """
    decay = 0.5 ** (1.0 / half_life_windows)
    acc = tests = 0.0
    out = []
    for n_emitted, k, status in batches:
        for w, ne in enumerate(n_emitted):
            if status is not None and status[w] != 0:
                continue
            if ne < 1 or ne > k + 1:
                continue
            j = ne - 1
            acc = acc * decay + j
            tests = tests * decay + j + (1 if j < k else 0)
        if tests <= 0.0:
            out.append((None, k_max))
            continue
        a = acc / tests
        out.append((a, 1 if a < threshold else best_depth(a, draft_cost, k_max)))
    return out
