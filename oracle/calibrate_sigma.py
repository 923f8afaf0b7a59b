"""Calibrates the drafter noise of the lm_head workload with the oracle only.

The workload's drafter logits are the target's logits plus N(0, sigma^2) noise, with sigma chosen
so that the expected acceptance alpha = sum_x min(p'(x), q'(x)) ("Decode is memory-bound ...",
section "Two things the math says to do") is about 0.5 after both distributions pass through the
production sampler (T 0.6, top-p 0.95, min-p 0.05).  Target logits are drawn N(0, s^2) with
s^2 = 5120 * E[scale^2] * E[(code - 8)^2], the variance of one synthetic lm_head output
(scales U(0.005, 0.02), codes uniform 0..15, activations N(0, 1)).

Writes tests/golden/drafter_sigma.json.  Run: python -m oracle.calibrate_sigma
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
from oracle import formulas
from speculative_decoding_verify_06_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(os.path.dirname(HERE), "tests", "golden", "drafter_sigma.json")


def logit_std() -> float:
    a, b = synth.SCALE_LO, synth.SCALE_HI
    e_s2 = (b ** 3 - a ** 3) / (3 * (b - a))
    e_c2 = np.mean((np.arange(16) - 8.0) ** 2)
    return float(np.sqrt(synth.HIDDEN * e_s2 * e_c2))


def mean_alpha(sigma: float, lp: np.ndarray, seed: int) -> float:
    lq = synth.perturb(lp, sigma, seed)
    p, *_ = oracle.sampler(lp, 0.6, 0.95, 0.05)
    q, *_ = oracle.sampler(lq, 0.6, 0.95, 0.05)
    return float(np.mean([formulas.acceptance_rate(p[r], q[r]) for r in range(len(lp))]))


def main(rows: int = 32, target: float = 0.5):
    std = logit_std()
    lp = synth.normal_logits(rows, synth.VOCAB, seed=2024, std=std)
    lo, hi = 0.0, 20.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if mean_alpha(mid, lp, seed=77) > target:
            lo = mid
        else:
            hi = mid
    sigma = 0.5 * (lo + hi)
    res = {"logit_std": std, "sigma": sigma, "alpha": mean_alpha(sigma, lp, seed=77),
           "rows": rows, "target_alpha": target, "sampler": [0.6, 0.95, 0.05],
           "script": "python -m oracle.calibrate_sigma"}
    with open(OUT, "w") as f:
        json.dump(res, f, indent=1)
    print(res)


if __name__ == "__main__":
    main()
