"""Pins of the closed forms against the values the pages print, and of the Philox generator
against its published known-answer vectors."""
import json
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import formulas

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_expected_tokens_table_reproduces_the_printed_table():
    t = json.load(open(os.path.join(GOLD, "expected_tokens_table.json")))
    for a, row in t["rows"].items():
        for k, printed in zip(t["k"], row):
            v = formulas.expected_tokens_per_pass(float(a), k)
            assert round(v + 1e-12, 2) == pytest.approx(printed, abs=1e-9), (a, k, v)
    assert formulas.expected_tokens_per_pass(0.9, 5) == pytest.approx(4.68559, abs=1e-5)


def test_expected_tokens_limits():
    assert formulas.expected_tokens_per_pass(0.0, 5) == 1.0      # everything rejected: 1 token
    assert formulas.expected_tokens_per_pass(1.0, 5) == 6.0      # everything accepted: k + 1
    # the sum of the geometric series it abbreviates
    for a in (0.2, 0.55, 0.95):
        for k in (1, 4, 7):
            assert formulas.expected_tokens_per_pass(a, k) == pytest.approx(sum(a ** i for i in range(k + 1)))


def test_consistency_check_inversion():
    c = json.load(open(os.path.join(GOLD, "ceilings.json")))["consistency_check"]
    # "at least 1.4 tokens per pass" is 82 / 59 = 1.39 rounded to one decimal
    assert round(c["tok_s"] / c["passes_s"], 1) == c["min_tokens_per_pass"]
    lo = formulas.alpha_from_tokens_per_pass(c["tokens_per_pass"][0], c["k"])
    hi = formulas.alpha_from_tokens_per_pass(c["tokens_per_pass"][1], c["k"])
    assert round(lo, 2) == pytest.approx(c["alpha_printed"][0], abs=0.011)
    assert round(hi, 2) == pytest.approx(c["alpha_printed"][1], abs=0.011)


def test_ceiling_arithmetic():
    for case in json.load(open(os.path.join(GOLD, "ceilings.json")))["cases"]:
        v = formulas.passes_ceiling(case["bandwidth_gb_s"], case["bytes_gb"])
        assert case["printed"] <= v < case["printed"] + 1


def test_speedup_closed_form():
    assert formulas.speedup(0.7, 3, 0.0) == pytest.approx(formulas.expected_tokens_per_pass(0.7, 3))
    assert formulas.speedup(0.0, 4, 0.1) == pytest.approx(1.0 / 1.4)
    assert formulas.speedup(0.8, 5, 0.05) == pytest.approx((1 - 0.8 ** 6) / (0.2 * 1.25))


def test_acceptance_rate_special_cases():
    p = np.array([0.5, 0.5, 0.0])
    assert formulas.acceptance_rate(p, p) == 1.0
    assert formulas.acceptance_rate(p, [0, 0, 1.0]) == 0.0
    assert formulas.greedy_drafter_acceptance(p, [0.1, 0.8, 0.1]) == 0.5


def test_philox_known_answer_vectors():
    kat = json.load(open(os.path.join(GOLD, "philox_kat.json")))
    for c in kat["cases"]:
        out = oracle.philox4x32_10([int(x, 16) for x in c["counter"]], [int(x, 16) for x in c["key"]])
        assert ["%08x" % w for w in out] == c["out"]


def test_uniform_mapping_and_uniformity():
    seed = 0xDEADBEEF12345
    u = np.array([oracle.uniforms(seed, w, i) for w in range(4000) for i in range(5)])
    assert np.all((u >= 0) & (u < 1))
    assert np.all(np.ldexp(u, 24) == np.floor(np.ldexp(u, 24)))  # multiples of 2^-24
    r = oracle.philox4x32_10([7, 0, 3, 0], [seed & 0xFFFFFFFF, seed >> 32])
    assert oracle.uniforms(seed, 7, 3) == ((r[0] >> 8) * 2.0 ** -24, (r[1] >> 8) * 2.0 ** -24)
    for col in range(2):
        assert stats.kstest(u[:, col], "uniform").pvalue > 1e-3
