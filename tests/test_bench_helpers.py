"""Host-side helpers of bench.py, run on CPU tensors: the per-pair bisection that gives every
(p, q) pair of the acceptance pools its target overlap sum min(p, q), and the two oracle
timings reported beside the KV-read and acceptance sections and the whole-pass oracle timing of
the main line (they must return a positive rate with the thread count they used)."""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verify_06_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("alpha", [0.35, 0.6, 0.9])
def test_accept_pool_pairs_have_the_target_overlap(alpha):
    g = torch.Generator()
    g.manual_seed(3)
    P, Q = bench.accept_pool(torch.device("cpu"), 3000, 6, alpha, g)
    assert torch.allclose(P.sum(1), torch.ones(6), atol=1e-5)
    assert torch.allclose(Q.sum(1), torch.ones(6), atol=1e-5)
    overlap = torch.minimum(P, Q).sum(1)
    assert torch.all((overlap - alpha).abs() <= 1e-4), overlap


def test_kv_oracle_sample_reports_a_rate():
    C, n_past = 4, 124
    kc, ks, vc, vs = synth.kv_cache_torch(8, n_past + C, synth.HEAD_DIM, 1, torch.device("cpu"))
    q = torch.randn((C, synth.N_Q_HEADS, synth.HEAD_DIM)).to(torch.bfloat16)
    r = bench.kv_oracle_sample(q, kc, ks, vc, vs, n_past, C)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0 and r["cores"] >= 1


def test_accept_oracle_sample_reports_a_rate():
    g = torch.Generator()
    g.manual_seed(5)
    P, Q = bench.accept_pool(torch.device("cpu"), 500, 4, 0.6, g)
    samples = torch.multinomial(Q, 64, replacement=True, generator=g)
    r = bench.accept_oracle_sample(P, Q, samples, 4, 50, g, torch.device("cpu"))
    assert r["kind"] == "oracle" and r["unit"] == "windows/s" and r["value"] > 0
    assert np.isfinite(r["seconds"]) and r["cores"] >= 1


def test_pass_oracle_sample_scales_a_one_layer_step():
    smp = bench.OracleSample(layers=1)
    dt = smp.step()
    assert dt > 0 and smp.fraction == 1 / 64
    assert smp.passes_per_s([dt]) == pytest.approx(1 / (64 * dt))
    assert "1 of the 64 layers" in smp.describe(1) and smp.threads >= 1
