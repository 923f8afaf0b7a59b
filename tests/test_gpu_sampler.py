"""GPU parity of the sampler (svd_sampler_probs) and of lm_head + sampler against the oracle on
identical fp32 logits: argmax exact; the kept set exact wherever the oracle reports no decision
within rounding of a filter boundary; kept probabilities within 1e-5 relative.  Where the oracle
does flag a boundary decision, the two kept sets must still be prefixes of the same (p
descending, id ascending) order and may differ only by tokens inside the flagged band: a top-p
crossing within 1e-5 of top_p, or a probability within relative 1e-6 of min_p * max p."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_06_gb300 import svd, synth
from gpu_helpers import DEV, assert_gemm_parity, lib, native_weight, sampler, to_dev

pytestmark = pytest.mark.gpu

F32 = np.float32


def check_flagged_row(pg, pr, base, flags, top_p, min_p):
    """A row whose decision the oracle flags: the GPU's kept set is a prefix of the oracle's
    order, it differs from the oracle's only by tokens inside the flagged band, and the
    probabilities of the tokens both keep agree after renormalising over them."""
    V = len(base)
    order = np.lexsort((np.arange(V), -base))
    kg, kr = pg[order] > 0, pr[order] > 0
    ng, nr = int(kg.sum()), int(kr.sum())
    assert kg[:ng].all() and kr[:nr].all()
    if ng != nr:
        lo, hi = min(ng, nr), max(ng, nr)
        cum = np.cumsum(base[order])
        # top-p: the GPU's cut lies where the oracle's running mass is within the band
        in_top = bool(flags & 2) and (
            cum[ng - 2] - top_p < 1e-5 if ng > nr else top_p - cum[ng - 1] <= 1e-5)
        # min-p: every token on which the two differ sits at the threshold
        thr = min_p * base.max()
        in_min = bool(flags & 1) and np.all(np.abs(base[order[lo:hi]] - thr) <= 2e-6 * thr)
        assert in_top or in_min, (ng, nr, flags)
    common = (pg > 0) & (pr > 0)
    a = pg[common].astype(np.float64)
    b = pr[common]
    assert np.allclose(a / a.sum(), b / b.sum(), rtol=1e-5, atol=1e-12)


def check(logits, T, top_p, min_p, greedy=False):
    lib()
    smp = svd.Sampler(T, top_p, min_p, greedy)
    pg, amg = sampler(logits, smp)
    pr, amr, nk, fl = oracle.sampler(logits, F32(T), F32(top_p), F32(min_p), greedy)
    assert np.array_equal(amg, amr)
    base = None
    for r in range(len(logits)):
        kept_g, kept_r = pg[r] > 0, pr[r] > 0
        assert kept_g[amr[r]]
        assert abs(pg[r].astype(np.float64).sum() - 1.0) < 1e-5
        if fl[r] == 0:
            assert np.array_equal(kept_g, kept_r), (r, kept_g.sum(), kept_r.sum())
            assert np.allclose(pg[r], pr[r], rtol=1e-5, atol=1e-12)
        else:
            if base is None:  # the unfiltered softmax at T, in the oracle's fp64
                base, *_ = oracle.sampler(logits, F32(T), F32(1.0), F32(0.0))
            check_flagged_row(pg[r], pr[r], base[r], int(fl[r]), float(F32(top_p)),
                              float(F32(min_p)))
    return pg, pr, fl


def test_small_vocabulary_window():
    check(synth.normal_logits(4, 4096, seed=0, std=2.0), 0.6, 0.95, 0.05)


def test_lm_head_sized_rows():
    check(synth.normal_logits(6, synth.VOCAB, seed=1, std=4.389), 0.6, 0.95, 0.05)


def test_plain_softmax_special_case_general_path():
    # min_p = 0 makes every token a survivor: the radix-select path; top_p = 1 keeps all
    pg, pr, _ = check(synth.normal_logits(2, 20000, seed=2, std=1.0), 1.0, 1.0, 0.0)
    assert np.all(pg > 0)


def _survivors(logits, T, min_p):
    """Tokens with exp((l - max) / T) >= min_p, per row (fp64 count; the paths are chosen on it)."""
    l = logits.astype(np.float64)
    return ((l - l.max(axis=1, keepdims=True)) / T >= np.log(min_p)).sum(axis=1)


def test_sorted_survivor_path():
    """33 to 2048 min-p survivors per row: the CTA-wide shared-memory sort of the survivors (up
    to 32 take the one-warp register sort)."""
    logits = synth.normal_logits(3, 20000, seed=34, std=0.8)
    m = _survivors(logits, 0.6, 0.05)
    assert ((m > 32) & (m <= 2048)).all(), m
    check(logits, 0.6, 0.95, 0.05)


def test_min_p_survivors_beyond_the_sort_capacity():
    """More than 2048 survivors with min-p on: the radix select over the whole row, and every
    slice's survivor list overflows, so the renormalisation reads e back."""
    logits = synth.normal_logits(2, synth.VOCAB, seed=32, std=0.5)
    assert (_survivors(logits, 0.6, 0.05) > 8 * 256).all()
    check(logits, 0.6, 0.95, 0.05)


def test_survivors_crowded_into_one_slice():
    """The first eighth of the row (the first CTA's slice) is all survivors and overflows its
    list, while the other slices hold a few: that CTA reads e back, the others write zeros and
    then their kept survivors (kept ones ranked above the crowd, and survivors ranked below
    the top-p crossing)."""
    rng = np.random.default_rng(33)
    V = synth.VOCAB
    logits = rng.normal(0.0, 0.1, size=(2, V)).astype(np.float32)
    logits[:, : V // 8] += 5.0
    for r in range(2):
        idx = rng.choice(np.arange(V // 8, V), size=40, replace=False)
        logits[r, idx[:20]] = (5.6 + 0.05 * rng.standard_normal(20)).astype(np.float32)
        logits[r, idx[20:]] = (4.2 + 0.05 * rng.standard_normal(20)).astype(np.float32)
    assert (_survivors(logits, 0.6, 0.05) > 2048).all()
    pg, pr, fl = check(logits, 0.6, 0.95, 0.05)
    assert (pg[:, V // 8:] > 0).sum() >= 20


def test_cluster_sizes_give_the_same_bits():
    """Up to 8 rows run on clusters of 16 CTAs per row, more rows on clusters of 8: the slices
    differ, the probabilities, argmaxes and kept sets must not (the masses are exact integer sums
    and every element's value is computed alone)."""
    logits = synth.normal_logits(12, synth.VOCAB, seed=43, std=4.389)
    smp = svd.Sampler(0.6, 0.95, 0.05)
    p12, a12 = sampler(logits, smp)
    p4, a4 = sampler(logits[:4], smp)
    assert np.array_equal(a12[:4], a4)
    assert np.array_equal(p12[:4].view(np.uint32), p4.view(np.uint32))


def test_top_p_general_path_radix_select():
    check(synth.normal_logits(3, synth.VOCAB, seed=3, std=1.5), 0.8, 0.9, 0.0)


def test_top_p_general_path_with_heavy_ties():
    g = synth.rng(4)
    logits = g.integers(0, 4, size=(3, 30000)).astype(np.float32)
    check(logits, 1.0, 0.7, 0.0)


def test_flat_distribution_ties_resolved_by_id():
    logits = np.zeros((2, 1000), np.float32)
    pg, pr, _ = check(logits, 0.6, 0.95, 0.05)
    assert (pg[0] > 0).sum() == 950 and np.all(pg[0, :950] > 0)


def test_greedy_one_hot():
    logits = synth.normal_logits(5, 5000, seed=6)
    logits[0, 10] = logits[0, 20] = 50.0
    pg, _, _ = check(logits, 0.6, 0.95, 0.05, greedy=True)
    assert pg[0, 10] == 1.0 and pg[0].sum() == 1.0


def test_hand_example_five_tokens():
    p = np.array([0.5, 0.25, 0.15, 0.07, 0.03])
    logits = np.log(p).astype(np.float32)[None]
    pg, _, _ = check(logits, 1.0, 0.8, 0.0)
    assert np.allclose(pg[0], np.r_[p[:3] / p[:3].sum(), 0, 0], rtol=1e-5)
    pg, _, _ = check(logits, 1.0, 1.0, 0.2)
    assert np.allclose(pg[0], np.r_[p[:3] / p[:3].sum(), 0, 0], rtol=1e-5)


def log_partition(logits, T):
    """log sum_v exp(l_v / T) per row in fp64 (the plain definition, shifted by the max)."""
    z = logits.astype(np.float64) / T
    m = np.max(z, axis=1, keepdims=True)
    return (m[:, 0] + np.log(np.sum(np.exp(z - m), axis=1)))


def _lm_head(hidden, vocab, C, seed, smp, want_lse=True):
    codes, scales = synth.qweight(vocab, hidden, seed=seed)
    W, _ = native_weight(codes, scales)
    H = to_dev(synth.activations(C, hidden, seed=seed + 1))
    logits = torch.empty((C, vocab), dtype=torch.float32, device=DEV)
    probs = torch.empty_like(logits)
    am = torch.empty(C, dtype=torch.int32, device=DEV)
    lse = torch.full((C,), float("nan"), dtype=torch.float32, device=DEV) if want_lse else None
    ws = torch.zeros(svd.svd_lm_head_workspace_bytes(hidden, vocab, C), dtype=torch.uint8, device=DEV)
    svd.svd_lm_head_softmax(W, H, C, smp, logits, probs, am, ws, lse=lse)
    torch.cuda.synchronize()
    return (codes, scales, H, logits.cpu().numpy(), probs.cpu().numpy(), am.cpu().numpy(),
            None if lse is None else lse.cpu().numpy())


@pytest.mark.parametrize("hidden,vocab,C", [(512, 1000, 3), (256, 64, 8), (512, 4133, 5), (1024, 9000, 12)])
def test_lm_head_epilogue_statistics(hidden, vocab, C):
    """Ragged vocabularies (a last block of fewer than 64 rows), C <= 8 through the GEMM
    epilogue's block statistics and C = 12 through the sampler's own max pass: the argmax, the
    distribution and the log-normaliser match the oracle on the GPU's logits, and the logits
    match the GEMM oracle."""
    lib()
    smp = svd.Sampler(0.7, 0.9, 0.02)
    codes, scales, H, lg, pg, am, lse = _lm_head(hidden, vocab, C, seed=vocab + C, smp=smp)
    y_ref, a_ref = oracle.verify_linear(codes, scales, H.view(torch.int16).cpu().numpy().view(np.uint16))
    assert_gemm_parity(lg, y_ref, a_ref)
    pr, amr, nk, fl = oracle.sampler(lg, F32(0.7), F32(0.9), F32(0.02))
    assert np.array_equal(am, amr)
    base, *_ = oracle.sampler(lg, F32(0.7), F32(1.0), F32(0.0))
    for r in range(C):
        if fl[r] == 0:
            assert np.array_equal(pg[r] > 0, pr[r] > 0)
            assert np.allclose(pg[r], pr[r], rtol=1e-5, atol=1e-12)
        else:
            check_flagged_row(pg[r], pr[r], base[r], int(fl[r]), float(F32(0.9)), float(F32(0.02)))
    assert np.allclose(lse, log_partition(lg, 0.7), rtol=0, atol=2e-5)
    # greedy: one-hot of the argmax, lse left untouched
    g = svd.Sampler(greedy=True)
    _, _, _, lg2, pg2, am2, lse2 = _lm_head(hidden, vocab, C, seed=vocab + C, smp=g)
    assert np.array_equal(am2, np.argmax(lg2, axis=1))
    assert np.all(pg2[np.arange(C), am2] == 1.0) and np.all(pg2.sum(axis=1) == 1.0)
    assert np.all(np.isnan(lse2))


def test_lm_head_softmax_matches_oracle():
    lib()
    hidden, vocab, C = synth.HIDDEN, synth.VOCAB, 6
    codes, scales = synth.qweight_torch(vocab, hidden, seed=99, device=DEV)
    cb, sb = svd.svd_native_sizes(hidden, vocab)
    nc = torch.empty(cb, dtype=torch.uint8, device=DEV)
    ns = torch.empty(sb, dtype=torch.uint8, device=DEV)
    svd.svd_repack_weights(svd.QWeight(codes, scales, hidden, vocab, svd.SVD_LAYOUT_CANONICAL), nc, ns)
    W = svd.QWeight(nc, ns, hidden, vocab, svd.SVD_LAYOUT_NATIVE)
    H = synth.activations_torch(C, hidden, seed=5, device=DEV)
    logits = torch.empty((C, vocab), dtype=torch.float32, device=DEV)
    probs = torch.empty_like(logits)
    am = torch.empty(C, dtype=torch.int32, device=DEV)
    ws = torch.zeros(svd.svd_lm_head_workspace_bytes(hidden, vocab, C), dtype=torch.uint8, device=DEV)
    smp = svd.Sampler(0.6, 0.95, 0.05)
    lse = torch.full((C,), float("nan"), dtype=torch.float32, device=DEV)
    svd.svd_lm_head_softmax(W, H, C, smp, logits, probs, am, ws, lse=lse)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    # C <= 8: the GEMM epilogue's block statistics give the max, the argmax and the normaliser
    assert np.allclose(lse.cpu().numpy(), log_partition(lg, 0.6), rtol=0, atol=2e-5)
    rows = np.unique(np.r_[synth.rng(1).choice(vocab, 100, replace=False), 0, vocab - 1,
                           am.cpu().numpy()])
    y_ref, a_ref = oracle.verify_linear(codes[rows].cpu().numpy(),
                                        scales[rows].cpu().numpy().view(np.uint16),
                                        H.view(torch.int16).cpu().numpy().view(np.uint16))
    assert_gemm_parity(lg[:, rows], y_ref, a_ref)
    pr, amr, nk, fl = oracle.sampler(lg, F32(0.6), F32(0.95), F32(0.05))
    pg = probs.cpu().numpy()
    assert np.array_equal(am.cpu().numpy(), amr)
    for r in range(C):
        if fl[r] == 0:
            assert np.array_equal(pg[r] > 0, pr[r] > 0)
            assert np.allclose(pg[r], pr[r], rtol=1e-5, atol=1e-12)


def test_many_rows_bound_the_excused_rows():
    """512 rows of the tiny window's vocabulary: every unflagged row matches the oracle's kept
    set exactly and every flagged row within its band.  The top-p band (1e-5 of the mass) is
    wider than many tokens near the crossing (about 1e-4 each here), so it flags a few percent
    of the rows; the min-p band (relative 1e-6) stays under 1 % of them."""
    _, _, fl = check(synth.normal_logits(512, 4096, seed=9, std=2.0), 0.6, 0.95, 0.05)
    print("sampler rows flagged: top-p", int(((fl & 2) != 0).sum()), "min-p",
          int(((fl & 1) != 0).sum()), "of", len(fl))
    assert ((fl & 1) != 0).sum() <= len(fl) // 100, fl


@pytest.mark.parametrize("V", [1, 3, 7, 9, 17])
def test_vocabularies_smaller_than_the_cluster(V):
    """Rows shorter than the eight slices of a row's cluster: the slices past the row's end
    are empty and must not disturb the max, the masses or the survivors."""
    logits = synth.normal_logits(5, V, seed=V, std=2.0)
    logits[1, 0] = logits[1, V - 1] = 9.0  # a tie at the ends: the lowest id wins
    check(logits, 0.6, 0.95, 0.05)
    check(logits, 1.0, 0.5, 0.0)
    check(logits, 0.6, 0.95, 0.05, greedy=True)


def test_thirty_two_rows_one_call():
    """The largest window the ABI takes in one call (SVD_C_MAX rows), one cluster per row."""
    check(synth.normal_logits(32, 20000, seed=77, std=3.0), 0.6, 0.95, 0.05)


@pytest.mark.parametrize("vocab", [1, 5, 63, 64, 65, 129])
@pytest.mark.parametrize("C", [1, 8])
def test_lm_head_epilogue_tiny_vocabularies(vocab, C):
    """Vocabularies of one partial block, exactly one block, one block and a row: the epilogue's
    padding rows take no part in the max, the argmax or the normaliser."""
    lib()
    smp = svd.Sampler(0.6, 0.95, 0.05)
    codes, scales, H, lg, pg, am, lse = _lm_head(256, vocab, C, seed=vocab * 7 + C, smp=smp)
    pr, amr, nk, fl = oracle.sampler(lg, F32(0.6), F32(0.95), F32(0.05))
    assert np.array_equal(am, amr)
    assert np.all(am >= 0) and np.all(am < vocab)
    assert np.allclose(lse, log_partition(lg, 0.6), rtol=0, atol=2e-5)
    for r in range(C):
        if fl[r] == 0:
            assert np.array_equal(pg[r] > 0, pr[r] > 0)
            assert np.allclose(pg[r], pr[r], rtol=1e-5, atol=1e-12)
