"""Pins for the oracle's log-probabilities, decision margins and the race's
partial last block.

* Log-probabilities (inclusionAI/AReno PR #550, "What does this PR do?",
  Phase 2: the reported logprobs are those of the sampler's own
  distribution).  Under sampling the reported value is ln p_j(token) of the
  filtered, tempered distribution: a hand-worked top-k + top-p case at
  T = 0.7, the unfiltered T = 1 case against scipy's log_softmax, and random
  filter mixes against ln of the pinned distribution.
* Margins (the verify method's exactness bar exempts decisions whose margin
  is below 1e-6).  Accept tests and draws are built so that the decisive
  quantity sits at a chosen multiple of the margin: half of it must flag,
  twice it must not.  Draws are checked at both levels of the race.
* The race's last block may be partial (V not a multiple of 256): the
  winner law must still be r / sum(r) with weight in that block.
"""
import numpy as np
import pytest
from scipy import stats
from scipy.special import log_softmax

from oracle import philox
from oracle import verify as ov


# ---------------------------------------------------------------------------
# Log-probabilities
# ---------------------------------------------------------------------------
def test_sampling_logprob_hand_worked_topk_topp():
    # probabilities 0.4, 0.3, 0.2, 0.1 at T = 1; at T = 0.7 the weights are
    # prob^(1/0.7); top-k 3 keeps the first three; renormalised they are
    # 0.4915, 0.3259, 0.1826, so top-p 0.8 keeps two (0.4915 < 0.8 <= 0.8174).
    probs = np.array([0.4, 0.3, 0.2, 0.1])
    l = np.log(probs)
    T, K, P = 0.7, 3, 0.8
    w = probs[:2] ** (1.0 / T)
    p_kept = w / w.sum()
    t = ov.target_distribution(l, T, K, P)
    for tok in (0, 1):
        np.testing.assert_allclose(ov.token_logprob(l, t, tok, T), np.log(p_kept[tok]), rtol=1e-13)
    # both plausible mistakes give other numbers
    lp1 = ov.token_logprob(l, t, 1, T)
    assert abs(lp1 - np.log(probs[1] / probs[:2].sum())) > 1e-3          # temperature dropped
    w_all = probs ** (1.0 / T)
    assert abs(lp1 - np.log(w_all[1] / w_all.sum())) > 1e-3              # normaliser over everything


def test_sampling_logprob_unfiltered_is_log_softmax():
    rng = np.random.default_rng(21)
    l = rng.normal(0, 3, 4000)
    t = ov.target_distribution(l, 1.0, 0, 1.0)
    ref = log_softmax(l)
    for tok in rng.integers(0, 4000, size=50):
        np.testing.assert_allclose(ov.token_logprob(l, t, int(tok), 1.0), ref[tok], rtol=1e-12, atol=1e-12)
    # at another temperature: log_softmax of l / T
    t = ov.target_distribution(l, 1.7, 0, 1.0)
    ref = log_softmax(l / 1.7)
    for tok in rng.integers(0, 4000, size=50):
        np.testing.assert_allclose(ov.token_logprob(l, t, int(tok), 1.7), ref[tok], rtol=1e-12, atol=1e-12)


def test_sampling_logprob_is_log_p_on_random_filters():
    rng = np.random.default_rng(22)
    for _ in range(60):
        V = int(rng.integers(2, 400))
        l = np.round(rng.normal(0, 2, V), 1)          # ties
        T = float(rng.choice([0.3, 0.7, 1.0, 2.0]))
        K = int(rng.integers(0, V + 1))
        P = float(rng.choice([1.0, 0.5, 0.9, 0.97]))
        t = ov.target_distribution(l, T, K, P)
        for tok in t.kept[:20]:
            np.testing.assert_allclose(ov.token_logprob(l, t, int(tok), T), np.log(t.p[tok]),
                                       rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# Accept margin
# ---------------------------------------------------------------------------
def _accept_case(delta, seed=5, row=3):
    """V = 2, k = 1, T = 1, no filter: draft 0 with q = 0.5 and p(0) = u q + delta."""
    u = philox.accept_uniform(seed, row, 0)
    p0 = u * 0.5 + delta
    l = np.zeros((2, 2))
    l[0, 1] = np.log(1.0 / p0 - 1.0)          # softmax([0, l1])[0] = p0
    q = np.array([[0.5, 0.5]])
    return ov.verify_row(l, q, np.array([0]), 1.0, 0, 1.0, seed, row)


@pytest.mark.parametrize("frac,flag", [(0.5, True), (-0.5, True), (2.0, False), (-2.0, False)])
def test_accept_margin_flags_inside_and_not_outside(frac, flag):
    r = _accept_case(frac * ov.MARGIN)
    assert bool(r.flags & ov.F_MARGIN_ACCEPT) == flag
    assert r.margin_accept == [flag]
    # the decision itself follows the sign of u q - p
    assert r.accept == [frac > 0]


def test_accept_margin_not_flagged_when_p_is_exactly_one_or_zero():
    rng = np.random.default_rng(3)
    l = rng.normal(0, 1, size=(2, 50))
    q = rng.dirichlet(np.ones(50), size=1)
    am = int(np.argmax(l[0]))
    # top-k 1: p(argmax) = 1 exactly; any other draft has p = 0 exactly
    for x in (am, (am + 1) % 50):
        r = ov.verify_row(l, q, np.array([x]), 1.0, 1, 1.0, seed=1, row=0)
        assert r.margin_accept == [False]


# ---------------------------------------------------------------------------
# Draw margins, level 2 (one block) and level 1 (two blocks)
# ---------------------------------------------------------------------------
def _ratio(frac):
    """s_a / s_b such that s_a - s_b = frac * MARGIN * (s_a + s_b)."""
    m = frac * ov.MARGIN
    return (1.0 + m) / (1.0 - m)


@pytest.mark.parametrize("frac,flag", [(0.5, True), (2.0, False)])
def test_draw_margin_within_a_block(frac, flag):
    seed, row, pos = 9, 2, 1
    a, b = 3, 10                                   # both in block 0
    E = philox.race_exponentials(seed, row, pos, np.array([a, b]))
    r = np.zeros(256)
    r[b] = 0.25
    r[a] = _ratio(frac) * (r[b] / E[1]) * E[0]     # s_a = ratio * s_b
    y, margin = ov.exponential_race(r, seed, row, pos, unc=r)
    assert y == a and margin == flag


@pytest.mark.parametrize("frac,flag", [(0.5, True), (2.0, False)])
def test_draw_margin_between_blocks(frac, flag):
    seed, row, pos = 4, 7, 0
    a, b = 5, 300                                  # blocks 0 and 1, one entry each
    Eb = philox.race_exponentials(seed, row, pos, np.array([0, 1]), stream=philox.STREAM_BLOCK)
    r = np.zeros(600)
    r[b] = 0.4
    r[a] = _ratio(frac) * (r[b] / Eb[1]) * Eb[0]
    y, margin = ov.exponential_race(r, seed, row, pos, unc=r)
    assert y == a and margin == flag


@pytest.mark.parametrize("frac,flag", [(0.5, True), (2.0, False)])
def test_draw_margin_reaches_the_row_flags(frac, flag):
    # A bonus draw (k = 0, T = 1) over two live entries of one block: p is
    # softmax of the two logits, the margin weights are p itself.
    seed, row = 12, 1
    a, b = 1, 6
    E = philox.race_exponentials(seed, row, 0, np.array([a, b]))
    ratio = _ratio(frac) * E[0] / E[1]             # p_a / p_b
    l = np.full((1, 8), -np.inf)
    l[0, b] = 0.0
    l[0, a] = np.log(ratio)
    r = ov.verify_row(l, np.zeros((0, 8)), np.zeros(0, np.int32), 1.0, 0, 1.0, seed, row)
    assert r.tokens[0] == a
    assert bool(r.flags & ov.F_MARGIN_DRAW) == flag and r.draw_margin == flag


# ---------------------------------------------------------------------------
# Two-level race with a partial last block
# ---------------------------------------------------------------------------
def test_two_level_race_partial_last_block_40k():
    # V = 700: blocks of 256, 256 and 188 entries; half the weight in the
    # partial block, including its very last entry.
    idx = np.array([10, 300, 512, 600, 650, 699])
    w = np.array([0.2, 0.15, 0.15, 0.1, 0.15, 0.25])
    r = np.zeros(700)
    r[idx] = w
    got = np.array([ov.exponential_race(r, seed=s, row=s % 3, pos=s % 5, unc=r)[0]
                    for s in range(40000)])
    counts = np.array([np.count_nonzero(got == i) for i in idx], dtype=float)
    assert counts.sum() == 40000
    tv = 0.5 * np.abs(counts / 40000 - w).sum()
    pv = stats.chisquare(counts, w * 40000).pvalue
    assert tv <= 0.015 and pv > 1e-3, (tv, pv)


# ---------------------------------------------------------------------------
# row_base: a batch split into row blocks reproduces the whole batch
# ---------------------------------------------------------------------------
def test_row_base_split_equals_whole_batch():
    rng = np.random.default_rng(8)
    B, k, V = 6, 2, 40
    logits = rng.normal(0, 1.5, size=(B, k + 1, V))
    q = rng.dirichlet(np.ones(V), size=(B, k))
    drafts = rng.integers(0, V, size=(B, k)).astype(np.int32)
    T = np.full(B, 1.0)
    K = np.zeros(B, np.int32)
    P = np.ones(B)
    whole = ov.verify(logits, q, drafts, T, K, P, seed=77)
    lo = ov.verify(logits[:4], q[:4], drafts[:4], T[:4], K[:4], P[:4], seed=77, row_base=0)
    hi = ov.verify(logits[4:], q[4:], drafts[4:], T[4:], K[4:], P[4:], seed=77, row_base=4)
    for key in ("tokens", "accept_len", "logprobs", "alpha", "flags"):
        np.testing.assert_array_equal(np.concatenate([lo[key], hi[key]]), whole[key])
    # without the base the second block would draw other numbers
    wrong = ov.verify(logits[4:], q[4:], drafts[4:], T[4:], K[4:], P[4:], seed=77)
    assert not (np.array_equal(wrong["tokens"], hi["tokens"])
                and np.array_equal(wrong["accept_len"], hi["accept_len"]))
