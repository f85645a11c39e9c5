"""Pins for the oracle's sampler-equivalent target distribution.

Each case is worked by hand or reduces to a library routine (scipy softmax /
log_softmax, numpy argmax), so a dropped term, a wrong filter order or a wrong
tie rule fails one of them.
"""
import numpy as np
import pytest
from scipy.special import log_softmax, softmax

from oracle import verify as ov


def test_temperature_one_no_filter_is_softmax():
    rng = np.random.default_rng(1)
    l = rng.normal(0, 3, 5000)
    t = ov.target_distribution(l, 1.0, 0, 1.0)
    np.testing.assert_allclose(t.p, softmax(l), rtol=1e-12, atol=0)
    assert len(t.kept) == 5000


def test_temperature_scales_logits():
    rng = np.random.default_rng(2)
    l = rng.normal(0, 3, 777)
    t = ov.target_distribution(l, 0.7, 0, 1.0)
    np.testing.assert_allclose(t.p, softmax(l / 0.7), rtol=1e-12, atol=1e-300)


def test_greedy_is_first_argmax_and_logprob_is_log_softmax():
    l = np.array([0.5, 2.0, -1.0, 2.0, 1.0])
    t = ov.target_distribution(l, 0.0, 0, 1.0)
    assert np.argmax(t.p) == 1 == np.argmax(l)      # np.argmax: first occurrence
    assert t.p.sum() == 1.0 and t.p[1] == 1.0
    lp = ov.token_logprob(l, t, 3, 0.0)
    np.testing.assert_allclose(lp, log_softmax(l)[3], rtol=1e-14)


def test_total_order_breaks_ties_by_index_and_signed_zero_ties():
    l = np.array([1.0, 3.0, 2.0, 3.0, 0.0, -0.0])
    assert list(ov.total_order(l)) == [1, 3, 2, 0, 4, 5]


def test_topk_keeps_exactly_k_with_index_tiebreak():
    l = np.array([1.0, 3.0, 2.0, 3.0, 0.0])
    t2 = ov.target_distribution(l, 1.0, 2, 1.0)
    np.testing.assert_allclose(t2.p, [0, 0.5, 0, 0.5, 0], atol=1e-15)
    t1 = ov.target_distribution(l, 1.0, 1, 1.0)
    assert t1.p[1] == 1.0 and t1.p.sum() == 1.0
    t3 = ov.target_distribution(l, 1.0, 3, 1.0)
    e = np.exp(np.array([3.0, 3.0, 2.0]) - 3.0)
    np.testing.assert_allclose(t3.p[[1, 3, 2]], e / e.sum(), rtol=1e-15)
    # K >= V and K <= 0 disable the filter
    for K in (0, -3, 5, 9):
        np.testing.assert_allclose(ov.target_distribution(l, 1.0, K, 1.0).p, softmax(l), rtol=1e-14)


def test_topp_keeps_crossing_entry():
    probs = np.array([0.5, 0.3, 0.15, 0.05])
    l = np.log(probs)
    t = ov.target_distribution(l, 1.0, 0, 0.75)       # cum 0.5, 0.8 -> keep 2
    np.testing.assert_allclose(t.p, [0.625, 0.375, 0, 0], rtol=1e-13)
    t = ov.target_distribution(l, 1.0, 0, 0.85)       # cum 0.5, 0.8, 0.95 -> keep 3
    np.testing.assert_allclose(t.p, [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0], rtol=1e-13)
    t = ov.target_distribution(l, 1.0, 0, 0.4)        # the top entry alone crosses
    assert t.p[0] == 1.0
    assert not t.topp_margin


def test_topk_applies_before_topp():
    # Renormalising over the top 3 first gives cum 4/9, 7/9 -> {0, 1} at P = 0.72;
    # top-p on the unfiltered distribution would keep {0, 1, 2} (cum 0.4, 0.7, 0.9).
    l = np.log(np.array([0.4, 0.3, 0.2, 0.1]))
    t = ov.target_distribution(l, 1.0, 3, 0.72)
    np.testing.assert_allclose(t.p, [4 / 7, 3 / 7, 0, 0], rtol=1e-13)


def test_temperature_applies_before_topp():
    # T = 2 flattens p to ~[0.41, 0.32, 0.26]: P = 0.45 keeps two entries.
    # Applying top-p to the T = 1 distribution would keep only the first.
    l = np.log(np.array([0.5, 0.3, 0.2]))
    t = ov.target_distribution(l, 2.0, 0, 0.45)
    e = np.sqrt(np.array([0.5, 0.3]))
    np.testing.assert_allclose(t.p[:2], e / e.sum(), rtol=1e-13)
    assert t.p[2] == 0


def test_topp_ties_cut_by_index():
    l = np.array([0.0, 2.0, 2.0, 2.0])
    t = ov.target_distribution(l, 1.0, 0, 0.5)   # three equal entries, need 2 of them
    np.testing.assert_allclose(t.p, [0, 0.5, 0.5, 0], rtol=1e-15)


def test_topp_margin_flag():
    l = np.log(np.array([0.5, 0.3, 0.2]))
    t = ov.target_distribution(l, 1.0, 0, 0.8)    # cum at crossing is 0.8 up to rounding
    assert t.topp_margin


def test_distribution_invariants_random():
    rng = np.random.default_rng(3)
    for _ in range(50):
        V = int(rng.integers(1, 300))
        l = np.round(rng.normal(0, 2, V), 1)       # coarse values -> many ties
        T = float(rng.choice([0.0, 0.3, 1.0, 2.5]))
        K = int(rng.integers(-1, V + 2))
        P = float(rng.choice([1.0, 0.5, 0.9, 0.99]))
        t = ov.target_distribution(l, T, K, P)
        assert abs(t.p.sum() - 1) < 1e-12 and np.all(t.p >= 0)
        order = ov.total_order(l)
        n = np.count_nonzero(t.p)
        # support is a prefix of the total order
        assert set(np.nonzero(t.p)[0]) == set(order[:n])
        if 0 < K < V and T > 0:
            assert n <= K


def test_params_validation():
    assert ov.params_valid(0.0, 1.0)
    assert ov.params_valid(0.7, 0.9)
    assert not ov.params_valid(-1.0, 1.0)
    assert not ov.params_valid(float("nan"), 1.0)
    assert not ov.params_valid(1e-40, 1.0)        # subnormal temperature
    assert not ov.params_valid(1.0, 0.0)
    assert not ov.params_valid(1.0, 1.5)
    assert not ov.params_valid(float("inf"), 1.0)
