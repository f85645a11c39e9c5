"""Pins for the draft-side sampler's oracle (oracle/draft.py).

* q against independent routines: the unfiltered distribution is
  scipy.special.softmax of the tempered logits; under greedy decoding q is
  one-hot at numpy's first argmax and the logprob is scipy's log_softmax;
  top-k keeps exactly the K largest entries (numpy's sort), renormalised by
  scipy's softmax over them.
* The draw follows q: over 40k stream rows the token frequencies pass a
  chi-square test against q (V = 700: a partial last race block with
  weight in it), with and without filters.
* The draft streams are not the verify's: the verify's bonus draw at the same
  (seed, row, position), and the draft draw at another position, agree only
  as often as independent draws do (sum of q^2), not always.
* Invalid input and invalid parameters follow the verify's rules.
"""
import numpy as np
import pytest
from scipy import special, stats

from oracle import draft as od
from oracle import verify as ov


def _logits(V=700, seed=3, scale=1.5):
    return np.random.default_rng(seed).normal(0, scale, size=V)


def test_unfiltered_q_is_scipy_softmax_and_logprob_is_log_softmax():
    l = _logits()
    for T in (1.0, 0.6):
        r = od.draft_row(l, T, 0, 1.0, seed=11, row=5, pos=2)
        assert np.allclose(r.q, special.softmax(l / T), rtol=1e-12, atol=1e-15)
        assert abs(r.logprob - special.log_softmax(l / T)[r.x]) < 1e-12
        assert r.flags == 0


def test_greedy_is_one_hot_at_first_argmax_with_raw_logprob():
    l = _logits()
    l[[40, 90]] = l.max() + 1.0          # an exact tie for the maximum
    r = od.draft_row(l, 0.0, 0, 1.0, seed=1, row=0, pos=0)
    assert r.x == int(np.argmax(l)) == 40
    assert r.q[40] == 1.0 and r.q.sum() == 1.0
    assert abs(r.logprob - special.log_softmax(l)[40]) < 1e-12


def test_top_k_keeps_the_k_largest():
    l = _logits(seed=8)
    K = 17
    r = od.draft_row(l, 0.8, K, 1.0, seed=2, row=3, pos=1)
    top = np.argsort(-l, kind="stable")[:K]
    assert set(np.nonzero(r.q)[0]) == set(top)
    assert np.allclose(r.q[top], special.softmax(l[top] / 0.8), rtol=1e-12)
    assert r.x in set(top)


def _chi2(p, draws, n):
    counts = np.bincount(draws, minlength=len(p))
    m = p * n >= 5
    stat = stats.chisquare(counts[m], p[m] * n * counts[m].sum() / (p[m] * n).sum())
    return stat.pvalue, counts


@pytest.mark.parametrize("T,K,P", [(1.0, 0, 1.0), (0.8, 40, 1.0), (1.2, 0, 0.9)])
def test_draws_follow_q_40k(T, K, P):
    l = _logits(V=700, seed=21, scale=1.0)
    n = 40000
    q = od.draft_row(l, T, K, P, seed=5, row=0, pos=0).q
    draws = np.array([od.draft_row(l, T, K, P, seed=5, row=r, pos=0).x for r in range(n)])
    pv, counts = _chi2(q, draws, n)
    assert pv > 1e-4
    # total variation within twice its expected sampling noise
    noise = 0.5 * np.sum(np.sqrt(2.0 * q * (1.0 - q) / (np.pi * n)))
    assert 0.5 * np.abs(counts / n - q).sum() < 2.0 * noise
    assert np.all(q[draws] > 0)


def test_streams_are_not_the_verifys_and_positions_differ():
    l = _logits(V=40, seed=4, scale=0.3)   # a flat q: independent draws rarely agree
    n = 3000
    q = od.draft_row(l, 1.0, 0, 1.0, 9, 0, 0).q
    d0 = np.array([od.draft_row(l, 1.0, 0, 1.0, 9, r, 0).x for r in range(n)])
    d1 = np.array([od.draft_row(l, 1.0, 0, 1.0, 9, r, 1).x for r in range(n)])
    # the verify's bonus draw of the same row at the same position (k = 0)
    v0 = ov.verify(l[None, None, :].repeat(n, 0), np.zeros((n, 0, 40)), np.zeros((n, 0), np.int32),
                   np.ones(n), np.zeros(n, np.int32), np.ones(n), 9)["tokens"][:, 0]
    indep = float(np.sum(q ** 2))
    for other in (d1, v0):
        agree = float(np.mean(d0 == other))
        assert agree < indep + 0.03, (agree, indep)
    assert np.array_equal(d0, np.array([od.draft_row(l, 1.0, 0, 1.0, 9, r, 0).x for r in range(n)]))


def test_invalid_input_and_parameters():
    l = _logits(V=50)
    bad = l.copy()
    bad[7] = np.nan
    r = od.draft_row(bad, 1.0, 0, 1.0, 1, 0, 0)
    assert r.flags == ov.F_NAN and r.x == -1 and not r.q.any() and r.logprob == 0.0
    r = od.draft_row(np.full(50, -np.inf), 1.0, 0, 1.0, 1, 0, 0)
    assert r.flags == ov.F_NAN and r.x == -1
    r = od.draft_row(l, -1.0, 0, 1.0, 1, 0, 0)        # a bad temperature: greedy, flagged
    assert r.flags & ov.F_BAD_PARAM and r.x == int(np.argmax(l)) and r.q[r.x] == 1.0


def test_batch_matches_rows_with_row_base():
    rng = np.random.default_rng(6)
    L = rng.normal(0, 2, size=(5, 300))
    T = np.array([1.0, 0.0, 0.7, 1.1, 0.9])
    K = np.array([0, 0, 30, 0, 5], np.int32)
    P = np.array([1.0, 1.0, 0.9, 0.8, 1.0])
    out = od.draft_sample(L, T, K, P, seed=44, pos=3, row_base=100)
    for r in range(5):
        one = od.draft_row(L[r], T[r], int(K[r]), P[r], 44, 100 + r, 3)
        assert out["tokens"][r] == one.x and np.array_equal(out["q"][r], one.q)
