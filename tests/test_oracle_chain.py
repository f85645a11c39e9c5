"""Pins for the oracle's chain rejection sampling, draw, alpha and accept length.

* The page's own criterion ("distribution preservation of rejection sampling,
  1.5% over 40k trials, exact under greedy"; inclusionAI/AReno PR #550, "How
  was it tested?"): with drafts drawn from q, the first emitted token follows
  p_0 and, after an accepted draft, the next one follows p_1.  Checked by total
  variation <= 0.015 and a chi-square test over 40k trials.
* Exact enumeration: for fixed drafts the outcome law of (accept length, drawn
  token) is written out from the method's definition and compared with the
  oracle's frequencies; the written law itself satisfies the
  marginal-preservation theorem exactly.
* Negative controls: an oracle with the residual replaced by p, or with the
  accept ratio inverted, must fail the distribution test.
* Closed forms: alpha = 1 - |p - q|_1 / 2, the Monte-Carlo acceptance rate,
  and the expected accept length, including the values printed in the page's
  accept-probability table (tests/golden/accept_table.txt).
"""
import os

import numpy as np
import pytest
from scipy import stats

from oracle import verify as ov

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_table.txt")


def _scenario(V=6, k=2, seed=0, T=1.0, K=0, P=1.0):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 1.2, size=(k + 1, V))
    q = rng.dirichlet(np.full(V, 0.6), size=k)
    targets = [ov.target_distribution(logits[j], T, K, P) for j in range(k + 1)]
    return logits, q, [t.p for t in targets]


def _chain_law(p, q, drafts):
    """Exact probability of each (a, y) for fixed drafts, from the definition."""
    k = len(q)
    law = {}
    pre = 1.0
    for j in range(k):
        x = drafts[j]
        px, qx = p[j][x], q[j][x]
        acc = (1.0 if px > 0 else 0.0) if qx == 0 else min(1.0, px / qx)
        r = np.maximum(p[j] - q[j], 0.0)
        r = p[j] if r.sum() == 0 else r
        for y in np.nonzero(r)[0]:
            law[(j, int(y))] = law.get((j, int(y)), 0.0) + pre * (1 - acc) * r[y] / r.sum()
        pre *= acc
    for y in np.nonzero(p[k])[0]:
        law[(k, int(y))] = law.get((k, int(y)), 0.0) + pre * p[k][y]
    return law


def _run_trials(logits, q, n, T=1.0, K=0, P=1.0, draw_seed=99, fixed_drafts=None):
    rng = np.random.default_rng(draw_seed)
    k = q.shape[0]
    res = []
    for t in range(n):
        if fixed_drafts is None:
            drafts = np.array([rng.choice(q.shape[1], p=q[j]) for j in range(k)])
        else:
            drafts = np.asarray(fixed_drafts)
        r = ov.verify_row(logits, q, drafts, T, K, P, seed=t, row=t % 7)
        res.append((drafts, r))
    return res


def _tv_and_chi2(counts, probs):
    n = counts.sum()
    tv = 0.5 * np.abs(counts / n - probs).sum()
    m = probs > 0
    assert counts[~m].sum() == 0
    chi = stats.chisquare(counts[m], probs[m] * n)
    return tv, chi.pvalue


def _first_token_stats(res, V, p0):
    c = np.bincount([r.tokens[0] for _, r in res], minlength=V)
    return _tv_and_chi2(c.astype(float), p0)


@pytest.mark.parametrize("T,K,P", [(1.0, 0, 1.0), (0.8, 4, 0.9)])
def test_distribution_preserved_40k(T, K, P):
    V = 6
    logits, q, p = _scenario(V=V, seed=4, T=T, K=K, P=P)
    res = _run_trials(logits, q, 40000, T, K, P)
    tv, pv = _first_token_stats(res, V, p[0])
    assert tv <= 0.015 and pv > 1e-3, (tv, pv)
    # after an accepted first draft, the second emitted token follows p_1
    sub = [r for _, r in res if r.accept_len >= 2]
    c = np.bincount([r.tokens[1] for r in sub], minlength=V).astype(float)
    tv1, pv1 = _tv_and_chi2(c, p[1])
    assert tv1 <= 0.015 + 0.5 / np.sqrt(len(sub)) and pv1 > 1e-3, (tv1, pv1, len(sub))


@pytest.mark.parametrize("mutation", ["residual_is_p", "inverted_accept"])
def test_planted_mistakes_fail_the_distribution_test(mutation):
    V = 6
    logits, q, p = _scenario(V=V, seed=4)
    ov.MUTATION = mutation
    try:
        res = _run_trials(logits, q, 40000)
    finally:
        ov.MUTATION = None
    tv, pv = _first_token_stats(res, V, p[0])
    assert pv < 1e-6 and tv > 0.015, (mutation, tv, pv)


def test_exact_enumeration_fixed_drafts():
    V = 5
    logits, q, p = _scenario(V=V, seed=7)
    # the written-out law preserves the marginal exactly: sum_x q(x) P(t0 | x) = p_0
    marg = np.zeros(V)
    for x0 in range(V):
        for x1 in range(V):
            w = q[0][x0] * q[1][x1]
            for (a, y), pr in _chain_law(p, q, [x0, x1]).items():
                t0 = x0 if a >= 1 else y
                marg[t0] += w * pr
    np.testing.assert_allclose(marg, p[0], atol=1e-12)
    # the oracle's outcome frequencies follow the law for fixed drafts
    for drafts in ([int(np.argmax(q[0])), int(np.argmax(q[1]))], [int(np.argmin(p[0])), 2]):
        law = _chain_law(p, q, drafts)
        keys = sorted(law)
        res = _run_trials(logits, q, 20000, fixed_drafts=drafts)
        idx = {kk: i for i, kk in enumerate(keys)}
        c = np.zeros(len(keys))
        for _, r in res:
            c[idx[(r.accept_len - 1, int(r.tokens[r.accept_len - 1]))]] += 1
        tv, pv = _tv_and_chi2(c, np.array([law[kk] for kk in keys]))
        assert pv > 1e-3 and tv < 0.02, (drafts, tv, pv)


def test_race_closed_form_two_entries():
    # Two competing weights, in one block and in two blocks: entry a wins with
    # probability r_a / (r_a + r_b) either way.
    for b_index in (1, 700):
        r = np.zeros(b_index + 1)
        r[0], r[b_index] = 0.3, 0.7
        wins = sum(ov.exponential_race(r, seed=s, row=0, pos=0, unc=r)[0] == 0 for s in range(20000))
        assert abs(wins / 20000 - 0.3) < 5 * np.sqrt(0.21 / 20000), b_index


def test_two_level_race_samples_the_weights_40k():
    # Weights spread over three blocks of the two-level race (and several
    # entries per block): the winner follows r / sum(r).
    idx = np.array([3, 100, 255, 256, 400, 700, 701])
    w = np.array([0.05, 0.2, 0.1, 0.15, 0.25, 0.05, 0.2])
    r = np.zeros(800)
    r[idx] = w
    got = np.array([ov.exponential_race(r, seed=s, row=s % 5, pos=s % 3, unc=r)[0] for s in range(40000)])
    counts = np.array([np.count_nonzero(got == i) for i in idx], dtype=float)
    assert counts.sum() == 40000
    tv, pv = _tv_and_chi2(counts, w)
    assert tv <= 0.015 and pv > 1e-3, (tv, pv)


def test_greedy_is_exact_argmax_chain():
    rng = np.random.default_rng(11)
    V, k = 40, 3
    for t in range(200):
        logits = np.round(rng.normal(0, 1, size=(k + 1, V)), 1)    # ties happen
        q = rng.dirichlet(np.ones(V), size=k)
        am = [int(np.argmax(logits[j])) for j in range(k + 1)]
        drafts = np.array([am[j] if rng.random() < 0.6 else int(rng.integers(V)) for j in range(k)])
        r = ov.verify_row(logits, q, drafts, 0.0, 0, 1.0, seed=t, row=t)
        a = next((j for j in range(k) if drafts[j] != am[j]), k)
        assert r.accept_len == a + 1
        assert list(r.tokens[:a]) == list(drafts[:a]) and r.tokens[a] == am[a]
        assert all(r.tokens[a + 1:] == -1)
        assert r.flags & (ov.F_MARGIN_ACCEPT | ov.F_MARGIN_DRAW) == 0
        np.testing.assert_allclose(r.alpha, [min(1.0, q[j][am[j]]) for j in range(k)], rtol=1e-15)


def test_alpha_closed_form_and_monte_carlo():
    V = 6
    logits, q, p = _scenario(V=V, seed=5, T=0.9, K=5, P=0.95)
    r = ov.verify_row(logits, q, np.array([0, 0]), 0.9, 5, 0.95, seed=0, row=0)
    for j in range(2):
        np.testing.assert_allclose(r.alpha[j], 1 - 0.5 * np.abs(p[j] - q[j]).sum(), rtol=1e-13)
    res = _run_trials(logits, q, 20000, 0.9, 5, 0.95)
    acc0 = np.mean([rr.accept_len >= 2 for _, rr in res])
    a0 = r.alpha[0]
    assert abs(acc0 - a0) < 5 * np.sqrt(a0 * (1 - a0) / 20000)
    # expected accept length with independent drafts
    mean_len = np.mean([rr.accept_len for _, rr in res])
    el = ov.expected_accept_length(r.alpha)
    sd = np.std([rr.accept_len for _, rr in res])
    assert abs(mean_len - el) < 5 * sd / np.sqrt(len(res))


def test_expected_accept_length_matches_page_table():
    vals = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        key, v = line.split()
        vals[key] = float(v)
    a1, a2 = vals["alpha_depth1"], vals["alpha_depth2_given_depth1"]
    assert round(ov.expected_accept_length([a1]), 2) == vals["expected_accept_length_k1"]
    assert round(ov.expected_accept_length([a1, a2]), 2) == vals["expected_accept_length_k2"]


def test_invalid_inputs():
    V, k = 8, 2
    rng = np.random.default_rng(0)
    logits = rng.normal(size=(k + 1, V))
    q = rng.dirichlet(np.ones(V), size=k)
    bad = logits.copy()
    bad[1, 3] = np.nan
    r = ov.verify_row(bad, q, np.array([0, 1]), 1.0, 0, 1.0, 0, 0)
    assert r.flags == ov.F_NAN and r.accept_len == 0 and all(r.tokens == -1)
    bad = logits.copy()
    bad[2, :] = -np.inf
    assert ov.verify_row(bad, q, np.array([0, 1]), 1.0, 0, 1.0, 0, 0).flags == ov.F_NAN
    r = ov.verify_row(logits, q, np.array([V, 1]), 1.0, 0, 1.0, 0, 0)
    assert r.flags & ov.F_BAD_TOKEN and r.accept_len == 1
    r = ov.verify_row(logits, q, np.array([0, 1]), -1.0, 0, 1.0, 0, 0)
    assert r.flags & ov.F_BAD_PARAM
    am0 = int(np.argmax(logits[0]))
    assert r.tokens[0] == am0 or r.accept_len > 1
    # a masked (-inf) entry is never drawn
    masked = logits.copy()
    masked[:, 0] = -np.inf
    for s in range(200):
        rr = ov.verify_row(masked, q, np.array([1, 2]), 1.0, 0, 1.0, s, 0)
        assert 0 not in rr.tokens[:rr.accept_len]
