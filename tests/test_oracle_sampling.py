"""Pins for oracle.sampling: the pages' promise that sampling-mode verification keeps
the target distribution (blog: 'acceptance probability for sampling', 'how to correct
after a rejection'), checked by a chi-square test on tiny vocabularies with drafts
redrawn from q every round; plus closed-form special cases of the acceptance rule."""
import math

import numpy as np
import pytest
from scipy import stats

import synth
from oracle import sampling


def _first_token_hist(target_row, draft_row, m, n_rounds, seed, temperature=1.0):
    g = synth.rng(seed)
    v = len(target_row)
    parent = np.array([-1] + [0] * m, dtype=np.int32)
    rows_t = np.stack([target_row] * (m + 1))
    rows_d = np.stack([draft_row] * (m + 1))
    hist = np.zeros(v, dtype=np.int64)
    for rnd in range(n_rounds):
        toks = synth.draw_children_from_draft(g, parent, rows_d, temperature)
        acc, tok, _, _ = sampling.sampling_walk(rows_t, rows_d, parent, toks, temperature, seed, rnd, 0)
        hist[int(toks[acc[0]]) if acc else tok] += 1
    return hist


@pytest.mark.parametrize("m,temp", [(1, 1.0), (2, 1.0), (3, 0.7)])
def test_first_token_follows_target(m, temp):
    v = 8
    g = synth.rng(100 + m)
    tgt = synth.normal(g, v, std=math.sqrt(2))
    drf = (tgt + synth.normal(g, v, std=1.0)).astype(np.float32)
    n = 12000
    hist = _first_token_hist(tgt, drf, m, n, seed=7 + m, temperature=temp)
    p = sampling.softmax_row(tgt, temp)
    chi2 = float(np.sum((hist - n * p) ** 2 / (n * p)))
    crit = stats.chi2.ppf(1 - 1e-3, df=v - 1)
    assert chi2 < crit, (chi2, crit, hist, n * p)


def test_chi_square_detects_a_wrong_residual():
    # Sanity of the test itself: drawing the correction from p instead of (p - q)+
    # must fail the same check.
    v, n = 8, 12000
    g = synth.rng(5)
    tgt = synth.normal(g, v, std=math.sqrt(2))
    drf = (tgt + synth.normal(g, v, std=1.0)).astype(np.float32)
    p = sampling.softmax_row(tgt, 1.0)
    q = sampling.softmax_row(drf, 1.0)
    gg = synth.rng(9)
    hist = np.zeros(v, dtype=np.int64)
    from oracle.philox import uniform
    for rnd in range(n):
        t = int(gg.choice(v, p=q))
        r = uniform(3, rnd, 0, 0, 1, 0)
        if r < min(1.0, p[t] / q[t]):
            hist[t] += 1
        else:
            hist[sampling.inverse_cdf(p, uniform(3, rnd, 0, 0, 0, 1))[0]] += 1
    chi2 = float(np.sum((hist - n * p) ** 2 / (n * p)))
    assert chi2 > stats.chi2.ppf(1 - 1e-3, df=v - 1)


def test_single_draft_acceptance_rate_is_min_one_p_over_q():
    v = 6
    g = synth.rng(21)
    tgt = synth.normal(g, v, std=math.sqrt(2))
    drf = synth.normal(g, v, std=math.sqrt(2))
    p = sampling.softmax_row(tgt, 1.0)
    q = sampling.softmax_row(drf, 1.0)
    t = int(np.argmax(q / p))  # a token the draft over-proposes: alpha < 1
    alpha = min(1.0, p[t] / q[t])
    parent = np.array([-1, 0], dtype=np.int32)
    toks = np.array([0, t], dtype=np.int32)
    n = 6000
    acc = sum(bool(sampling.sampling_walk(np.stack([tgt] * 2), np.stack([drf] * 2), parent, toks, 1.0, 77, r, 0)[0])
              for r in range(n))
    sd = math.sqrt(alpha * (1 - alpha) / n)
    assert abs(acc / n - alpha) < 4.5 * sd


def test_identical_distributions_always_accept():
    v = 10
    g = synth.rng(22)
    x = synth.normal(g, (4, v), std=math.sqrt(2))
    parent = np.array([-1, 0, 1, 2], dtype=np.int32)
    toks = np.array([0, 3, 5, 7], dtype=np.int32)
    for r in range(200):
        acc, tok, _, at = sampling.sampling_walk(x, x, parent, toks, 1.0, 5, r, 0)
        assert acc == [1, 2, 3] and at == 3


def test_rejection_draws_from_positive_residual():
    # p = (1/2, 1/2, 0, 0); the draft is certain of token 1.  alpha = 1/2; after a
    # rejection the residual (p - q)+ is all on token 0.
    ninf = -np.inf
    tgt = np.array([[0.0, 0.0, ninf, ninf]] * 2)
    drf = np.array([[ninf, 0.0, ninf, ninf]] * 2)
    parent = np.array([-1, 0], dtype=np.int32)
    toks = np.array([2, 1], dtype=np.int32)
    n_acc = 0
    for r in range(4000):
        acc, tok, _, at = sampling.sampling_walk(tgt, drf, parent, toks, 1.0, 11, r, 0)
        if acc:
            n_acc += 1
        else:
            assert tok == 0 and at == 0
    assert abs(n_acc / 4000 - 0.5) < 4.5 * math.sqrt(0.25 / 4000)


def test_zero_draft_probability_edge_cases():
    ninf = -np.inf
    parent = np.array([-1, 0], dtype=np.int32)
    # q(t) = 0, p(t) > 0 -> always accepted
    tgt = np.array([[0.0, 0.0, 0.0]] * 2)
    drf = np.array([[0.0, 0.0, ninf]] * 2)
    for r in range(100):
        acc, _, _, _ = sampling.sampling_walk(tgt, drf, parent, np.array([0, 2]), 1.0, 1, r, 0)
        assert acc == [1]
    # p(t) = 0 -> never accepted, and the correction never returns t
    tgt2 = np.array([[0.0, 0.0, ninf]] * 2)
    drf2 = np.array([[0.0, 0.0, 0.0]] * 2)
    for r in range(100):
        acc, tok, _, _ = sampling.sampling_walk(tgt2, drf2, parent, np.array([0, 2]), 1.0, 1, r, 0)
        assert acc == [] and tok != 2


def test_inverse_cdf_boundaries():
    p = np.array([0.25, 0.0, 0.5, 0.25])
    assert sampling.inverse_cdf(p, 0.0)[0] == 0
    assert sampling.inverse_cdf(p, 0.2499)[0] == 0
    assert sampling.inverse_cdf(p, 0.25)[0] == 2   # zero-mass token 1 is never drawn
    assert sampling.inverse_cdf(p, 0.7499)[0] == 2
    assert sampling.inverse_cdf(p, 0.75)[0] == 3
    assert sampling.inverse_cdf(p, 1.0 - 2 ** -24)[0] == 3
