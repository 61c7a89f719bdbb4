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


def _two_token_hist(p1_logits, p2_logits, q1_logits, q2_logits, m1, m2, n_rounds, seed):
    """Root with m1 drafted children, each with m2 drafted children; the target and draft
    rows of a depth-1 node depend on its token.  Returns the joint histogram of the first
    two tokens of the generated text: the round's accepted tokens and its final token,
    topped up, when the round ends after one token, by one plain target step from the
    context that token makes."""
    g = synth.rng(seed)
    v = len(p1_logits)
    parent = [-1] + [0] * m1
    for c in range(1, m1 + 1):
        parent += [c] * m2
    parent = np.array(parent, dtype=np.int32)
    n = len(parent)

    def probs(logits):
        z = logits.astype(np.float64)
        w = np.exp(z - z.max())
        return w / w.sum()

    hist = np.zeros((v, v), dtype=np.int64)
    for rnd in range(n_rounds):
        tok = np.zeros(n, dtype=np.int32)
        tok[1:m1 + 1] = g.choice(v, size=m1, replace=False, p=probs(q1_logits))
        rows_t = np.empty((n, v), dtype=np.float32)
        rows_d = np.empty((n, v), dtype=np.float32)
        rows_t[0], rows_d[0] = p1_logits, q1_logits
        for c in range(1, m1 + 1):
            rows_t[c], rows_d[c] = p2_logits[tok[c]], q2_logits[tok[c]]
            kids = np.flatnonzero(parent == c)
            tok[kids] = g.choice(v, size=m2, replace=False, p=probs(q2_logits[tok[c]]))
            for k in kids:
                # Depth-2 rows are never read for a decision about the first two tokens.
                rows_t[k], rows_d[k] = p1_logits, q1_logits
        acc, last, _, _ = sampling.sampling_walk(rows_t, rows_d, parent, tok, 1.0, seed, rnd, 0)
        out = [int(tok[c]) for c in acc] + [int(last)]
        if len(out) == 1:
            out.append(int(g.choice(v, p=probs(p2_logits[out[0]]))))
        hist[out[0], out[1]] += 1
    return hist


def test_first_two_tokens_follow_the_target_joint():
    # Losslessness one level down the tree: after an acceptance the walk restarts at the
    # accepted child with that child's rows, so the first two generated tokens follow
    # p1(x1) p2(x2 | x1) whatever the drafter does at either level.
    v, n = 4, 16000
    g = synth.rng(41)
    p1 = synth.normal(g, v, std=1.0)
    p2 = np.stack([synth.normal(g, v, std=1.0) for _ in range(v)])
    q1 = (p1 + synth.normal(g, v, std=1.0)).astype(np.float32)
    q2 = (p2 + np.stack([synth.normal(g, v, std=1.0) for _ in range(v)])).astype(np.float32)
    hist = _two_token_hist(p1, p2, q1, q2, 2, 2, n, seed=43)
    sp1 = sampling.softmax_row(p1, 1.0)
    joint = np.stack([sp1[a] * sampling.softmax_row(p2[a], 1.0) for a in range(v)])
    expect = n * joint
    assert expect.min() >= 5.0
    crit = stats.chi2.ppf(1 - 1e-3, df=v * v - 1)
    chi2 = float(np.sum((hist - expect) ** 2 / expect))
    assert chi2 < crit, (chi2, crit, hist, expect)
    # Power of the check: the same counts fail against a joint whose second token
    # ignores the first (every context's row replaced by the first context's row).
    wrong = n * np.outer(sp1, sampling.softmax_row(p2[0], 1.0))
    assert float(np.sum((hist - wrong) ** 2 / wrong)) > crit


def test_padded_rows_are_never_tried():
    # padding rows of a ragged batch are nobody's children: the walk, its draws and its
    # output equal those of the unpadded tree
    g = synth.rng(91)
    V, n, N = 12, 7, 11
    par = np.array([-1, 0, 0, 1, 1, 2, 3], dtype=np.int32)
    tgt = g.standard_normal((N, V)) * 2
    drf = tgt + g.standard_normal((N, V)) * 0.5
    tok = synth.draw_children_from_draft(g, par, drf[:n], 1.0)
    pad = np.concatenate([par, np.full(N - n, -1, np.int32)])
    tokp = np.concatenate([tok, np.full(N - n, -1, np.int32)])
    for seed in range(20):
        a = sampling.sampling_walk(tgt, drf, pad, tokp, 1.0, seed, 3, 0)
        b = sampling.sampling_walk(tgt[:n], drf[:n], par, tok, 1.0, seed, 3, 0)
        assert a[0] == b[0] and a[1] == b[1]
