"""Stochastic (sampling) acceptance walk down a draft tree (oracle, float64).

What it restates (speculative-decoding blog):
  * "acceptance probability for sampling": draft token y_i, proposed with draft
    probability q_i(y_i), is kept with probability alpha_i = min(1, p_i(y_i) / q_i(y_i)),
    p_i the target distribution under the same prefix;
  * "how to correct after a rejection": after the first rejection the replacement token
    is drawn from the positive residual (p_i - q_i)+ / sum_v (p_i(v) - q_i(v))+, and the
    drafts after it are discarded;
  * the point of the rule is that the output keeps the target's distribution.

Readings (the pages state the rule for one draft per position only):
  * p_u = softmax(target[u] / T), q_u = softmax(draft[u] / T); T applies to both.
  * At node u the children c_1..c_m (ascending node index) are tried in turn.  Child k
    uses r = U(seed, round, b, u, k, kind 0); it is accepted iff r < alpha, with
    alpha = min(1, p(t_k) / q(t_k)); if q(t_k) = 0 then alpha = 1 when p(t_k) > 0, else 0.
  * After rejecting t_k: p <- (p - q)+ / sum (p - q)+ (kept unchanged if that sum is 0),
    and q <- q with t_k removed and renormalised (drafts at one node are distinct tokens,
    i.e. drawn without replacement), q <- 0 if nothing is left.  With m = 1 this is
    exactly the pages' rule.
  * On acceptance the walk moves to the child and starts over with its rows.  When every
    child is rejected, or u is a leaf, the output token is drawn from the current p by
    inverse CDF with r = U(seed, round, b, u, 0, kind 1): the smallest v such that
    r * sum(p) < p(0) + ... + p(v).
Every random decision is also returned with its margin, as a (kind, margin) pair:
("accept", |r - alpha|) for an acceptance test and ("icdf", distance from r * sum(p) to
the nearest edge of the chosen bucket, relative to sum(p)) for the final draw, so that a
float implementation can be compared decision by decision.
"""
from __future__ import annotations

import numpy as np

from .philox import uniform
from .tree import children, validate


def softmax_row(x_row, temperature: float) -> np.ndarray:
    z = np.asarray(x_row, dtype=np.float64) / temperature
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def acceptance_prob(pt: float, qt: float) -> float:
    if qt > 0.0:
        return min(1.0, pt / qt)
    return 1.0 if pt > 0.0 else 0.0


def inverse_cdf(p: np.ndarray, r: float):
    """Smallest v with r * sum(p) < cumsum(p)[v]; returns (v, relative margin)."""
    cdf = np.cumsum(p)
    total = float(cdf[-1])
    target = r * total
    v = int(np.searchsorted(cdf, target, side="right"))
    v = min(v, len(p) - 1)
    lo = float(cdf[v - 1]) if v > 0 else 0.0
    hi = float(cdf[v])
    margin = min(target - lo, hi - target) / total if total > 0 else 0.0
    return v, margin


def sampling_walk(target_logits, draft_logits, parent, tokens, temperature: float,
                  seed: int, rnd: int, b: int):
    """One sequence.  Returns (accepted nodes excluding the root, output token,
    decision margins, the node at which the output token was drawn)."""
    validate(parent)
    kids = children(parent)
    u = 0
    accepted = []
    margins = []
    while True:
        p = softmax_row(target_logits[u], temperature)
        q = softmax_row(draft_logits[u], temperature)
        moved = False
        for k, c in enumerate(kids[u], start=1):
            t = int(tokens[c])
            r = uniform(seed, rnd, b, u, k, 0)
            alpha = acceptance_prob(float(p[t]), float(q[t]))
            margins.append(("accept", abs(r - alpha)))
            if r < alpha:
                accepted.append(c)
                u = c
                moved = True
                break
            resid = np.maximum(p - q, 0.0)
            z = float(resid.sum())
            if z > 0.0:
                p = resid / z
            q = q.copy()
            q[t] = 0.0
            qs = float(q.sum())
            q = q / qs if qs > 0.0 else np.zeros_like(q)
        if moved:
            continue
        r = uniform(seed, rnd, b, u, 0, 1)
        v, m = inverse_cdf(p, r)
        margins.append(("icdf", m))
        return accepted, v, margins, u
