"""One single-drafter tree-expansion step (oracle).

What it restates
  * TreeGraft §3.1 "standard single-drafter tree expansion": at drafting step k the
    drafter takes a candidate pool C_k of the current tree (for a single drafter, the
    nodes made in the previous step), ranks it by the cumulative path score s(v) and
    expands the frontier F_k = Top_W(C_k, s).  For every frontier node it runs one
    forward on the prefix ending at that node, and attaches the top-m tokens of the
    resulting next-token distribution as children; the drafter's probability of each
    attached token is the edge score p(u), and s(child) = s(parent) * p(u)
    (s(root) = 1).  The attached children form the next step's pool N_{k+1}.

Readings (not fixed by the page)
  * Ties in s when choosing the frontier go to the lower candidate position; ties in
    the logits when choosing children go to the lower token id (the order the pool
    convention elsewhere uses: probability descending, token ascending).
  * The drafter distribution is softmax(x / T); p is formed in float64 and rounded
    once to float32; s(child) = fl32(s(parent) * p), like the selection's fp32 path
    products.
  * The drafter forward itself is outside the path: its next-token logits (one row per
    frontier node) are the input.
"""
from __future__ import annotations

import numpy as np


def frontier_topw(scores, count: int, width: int):
    """Positions (into the candidate list) of the Top_W candidates among scores[:count],
    highest s first, ties by position; fewer if count < width."""
    s = [float(np.float32(x)) for x in scores[:count]]
    order = sorted(range(count), key=lambda i: (-s[i], i))
    return order[:width]


def attach_children(logits_row, parent_score: float, m: int, temperature: float = 1.0):
    """Top-m tokens of one drafter row with their edge and path scores.
    Returns (tokens int32 [m'], p float32 [m'], s float32 [m']) with m' = min(m, V)."""
    x = np.asarray(logits_row, dtype=np.float64)
    v = x.shape[0]
    z = x / float(temperature)
    zmax = z.max()
    lse = zmax + np.log(np.exp(z - zmax).sum())
    # highest logit first, ties by token id: a stable sort of -x keeps ascending ids
    order = np.argsort(-x, kind="stable")[:min(m, v)]
    p = np.exp(z[order] - lse).astype(np.float32)
    s = (np.float32(parent_score) * p).astype(np.float32)
    return order.astype(np.int32), p, s


def expand_step(logits, parent_scores, m: int, temperature: float = 1.0):
    """attach_children for every row of logits [R][V] with parent_scores [R]."""
    rows = [attach_children(logits[r], parent_scores[r], m, temperature) for r in range(logits.shape[0])]
    return (np.stack([t for t, _, _ in rows]), np.stack([p for _, p, _ in rows]),
            np.stack([s for _, _, s in rows]))
