"""Budgeted prefix-closed subtree selection from a block-marginal pool (oracle).

What it restates
  * TAPS §4.1 stage 1: a drafter emits per-position marginals for d future positions;
    the top-K tokens of every position form the candidate tree.  A candidate node at
    depth k is a rank path (r_1, ..., r_k), its token the rank-r_k token of position k.
  * TAPS §4.2: edge estimates q_cond(u -> v) = Pr(accept v | reach u) are propagated to a
    path-level reach probability; §1/§3.2: a compact prefix-closed subtree is chosen
    greedily under a verification budget to maximise the expected accepted tokens.
  * TreeGraft §3.1: the cumulative path score s(v) = product over the non-root nodes u
    on the root->v path of the edge score p(u); s(root) = 1.

Readings
  * q_cond(u -> v) := the child's per-position marginal (TAPS's learned scorer is
    truncated on the page and needs trained weights).
  * s is formed in fp32, left to right along the path: s = fl(...fl(fl(1*m_1)*m_2)...*m_k).
  * Budget B counts rows including the root: B - 1 candidates are selected.
  * Total order: score descending, then depth ascending, then rank path
    lexicographically ascending.  A child never precedes its parent in this order
    (its score is no larger, and ties go to the shallower node), so its first B - 1
    elements are prefix-closed; they also maximise the sum of s (= the expected number
    of accepted drafts under the reading) over all prefix-closed sets of that size.
  * Pool ranks are ordered by (probability desc, token asc) on input.
Output nodes are numbered in selection order (so parent < child), root = node 0.

Algorithm: best-first search over the candidate tree in its first-child / next-sibling
form, which is heap-ordered in the total order above (a first child and a next sibling
never precede the node they come from); popping B - 1 times yields the first B - 1.
"""
from __future__ import annotations

import heapq

import numpy as np


def path_score(marg, path) -> np.float32:
    s = np.float32(1.0)
    for k, r in enumerate(path):
        s = np.float32(s * np.float32(marg[k][r]))
    return s


def select_subtree(marg, pool_tokens, budget: int, root_token: int):
    """marg float32 [d][K], pool_tokens int32 [d][K].  Returns dict of arrays sized
    ``budget`` (parent, token, depth int32; score float32; rank path list) plus
    ``n_nodes`` (rows used; unused rows hold -1 / 0)."""
    marg = np.asarray(marg, dtype=np.float32)
    d, kk = marg.shape
    if budget < 1:
        raise ValueError("budget counts the root; it must be >= 1")
    parent = np.full(budget, -1, dtype=np.int32)
    token = np.full(budget, -1, dtype=np.int32)
    depth = np.full(budget, -1, dtype=np.int32)
    score = np.zeros(budget, dtype=np.float32)
    paths = [()]
    token[0] = root_token
    depth[0] = 0
    score[0] = np.float32(1.0)
    n = 1
    heap = []
    # entry: (-score, depth, rank path, parent node index, parent score)
    if d >= 1 and kk >= 1 and budget > 1:
        s0 = np.float32(np.float32(1.0) * marg[0][0])
        heapq.heappush(heap, (-float(s0), 1, (0,), 0, np.float32(1.0)))
    while heap and n < budget:
        neg_s, dep, path, par, par_s = heapq.heappop(heap)
        s = np.float32(-neg_s)
        me = n
        parent[me] = par
        token[me] = int(pool_tokens[dep - 1][path[-1]])
        depth[me] = dep
        score[me] = s
        paths.append(path)
        n += 1
        if dep < d:  # first child: rank 0 at the next position
            sc = np.float32(s * marg[dep][0])
            heapq.heappush(heap, (-float(sc), dep + 1, path + (0,), me, s))
        r = path[-1]
        if r + 1 < kk:  # next sibling under the same parent
            ss = np.float32(par_s * marg[dep - 1][r + 1])
            heapq.heappush(heap, (-float(ss), dep, path[:-1] + (r + 1,), par, par_s))
    return {"parent": parent, "token": token, "depth": depth, "score": score,
            "paths": paths, "n_nodes": n}


# ------------------------------------------------------------------------------------
# Cost-aware size of the verified tree.
#
# TAPS §3.1 (limitation 2): verification latency grows with the number of selected
# nodes (64 -> 512 nodes took 33 -> 81 ms in the paper's figure) while each round still
# commits one prefix; §3.2: the selector should pick a compact prefix-closed subtree
# that maximises expected accepted tokens per unit of verification cost rather than
# fill the budget.
#
# Readings
#   * Expected tokens of a round with the first n rows of the selection order (root
#     included) = 1 + sum of s over its n - 1 drafts: under the edge-score reading s(v)
#     is the probability that v is accepted, and every round also yields one token from
#     the target (the bonus or corrected token).
#   * Verification cost of n rows = cost_base + cost_per_row * n, a line fitted to the
#     measured step time against the tree size.
#   * n* = the smallest n in [1, available rows] that maximises
#     (1 + sum_{i<n} s_i) / (cost_base + cost_per_row * n).  For a result that does not
#     depend on the order of additions, every score is first rounded to a multiple of
#     2^-40 (round half to even) and the sums are exact integers; numerator, denominator
#     and quotient are then single IEEE double operations.
FIX_BITS = 40


def adaptive_rows(scores, cost_base: float, cost_per_row: float) -> int:
    """scores: the selected rows' scores in selection order, root first (any value)."""
    cost_base = float(np.float32(cost_base))
    cost_per_row = float(np.float32(cost_per_row))
    unit = 2 ** FIX_BITS
    best_n, best = 1, None
    acc = 0  # exact sum of the rounded draft scores so far
    for n in range(1, len(scores) + 1):
        if n > 1:
            acc += round(float(np.float32(scores[n - 1])) * unit)
        num = float(unit + acc)
        den = cost_base + cost_per_row * float(n)
        val = num / den
        if best is None or val > best:
            best, best_n = val, n
    return best_n


def select_subtree_adaptive(marg, pool_tokens, budget: int, root_token: int, cost_base: float,
                            cost_per_row: float):
    """select_subtree(budget) cut to its cost-aware prefix of n* rows (rows beyond it
    become -1 / score 0, like rows past the available candidates)."""
    res = select_subtree(marg, pool_tokens, budget, root_token)
    n_avail = int(res["n_nodes"])
    n = adaptive_rows(res["score"][:n_avail], cost_base, cost_per_row)
    for key, fill in (("parent", -1), ("token", -1), ("depth", -1), ("score", 0.0)):
        res[key][n:] = fill
    res["n_nodes"] = n
    return res
