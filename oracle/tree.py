"""Draft-tree structure (oracle).

Restates PTD (Progressive Tree Drafting, arXiv 2607.10661) §3.1 "tree construction":
the draft is a tree T = (V, E); each node v may attend only to its observable prefix
set pi(v) = {v} U pi(P(v)), P(v) its unique parent; the position encoding of v is fixed
by |pi(v)| so that the tree input stays compatible with causal attention.

Readings (the pages leave these open):
  * node 0 is the root (the last committed token), parent[0] = -1, and every other
    node has 0 <= parent[i] < i; a forest or a back edge is rejected;
  * ragged batches (TAPS §4.1 stage 3: the selected subtree is large when the drafter is
    confident and small otherwise, so sequences of one verify pass hold different node
    counts): rows after a sequence's last node hold parent -1 and are inactive padding.
    Padding is trailing only: the active rows are 0..n-1 with n = the first row i >= 1
    whose parent is -1 (or N).  Padding rows have no depth, position, mask bits,
    children or outputs; an active row after a padding row is rejected;
  * pi(root) = {root};
  * position id = P + |pi(v)| - 1 (0-based, P = committed prefix length), i.e. the root
    sits at position P, right after the prefix;
  * children are ordered by node index.
"""
from __future__ import annotations

import numpy as np


def active_count(parent) -> int:
    """n = number of active rows: the first row i >= 1 whose parent is -1, else N."""
    for i in range(1, len(parent)):
        if int(parent[i]) == -1:
            return i
    return len(parent)


def is_padding(parent, v: int) -> bool:
    return v >= 1 and int(parent[v]) == -1


def validate(parent) -> None:
    parent = [int(x) for x in parent]
    if len(parent) < 1:
        raise ValueError("empty tree")
    if parent[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    n = active_count(parent)
    for i in range(1, n):
        if not (0 <= parent[i] < i):
            raise ValueError(f"parent[{i}] = {parent[i]} violates 0 <= parent[i] < i")
    for i in range(n, len(parent)):
        if parent[i] != -1:
            raise ValueError(f"row {i} follows padding row {n} but has parent {parent[i]}")


def observable_set(parent, v: int) -> frozenset:
    """pi(v) = {v} U pi(P(v)), with pi(root) = {root}.

    The recursion is unrolled into its sequence of steps: v, P(v), P(P(v)), ... are added
    until the root's parent (-1) is reached (an explicit loop, so that trees deeper than
    Python's recursion limit work).
    """
    out = set()
    n = len(parent)
    while v >= 0:
        if v in out or len(out) > n:
            raise ValueError("parent array has a cycle")
        out.add(int(v))
        v = int(parent[v])
    return frozenset(out)


def root_path(parent, v: int) -> list:
    """Nodes on the root -> v path, root first (the ancestor set in sequence order)."""
    out = []
    while v >= 0:
        out.append(int(v))
        v = int(parent[v])
    return out[::-1]


def depth(parent) -> np.ndarray:
    """Edges from the root: |pi(v)| - 1 (-1 for padding rows)."""
    validate(parent)
    return np.array([-1 if is_padding(parent, v) else len(observable_set(parent, v)) - 1
                     for v in range(len(parent))], dtype=np.int32)


def position_ids(parent, prefix_len: int) -> np.ndarray:
    """0-based position of each node: P + |pi(v)| - 1 (-1 for padding rows)."""
    d = depth(parent)
    return np.where(d >= 0, prefix_len + d, -1).astype(np.int32)


def visibility(parent) -> np.ndarray:
    """Boolean [N][N]: entry (i, j) is True iff j is in pi(i) (padding rows: none)."""
    validate(parent)
    n = len(parent)
    vis = np.zeros((n, n), dtype=bool)
    for i in range(active_count(parent)):
        for j in observable_set(parent, i):
            vis[i, j] = True
    return vis


def packed_mask(parent) -> np.ndarray:
    """uint32 [N][ceil(N/32)]: bit (j % 32) of word j // 32 set iff j in pi(i)."""
    vis = visibility(parent)
    n = vis.shape[0]
    w = (n + 31) // 32
    out = np.zeros((n, w), dtype=np.uint32)
    for i in range(n):
        for j in range(n):
            if vis[i, j]:
                out[i, j // 32] |= np.uint32(1) << np.uint32(j % 32)
    return out


def children(parent) -> list:
    """children[u] = nodes whose parent is u, in ascending node index (padding rows are
    nobody's children and have none)."""
    n = len(parent)
    out = [[] for _ in range(n)]
    for i in range(1, active_count(parent)):
        out[int(parent[i])].append(i)
    return out


def child_csr(parent):
    """(offsets [N+1], child index list) with each node's children in ascending order."""
    ch = children(parent)
    off = np.zeros(len(parent) + 1, dtype=np.int32)
    idx = []
    for u, cs in enumerate(ch):
        off[u + 1] = off[u] + len(cs)
        idx.extend(cs)
    return off, np.array(idx, dtype=np.int32)
