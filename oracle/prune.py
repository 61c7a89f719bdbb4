"""Width and depth control of a draft tree (oracle).

What it restates
  * PTD (Progressive Tree Drafting) §3.1, "overhead constraints": the tree's growth is
    bounded in two dimensions.  Width control caps the number of children of every
    parent, so that low-confidence tokens do not branch out.  Depth control is a
    sliding-window "stepping" mechanism: when the (sub)tree exceeds a depth threshold,
    the earliest-added child and its descendants are kept as the new subtree and every
    other, stale branch is pruned.  (The page is cut off inside this paragraph.)

Readings (not fixed by the page)
  * Nodes are numbered in the order they were added (parent < child), so "earliest
    added" = lowest index.  Each node carries a confidence (e.g. its drafter
    probability); width control keeps, per parent, the max_children children with the
    highest confidence (ties to the lower index) and drops the rest with their subtrees.
  * Depth of a node = edges from the current root.  While the kept tree's depth exceeds
    depth_limit, the root's lowest-index kept child becomes the root (everything outside
    its subtree is pruned).  depth_limit >= 1.
  * The result is compacted in the original order: old_to_new[v] is v's new index or -1,
    new_parent[i] the new index of i's parent (-1 for the new root), n_kept the count.
"""
from __future__ import annotations

import numpy as np

from .tree import children, validate


def prune_tree(parent, conf, max_children: int, depth_limit: int):
    parent = [int(p) for p in parent]
    n = len(parent)
    validate(parent)
    conf = [float(np.float32(c)) for c in conf]
    kids = children(parent)
    keep = [True] * n
    # width control
    for u in range(n):
        ranked = sorted(kids[u], key=lambda c: (-conf[c], c))
        for c in ranked[max_children:]:
            keep[c] = False
    for v in range(1, n):  # a dropped node takes its subtree with it (parent < child)
        if not keep[parent[v]]:
            keep[v] = False
    # depth control
    depth = [0] * n
    for v in range(1, n):
        depth[v] = depth[parent[v]] + 1
    root = 0

    def in_subtree(v, r):
        while v != -1 and depth[v] >= depth[r]:
            if v == r:
                return True
            v = parent[v]
        return False

    while True:
        sub = [v for v in range(n) if keep[v] and in_subtree(v, root)]
        if max(depth[v] for v in sub) - depth[root] <= depth_limit:
            break
        first = [c for c in kids[root] if keep[c]]
        if not first:
            break
        root = min(first)
    for v in range(n):
        if keep[v] and not in_subtree(v, root):
            keep[v] = False
    old_to_new = [-1] * n
    new_parent = []
    for v in range(n):
        if keep[v]:
            old_to_new[v] = len(new_parent)
            new_parent.append(-1 if v == root else old_to_new[parent[v]])
    return {"old_to_new": np.array(old_to_new, dtype=np.int32),
            "new_parent": np.array(new_parent, dtype=np.int32),
            "n_kept": len(new_parent), "root": root}
