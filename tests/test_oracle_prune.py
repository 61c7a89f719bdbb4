"""Pins of oracle.prune (CPU): hand-built trees, closed forms and brute force."""
import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import prune, tree


def test_width_cap_keeps_the_most_confident_children():
    #      0
    #   1  2  3        conf 0.2 0.9 0.5  -> keep 2 and 3 with cap 2
    #   |     |
    #   4     5
    parent = [-1, 0, 0, 0, 1, 3]
    conf = [1, 0.2, 0.9, 0.5, 0.9, 0.9]
    r = prune.prune_tree(parent, conf, 2, 10)
    assert r["old_to_new"].tolist() == [0, -1, 1, 2, -1, 3]  # node 1 and its child 4 are gone
    assert r["new_parent"].tolist() == [-1, 0, 0, 2]
    assert r["n_kept"] == 4 and r["root"] == 0


def test_width_ties_go_to_the_earlier_child():
    parent = [-1, 0, 0, 0]
    r = prune.prune_tree(parent, [1, 0.5, 0.5, 0.5], 1, 10)
    assert r["old_to_new"].tolist() == [0, 0 + 1, -1, -1]


def test_depth_stepping_moves_the_root_down_the_earliest_branch():
    # chain 0-1-2-3-4-5 plus a side branch 0-6-7; limit 3
    parent = [-1, 0, 1, 2, 3, 4, 0, 6]
    r = prune.prune_tree(parent, [1] * 8, 8, 3)
    # depth 5 > 3: root -> 1 (earliest child; depth below it 4 > 3) -> 2 (depth 3): stop
    assert r["root"] == 2
    assert r["old_to_new"].tolist() == [-1, -1, 0, 1, 2, 3, -1, -1]
    assert r["new_parent"].tolist() == [-1, 0, 1, 2]


def test_depth_stepping_can_cut_away_the_deep_branch():
    # the deep branch hangs under the later child: stepping into the earliest child ends it
    parent = [-1, 0, 0, 2, 3, 4]
    r = prune.prune_tree(parent, [1] * 6, 8, 2)
    assert r["root"] == 1 and r["n_kept"] == 1
    assert r["new_parent"].tolist() == [-1]


def test_no_constraint_active_is_identity():
    g = synth.rng(21)
    parent, _ = W.trees(g, 1, 60, 5, 100)
    r = prune.prune_tree(parent[0], np.ones(60), 60, 10)
    assert r["old_to_new"].tolist() == list(range(60))
    assert r["new_parent"].tolist() == parent[0].tolist()


def test_random_trees_satisfy_both_constraints_and_stay_prefix_closed():
    g = synth.rng(22)
    for _ in range(40):
        n = int(g.integers(2, 80))
        parent, _ = W.trees(g, 1, n, int(g.integers(1, 12)), 1000)
        conf = g.random(n).astype(np.float32)
        cap, lim = int(g.integers(1, 4)), int(g.integers(1, 6))
        r = prune.prune_tree(parent[0], conf, cap, lim)
        newp = r["new_parent"]
        tree.validate(newp)  # a valid tree: root first, parent < child
        assert max(np.bincount(newp[1:], minlength=len(newp)).max(initial=0), 0) <= cap
        assert tree.depth(newp).max() <= lim or all(  # no child to step into
            r["old_to_new"][c] == -1 for c in range(n) if parent[0][c] == r["root"])
        # every kept node's kept parent is its original parent
        inv = {v: int(r["old_to_new"][v]) for v in range(n) if r["old_to_new"][v] >= 0}
        for v, i in inv.items():
            if v != r["root"]:
                assert newp[i] == inv[int(parent[0][v])]
