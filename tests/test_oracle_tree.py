"""Pins for oracle.tree against PTD §3.1 (observable set pi(v), position from |pi(v)|)."""
import numpy as np
import pytest

from oracle import tree


# hand-built tree:      0
#                     /   \
#                    1     2
#                   / \     \
#                  3   4     5
#                      |
#                      6
PARENT = [-1, 0, 0, 1, 1, 2, 4]


def test_observable_sets_by_hand():
    expect = {0: {0}, 1: {0, 1}, 2: {0, 2}, 3: {0, 1, 3}, 4: {0, 1, 4}, 5: {0, 2, 5}, 6: {0, 1, 4, 6}}
    for v, s in expect.items():
        assert set(tree.observable_set(PARENT, v)) == s


def test_depth_and_positions_by_hand():
    assert tree.depth(PARENT).tolist() == [0, 1, 1, 2, 2, 2, 3]
    assert tree.position_ids(PARENT, 100).tolist() == [100, 101, 101, 102, 102, 102, 103]


def test_chain_positions_are_causal_positions():
    n, p = 9, 17
    par = list(range(-1, n - 1))
    assert tree.position_ids(par, p).tolist() == list(range(p, p + n))
    vis = tree.visibility(par)
    assert np.array_equal(vis, np.tril(np.ones((n, n), dtype=bool)))


def test_star_sees_root_and_self():
    n = 6
    par = [-1] + [0] * (n - 1)
    vis = tree.visibility(par)
    for i in range(1, n):
        assert set(np.nonzero(vis[i])[0].tolist()) == {0, i}


def test_packed_mask_bits():
    par = list(range(-1, 39))  # chain of 40 -> 2 words per row
    m = tree.packed_mask(par)
    assert m.shape == (40, 2)
    assert m[0].tolist() == [1, 0]
    assert m[31].tolist() == [0xFFFFFFFF, 0]
    assert m[32].tolist() == [0xFFFFFFFF, 1]
    assert m[39].tolist() == [0xFFFFFFFF, 0xFF]


def test_children_csr():
    off, idx = tree.child_csr(PARENT)
    assert off.tolist() == [0, 2, 4, 5, 5, 6, 6, 6]
    assert idx.tolist() == [1, 2, 3, 4, 5, 6]


@pytest.mark.parametrize("bad", [[0, 0], [-1, 1], [-1, 0, 3, 1], [-1, -1, 0], [-1, 0, -1, 1], []])
def test_rejects_malformed(bad):
    # [-1, -1, 0] and [-1, 0, -1, 1]: an active row after a padding row
    with pytest.raises(ValueError):
        tree.validate(bad)


def _padded(parent, n_total):
    return np.concatenate([np.asarray(parent, dtype=np.int32), np.full(n_total - len(parent), -1, np.int32)])


@pytest.mark.parametrize("n,n_total", [(1, 4), (10, 16), (33, 64), (40, 40)])
def test_trailing_padding_rows_are_inactive(n, n_total):
    # a ragged batch pads a sequence's tree with parent -1 rows: the active rows keep the
    # unpadded tree's depth, positions, mask bits and children; padding rows get none
    g = np.random.default_rng(n + n_total)
    par = [-1] + [int(g.integers(i)) for i in range(1, n)]
    pad = _padded(par, n_total)
    tree.validate(pad)
    assert tree.active_count(pad) == n
    d0, dp = tree.depth(par), tree.depth(pad)
    assert dp[:n].tolist() == d0.tolist() and (dp[n:] == -1).all()
    pp = tree.position_ids(pad, 100)
    assert pp[:n].tolist() == (100 + d0).tolist() and (pp[n:] == -1).all()
    m0, mp = tree.packed_mask(par), tree.packed_mask(pad)
    assert (mp[n:] == 0).all()
    assert (mp[:n, :m0.shape[1]] == m0).all() and (mp[:n, m0.shape[1]:] == 0).all()
    assert tree.children(pad)[:n] == tree.children(par) and all(not c for c in tree.children(pad)[n:])
    off, idx = tree.child_csr(pad)
    assert off[n:].tolist() == [n - 1] * (n_total + 1 - n) and idx.tolist() == tree.child_csr(par)[1].tolist()
