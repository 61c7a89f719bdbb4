"""Pins of oracle.kvcommit (CPU)."""
import numpy as np
import pytest

import synth
from oracle import attention, kvcommit


def _cache(g, B, Hkv, S, D):
    return synth.normal(g, (B, Hkv, S, D)), synth.normal(g, (B, Hkv, S, D))


def test_chain_path_is_identity():
    g = synth.rng(7)
    k, v = _cache(g, 1, 2, 12, 8)
    parent = np.array([[-1, 0, 1, 2, 3]])
    k2, v2 = kvcommit.commit_accepted(k, v, parent, np.array([[1, 2, 3, 4, -1]]), [4], 7)
    assert np.array_equal(k2, k) and np.array_equal(v2, v)


def test_hand_built_branch():
    # tree: 0 -> {1, 2}, 2 -> {3}, 3 -> {4}; accepted path 2, 3, 4 (node 1 rejected)
    g = synth.rng(8)
    P = 5
    k, v = _cache(g, 1, 1, P + 5, 4)
    parent = np.array([[-1, 0, 0, 2, 3]])
    k2, v2 = kvcommit.commit_accepted(k, v, parent, np.array([[2, 3, 4, -1, -1]]), [3], P)
    assert np.array_equal(k2[0, 0, P + 1], k[0, 0, P + 2])
    assert np.array_equal(k2[0, 0, P + 2], k[0, 0, P + 3])
    assert np.array_equal(v2[0, 0, P + 3], v[0, 0, P + 4])
    assert np.array_equal(k2[0, 0, :P + 1], k[0, 0, :P + 1])  # prefix and root untouched
    assert np.array_equal(k2[0, 0, P + 4:], k[0, 0, P + 4:])  # rows past the path untouched


def test_zero_accepted_changes_nothing():
    g = synth.rng(9)
    k, v = _cache(g, 2, 1, 10, 4)
    parent = np.array([[-1, 0, 0, 1], [-1, 0, 1, 1]])
    k2, v2 = kvcommit.commit_accepted(k, v, parent, np.full((2, 4), -1), [0, 0], 6)
    assert np.array_equal(k2, k) and np.array_equal(v2, v)


def test_rejects_non_paths():
    parent = np.array([-1, 0, 0, 2])
    with pytest.raises(ValueError):
        kvcommit.check_path(parent, [1, 3], 2)  # 3 is a child of 2, not of 1
    with pytest.raises(ValueError):
        kvcommit.check_path(parent, [3], 1)  # does not start at a child of the root
    kvcommit.check_path(parent, [2, 3], 2)


def test_committed_cache_is_the_causal_cache_of_the_path():
    """Tree attention of the path's last node over (prefix + its ancestors) equals plain
    causal attention over the committed rows [0, P + L]: the compaction lays the path out
    as an ordinary sequence."""
    g = synth.rng(10)
    B, Hq, Hkv, D, P, N = 1, 4, 2, 16, 6, 9
    parent = np.array([[-1, 0, 0, 1, 2, 4, 4, 6, 3]])
    path = [2, 4, 6, 7]  # root -> 2 -> 4 -> 6 -> 7
    q = synth.normal(g, (B, Hq, N, D))
    k, v = _cache(g, B, Hkv, P + N, D)
    k2, v2 = kvcommit.commit_accepted(k, v, parent, np.array([path + [-1] * (N - 4)]), [4], P)
    L = len(path)
    tree = attention.tree_attention(q, k, v, parent, P, nodes=[path[-1]])
    scale = 1.0 / np.sqrt(D)
    for h in range(Hq):
        kh = h // (Hq // Hkv)
        seq_q = np.zeros((P + L + 1, D))
        seq_q[-1] = q[0, h, path[-1]]
        causal = attention.causal_attention(seq_q, k2[0, kh, :P + L + 1], v2[0, kh, :P + L + 1], scale)
        np.testing.assert_allclose(tree[0, h, path[-1]], causal[-1], rtol=1e-12, atol=1e-12)
