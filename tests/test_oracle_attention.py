"""Pins for oracle.attention: chain == textbook causal attention, per-node brute force
over the explicit root->node sequence, star trees, relabelling, closed forms."""
import math

import numpy as np
import pytest

import synth
from oracle import attention, tree


def _data(seed, b, hq, hkv, n, d, p, extra=0):
    g = synth.rng(seed)
    q = g.standard_normal((b, hq, n, d))
    k = g.standard_normal((b, hkv, p + n + extra, d))
    v = g.standard_normal((b, hkv, p + n + extra, d))
    return q, k, v


@pytest.mark.parametrize("hq,hkv", [(4, 1), (6, 2)])
def test_chain_equals_causal(hq, hkv):
    b, n, d, p = 2, 7, 16, 11
    q, k, v = _data(1, b, hq, hkv, n, d, p)
    par = np.stack([synth.chain_parents(n)] * b)
    out = attention.tree_attention(q, k, v, par, p)
    scale = 1 / math.sqrt(d)
    g = hq // hkv
    for bb in range(b):
        for h in range(hq):
            ref = attention.causal_attention(q[bb, h], k[bb, h // g, : p + n], v[bb, h // g, : p + n], scale)
            np.testing.assert_allclose(out[bb, h], ref, rtol=1e-12, atol=1e-12)


def test_matches_per_node_bruteforce():
    b, hq, hkv, n, d, p = 2, 4, 2, 13, 8, 5
    q, k, v = _data(2, b, hq, hkv, n, d, p, extra=3)
    g = synth.rng(3)
    par = np.stack([synth.random_parents(g, n, 4) for _ in range(b)])
    out = attention.tree_attention(q, k, v, par, p)
    for bb in range(b):
        for h in range(hq):
            for i in range(n):
                ref = attention.per_node_bruteforce(q, k, v, par, p, bb, h, i)
                np.testing.assert_allclose(out[bb, h, i], ref, rtol=1e-11, atol=1e-12)


def test_star_tree_rows():
    b, hq, hkv, n, d, p = 1, 2, 1, 6, 4, 3
    q, k, v = _data(4, b, hq, hkv, n, d, p)
    par = synth.star_parents(n)[None]
    out = attention.tree_attention(q, k, v, par, p)
    for h in range(hq):
        for i in range(1, n):
            rows = [0, 1, 2, p + 0, p + i]
            s = k[0, 0, rows] @ q[0, h, i] / 2.0
            w = np.exp(s - s.max())
            ref = (w / w.sum()) @ v[0, 0, rows]
            np.testing.assert_allclose(out[0, h, i], ref, rtol=1e-12)


def test_relabelling_permutes_outputs():
    # A different topological numbering of the same tree gives the same per-node outputs.
    n, d, p = 8, 8, 4
    g = synth.rng(5)
    par = synth.random_parents(g, n, 3)
    # relabel: order nodes by (depth, old index) -> still parent < child
    dep = tree.depth(par)
    order = sorted(range(n), key=lambda i: (dep[i], i))
    new_of = {old: new for new, old in enumerate(order)}
    par2 = np.array([-1] + [new_of[par[order[j]]] for j in range(1, n)], dtype=np.int32)
    q, k, v = _data(6, 1, 2, 1, n, d, p)
    q2 = q[:, :, order]
    k2 = k.copy()
    v2 = v.copy()
    k2[:, :, p:p + n] = k[:, :, [p + o for o in order]]
    v2[:, :, p:p + n] = v[:, :, [p + o for o in order]]
    o1 = attention.tree_attention(q, k, v, par[None], p)
    o2 = attention.tree_attention(q2, k2, v2, par2[None], p)
    np.testing.assert_allclose(o2, o1[:, :, order], rtol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    n, d, p = 5, 4, 3
    par = np.array([[-1, 0, 1, 0, 3]])
    _, k, v = _data(7, 1, 1, 1, n, d, p)
    q = np.zeros((1, 1, n, d))
    out = attention.tree_attention(q, k, v, par, p)
    # node 4 sees prefix rows 0..2 and tree nodes {0, 3, 4}
    rows = [0, 1, 2, p + 0, p + 3, p + 4]
    np.testing.assert_allclose(out[0, 0, 4], v[0, 0, rows].mean(axis=0), rtol=1e-12)


def test_root_alone_returns_its_value():
    d = 6
    q, k, v = _data(8, 1, 1, 1, 1, d, 0)
    out = attention.tree_attention(q, k, v, np.array([[-1]]), 0)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 0], rtol=1e-14)


def test_dominant_key_selects_its_value():
    n, d, p = 3, 4, 2
    par = np.array([[-1, 0, 1]])
    q = np.zeros((1, 1, n, d))
    k = np.zeros((1, 1, p + n, d))
    v = synth.rng(9).standard_normal((1, 1, p + n, d))
    q[0, 0, 2, 0] = 1.0
    k[0, 0, p + 1, 0] = 400.0  # node 1 is an ancestor of node 2
    out = attention.tree_attention(q, k, v, par, p, scale=1.0)
    np.testing.assert_allclose(out[0, 0, 2], v[0, 0, p + 1], rtol=1e-12)
    # a key that node 2 cannot see must not win, however large
    k[0, 0, p + 1, 0] = 0.0
    par2 = np.array([[-1, 0, 0]])
    k[0, 0, p + 1, 0] = 400.0
    out2 = attention.tree_attention(q, k, v, par2, p, scale=1.0)
    assert not np.allclose(out2[0, 0, 2], v[0, 0, p + 1])


def test_padded_rows_of_a_ragged_batch():
    # a tree of n nodes padded with parent -1 rows to N: active rows equal the unpadded
    # tree's attention (the padding keys at rows P + n.. are seen by nobody), padding
    # rows stay zero; the per-node brute force agrees on the active rows
    g = np.random.default_rng(77)
    n, N, P, Hq, Hkv, D = 9, 14, 20, 4, 2, 16
    par = np.array([-1] + [int(g.integers(i)) for i in range(1, n)], dtype=np.int32)
    pad = np.concatenate([par, np.full(N - n, -1, np.int32)])[None]
    q = g.standard_normal((1, Hq, N, D))
    k = g.standard_normal((1, Hkv, P + N, D))
    v = g.standard_normal((1, Hkv, P + N, D))
    got = attention.tree_attention(q, k, v, pad, P)
    ref = attention.tree_attention(q[:, :, :n], k[:, :, :P + n], v[:, :, :P + n], par[None], P)
    assert np.allclose(got[:, :, :n], ref, atol=1e-12) and (got[:, :, n:] == 0).all()
    for i in (0, n - 1):
        assert np.allclose(got[0, 1, i], attention.per_node_bruteforce(q, k, v, pad, P, 0, 1, i), atol=1e-12)
