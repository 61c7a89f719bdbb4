"""Tree-masked grouped-query attention (oracle, float64).

What it restates
  * PTD §3.1 "tree construction": node v attends only to its observable prefix set
    pi(v) = {v} U pi(P(v)).
  * Speculative-decoding blog, section "why target verification can be parallel": the
    target scores every drafted position in one forward pass, each position seeing the
    committed context plus the drafted tokens to its left (causal mask); a tree replaces
    "to its left" by "its ancestors".
  * TAPS §4.1: the selected subtree is verified by the target with tree attention.

Readings (not fixed by the pages)
  * Layout: q, out [B][Hq][N][D]; k_cache, v_cache [B][Hkv][S][D] with S >= P + N; cache
    rows 0..P-1 are the committed prefix and row P + t holds tree node t's key/value.
  * Grouped-query attention: query head h reads KV head h // (Hq / Hkv).
  * Scale 1/sqrt(D) unless given; softmax over the visible keys only.
  * Node i's visible keys are rows [0, P) and {P + t : t in pi(i)}.
  * Padding rows of a ragged batch (parent -1 after the last node, see tree.py) have no
    output; their rows of the result stay zero.
"""
from __future__ import annotations

import math

import numpy as np

from .tree import is_padding, observable_set, root_path, validate


def _softmax_attend(qvec: np.ndarray, keys: np.ndarray, vals: np.ndarray, scale: float) -> np.ndarray:
    s = (keys @ qvec) * scale
    s = s - s.max()
    w = np.exp(s)
    w = w / w.sum()
    return w @ vals


def tree_attention(q, k_cache, v_cache, parent, prefix_len: int, scale: float | None = None,
                   nodes=None, heads=None) -> np.ndarray:
    """out[b,h,i,:] = softmax over visible j of (q[b,h,i] . k[b,h//G,j]) * scale, applied to v.

    ``parent`` is [B][N].  Everything is promoted to float64.  ``nodes`` / ``heads``
    optionally restrict the computation to those indices (other rows stay zero).
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    bsz, hq, n, d = q.shape
    hkv = k_cache.shape[1]
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros_like(q)
    for b in range(bsz):
        validate(parent[b])
        for i in (range(n) if nodes is None else nodes):
            if is_padding(parent[b], i):
                continue
            anc = sorted(observable_set(parent[b], i))
            rows = list(range(prefix_len)) + [prefix_len + t for t in anc]
            for h in (range(hq) if heads is None else heads):
                kh = h // group
                out[b, h, i] = _softmax_attend(q[b, h, i], k_cache[b, kh, rows], v_cache[b, kh, rows], scale)
    return out


def causal_attention(q_seq, k_seq, v_seq, scale: float) -> np.ndarray:
    """Textbook causal attention over ONE sequence, written as a full score matrix.

    q_seq [Lq][D] are the queries of the LAST Lq positions of a sequence of length L
    (k_seq, v_seq [L][D]); query t (absolute position L - Lq + t) sees keys 0..L-Lq+t.
    This is an independent formulation used to pin ``tree_attention`` on chain trees.
    """
    q_seq = np.asarray(q_seq, dtype=np.float64)
    k_seq = np.asarray(k_seq, dtype=np.float64)
    v_seq = np.asarray(v_seq, dtype=np.float64)
    lq = q_seq.shape[0]
    total = k_seq.shape[0]
    scores = (q_seq @ k_seq.T) * scale
    pos_q = np.arange(total - lq, total)[:, None]
    pos_k = np.arange(total)[None, :]
    scores = np.where(pos_k <= pos_q, scores, -np.inf)
    scores = scores - scores.max(axis=1, keepdims=True)
    w = np.exp(scores)
    w = w / w.sum(axis=1, keepdims=True)
    return w @ v_seq


def per_node_bruteforce(q, k_cache, v_cache, parent, prefix_len: int, b: int, h: int, i: int,
                        scale: float | None = None) -> np.ndarray:
    """Build node i's explicit sequence (prefix ++ root..i path, by walking parent
    pointers) and run single-query attention over all of it."""
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    d = q.shape[3]
    group = q.shape[1] // k_cache.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    path = root_path(parent[b], i)
    rows = list(range(prefix_len)) + [prefix_len + t for t in path]
    kh = h // group
    # plain scalar loops, sharing nothing with tree_attention's vectorised softmax
    logits = [float(np.dot(q[b, h, i], k_cache[b, kh, r])) * scale for r in rows]
    top = max(logits)
    weights = [math.exp(x - top) for x in logits]
    total = math.fsum(weights)
    out = np.zeros(d)
    for w, r in zip(weights, rows):
        out += (w / total) * v_cache[b, kh, r]
    return out
