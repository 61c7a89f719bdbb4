"""Seeded synthetic inputs for the tree-verification path.

This module only *makes data*: random draft trees, random Q/K/V, random logits,
candidate pools and the planting of a target argmax.  It computes nothing that the
verification method computes (no attention, no log-sum-exp, no acceptance test, no
path scores, no selection).  Both the CUDA library's tests/bench and the CPU oracle
are fed from here, and from nowhere else.

Every generator takes a ``numpy.random.Generator`` (PCG64, ``np.random.default_rng``)
so that a (seed, recipe) pair names the bytes exactly.

bf16 data is produced as float32 arrays whose values are exactly representable in
bfloat16 (round-to-nearest-even of an fp32 draw), plus the raw uint16 bit patterns,
so that the oracle (fp64) and the GPU (bf16) read the very same numbers.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng",
    "round_to_bf16",
    "bf16_bits",
    "random_parents",
    "chain_parents",
    "star_parents",
    "distinct_child_tokens",
    "normal",
    "plant_first_child_argmax",
    "marginal_pool",
    "draw_children_from_draft",
    "first_children",
]


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    bias = ((bits >> 16) & 1) + 0x7FFF
    out = (((bits + bias) >> 16) << 16).astype(np.uint32)
    return out.view(np.float32).reshape(x.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("values are not bf16-exact; call round_to_bf16 first")
    return (bits >> 16).astype(np.uint16)


def chain_parents(n: int) -> np.ndarray:
    """parent = [-1, 0, 1, ..., n-2]: a single draft sequence."""
    p = np.arange(-1, n - 1, dtype=np.int32)
    return p


def star_parents(n: int) -> np.ndarray:
    """Every draft node hangs off the root."""
    p = np.zeros(n, dtype=np.int32)
    p[0] = -1
    return p


def random_parents(g: np.random.Generator, n: int, depth_cap: int) -> np.ndarray:
    """Random rooted tree on nodes 0..n-1 with parent[i] < i.

    parent[i] is drawn uniformly from the earlier nodes whose depth is below
    ``depth_cap`` (so no node is deeper than ``depth_cap`` edges from the root).
    """
    if n < 1:
        raise ValueError("a tree has at least its root")
    parent = np.empty(n, dtype=np.int32)
    level = np.empty(n, dtype=np.int64)
    parent[0] = -1
    level[0] = 0
    open_nodes = [0] if depth_cap > 0 else []
    for i in range(1, n):
        if not open_nodes:
            raise ValueError("depth_cap 0 allows only the root")
        j = open_nodes[int(g.integers(len(open_nodes)))]
        parent[i] = j
        level[i] = level[j] + 1
        if level[i] < depth_cap:
            open_nodes.append(i)
    return parent


def first_children(parent: np.ndarray) -> np.ndarray:
    """For each node, its lowest-index child (or -1)."""
    n = len(parent)
    fc = np.full(n, -1, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        fc[parent[i]] = i
    return fc


def distinct_child_tokens(g: np.random.Generator, parent: np.ndarray, vocab: int) -> np.ndarray:
    """Token per node; siblings get distinct tokens, uniform over [0, vocab)."""
    n = len(parent)
    tok = np.empty(n, dtype=np.int32)
    tok[0] = int(g.integers(vocab))
    kids: dict[int, list[int]] = {}
    for i in range(1, n):
        kids.setdefault(int(parent[i]), []).append(i)
    for u, cs in kids.items():
        if len(cs) > vocab:
            raise ValueError("more children than vocabulary entries")
        draw = g.choice(vocab, size=len(cs), replace=False)
        for c, t in zip(cs, draw):
            tok[c] = int(t)
    return tok


def normal(g: np.random.Generator, shape, std: float = 1.0, bf16: bool = False) -> np.ndarray:
    x = (g.standard_normal(shape) * std).astype(np.float32)
    return round_to_bf16(x) if bf16 else x


def plant_first_child_argmax(g: np.random.Generator, logits: np.ndarray, parent: np.ndarray,
                             tokens: np.ndarray, prob: float, bf16: bool) -> np.ndarray:
    """With probability ``prob``, make the first child's token the row's strict maximum.

    ``logits`` is [N][V] (one sequence); row u is the target distribution for the
    token after node u, so the planted entry is x[u][tok(first child of u)] = max(x[u]) + 1.
    """
    out = np.array(logits, dtype=np.float32, copy=True)
    fc = first_children(parent)
    for u in range(len(parent)):
        if fc[u] < 0:
            continue
        if g.random() < prob:
            val = np.float32(out[u].max() + np.float32(1.0))
            if bf16:
                val = round_to_bf16(np.array([val], dtype=np.float32))[0]
            out[u, tokens[fc[u]]] = val
    return out


def marginal_pool(g: np.random.Generator, d: int, k: int, vocab: int, std: float = np.sqrt(2.0)):
    """Block-marginal candidate pool: d positions x top-k (probability, token).

    Each position's k probabilities are a softmax of N(0, std^2) draws (the drafter's
    per-position marginal restricted to its top-k), rounded to fp32, and sorted by
    (probability desc, token asc).  Tokens are distinct within a position.
    Returns (marg float32 [d][k], tok int32 [d][k]).
    """
    z = g.standard_normal((d, k)) * std
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    prob = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    tok = np.stack([g.choice(vocab, size=k, replace=False) for _ in range(d)]).astype(np.int32)
    marg = np.empty_like(prob)
    ptok = np.empty_like(tok)
    for r in range(d):
        order = sorted(range(k), key=lambda j: (-float(prob[r, j]), int(tok[r, j])))
        marg[r] = prob[r, order]
        ptok[r] = tok[r, order]
    return marg, ptok


def draw_children_from_draft(g: np.random.Generator, parent: np.ndarray, draft_logits: np.ndarray,
                             temperature: float) -> np.ndarray:
    """Stand-in drafter: each node's children take tokens drawn without replacement
    from the draft distribution of that node's row, softmax(draft_logits[u] / T).
    The root keeps a uniformly drawn token.
    """
    n, vocab = draft_logits.shape
    tok = np.empty(n, dtype=np.int32)
    tok[0] = int(g.integers(vocab))
    kids: dict[int, list[int]] = {}
    for i in range(1, n):
        kids.setdefault(int(parent[i]), []).append(i)
    for u, cs in kids.items():
        z = draft_logits[u].astype(np.float64) / temperature
        w = np.exp(z - z.max())
        w /= w.sum()
        draw = g.choice(vocab, size=len(cs), replace=False, p=w)
        for c, t in zip(cs, draw):
            tok[c] = int(t)
    return tok
