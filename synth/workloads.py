"""Named synthetic workloads for tree verification (shapes of the pages' settings).

Each recipe states sizes, dtypes and the value distributions; ``N(0, 2)`` is read as
variance 2 (std sqrt 2).  Stand-ins: the pages evaluate on real models and unnamed
datasets that are not available here, so every tensor is a seeded random draw of the
same shape.  Nothing here computes any part of verification.

  tiny_fp32      B=1 fp32, Hq=4 / Hkv=1, D=64, prefix 128, 16-node tree (depth <= 4),
                 V=1024 logits N(0,2) with the first child's token planted as argmax
                 with probability 0.7; greedy.
  qwen3_4b_layer B=1 bf16, 32/8 heads, D=128, prefix 2048, 64-node tree selected from a
                 16 x top-4 block-marginal pool (budget 64), V=151936 planted logits;
                 greedy.
  sampling       B=4 bf16, 32/8, D=128, prefix 8192, 256-node trees depth <= 16,
                 target logits N(0,2), draft = target + N(0, 0.5^2), T = 1, child tokens
                 drawn without replacement from the draft distribution; sampling.
  long_context   B=8 bf16, 32/8, D=128, prefix 32768, 128-node trees depth <= 16,
                 planted logits; greedy.
  budget_sweep   B=16, pool 16 x top-32 (softmax of N(0,2)), budgets 16/64/256/1024,
                 verified with 32/8 heads, D=128, prefix 4096, planted logits; greedy.
"""
from __future__ import annotations

import math

import numpy as np

from . import (distinct_child_tokens, draw_children_from_draft, marginal_pool, normal,
               plant_first_child_argmax, random_parents, rng, round_to_bf16)

SQRT2 = math.sqrt(2.0)

WORKLOADS = {
    "tiny_fp32": dict(B=1, bf16=False, Hq=4, Hkv=1, D=64, P=128, N=16, V=1024, depth_cap=4,
                      mode="greedy", seed=1001),
    "qwen3_4b_layer": dict(B=1, bf16=True, Hq=32, Hkv=8, D=128, P=2048, N=64, V=151936, pool_d=16,
                           pool_k=4, mode="greedy", seed=1002),
    "sampling": dict(B=4, bf16=True, Hq=32, Hkv=8, D=128, P=8192, N=256, V=151936, depth_cap=16,
                     mode="sample", temperature=1.0, seed=1003),
    "long_context": dict(B=8, bf16=True, Hq=32, Hkv=8, D=128, P=32768, N=128, V=151936, depth_cap=16,
                         mode="greedy", seed=1004),
    "budget_sweep": dict(B=16, bf16=True, Hq=32, Hkv=8, D=128, P=4096, V=151936, pool_d=16, pool_k=32,
                         budgets=(16, 64, 256, 1024), mode="greedy", seed=1005),
}


def qkv_host(g, B, Hq, Hkv, D, P, N, bf16, extra_rows=0):
    """Q [B][Hq][N][D], K and V caches [B][Hkv][P+N+extra][D], all N(0, 1)."""
    q = normal(g, (B, Hq, N, D), 1.0, bf16)
    k = normal(g, (B, Hkv, P + N + extra_rows, D), 1.0, bf16)
    v = normal(g, (B, Hkv, P + N + extra_rows, D), 1.0, bf16)
    return q, k, v


def trees(g, B, N, depth_cap, V):
    parent = np.stack([random_parents(g, N, depth_cap) for _ in range(B)])
    tokens = np.stack([distinct_child_tokens(g, parent[b], V) for b in range(B)])
    return parent.astype(np.int32), tokens.astype(np.int32)


def planted_logits(g, parent, tokens, V, bf16, prob=0.7):
    """[B][N][V] N(0,2) logits; with probability ``prob`` the first child's token of
    each internal node is made the strict row maximum."""
    B, N = parent.shape
    out = np.empty((B, N, V), dtype=np.float32)
    for b in range(B):
        x = normal(g, (N, V), SQRT2, bf16)
        out[b] = plant_first_child_argmax(g, x, parent[b], tokens[b], prob, bf16)
    return out


def pools(g, B, d, K, V):
    marg = np.empty((B, d, K), dtype=np.float32)
    ptok = np.empty((B, d, K), dtype=np.int32)
    for b in range(B):
        marg[b], ptok[b] = marginal_pool(g, d, K, V)
    return marg, ptok


def sampling_logits(g, parent, V, bf16, temperature=1.0, noise=0.5):
    """Target N(0,2), draft = target + N(0, noise^2); child tokens drawn from the draft."""
    B, N = parent.shape
    tgt = normal(g, (B, N, V), SQRT2, False)
    drf = tgt + normal(g, (B, N, V), noise, False)
    if bf16:
        tgt = round_to_bf16(tgt)
        drf = round_to_bf16(drf)
    tokens = np.stack([draw_children_from_draft(g, parent[b], drf[b], temperature) for b in range(B)])
    return tgt.astype(np.float32), drf.astype(np.float32), tokens.astype(np.int32)


def device_normal(shape, std, seed, dtype, device):
    """Large N(0, std^2) tensors drawn on the GPU with torch's seeded generator (for sizes
    that would not fit a host-side draw); the oracle reads the same bytes back."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)
