"""Per-node vocabulary statistics (oracle, float64).

What it restates (speculative-decoding blog: "greedy decoding, intuitive version" and
"acceptance probability for sampling"): for every drafted position the target yields a
distribution p_i over the vocabulary; greedy verification compares the draft token with
the target's most likely token, sampling verification needs p_i(y_i), the target
probability of the drafted token under the same prefix.

Readings
  * Row u of the logits is the target distribution for the token that follows node u,
    so draft node c (c >= 1) is judged with row parent(c).
  * Temperature T divides the logits: p = softmax(x / T).
  * argmax compares the raw logit values and returns the lowest index among ties.
"""
from __future__ import annotations

import math

import numpy as np


def row_stats(x_row, temperature: float = 1.0):
    """(max of x/T, log-sum-exp of x/T, argmax) for one row, in float64."""
    z = np.asarray(x_row, dtype=np.float64) / temperature
    m = float(z.max())
    lse = m + math.log(float(np.exp(z - m).sum()))
    return m, lse, int(np.argmax(np.asarray(x_row)))  # numpy argmax: first maximal index


def vocab_stats(logits, temperature: float = 1.0):
    """For a [N][V] block: arrays (max, lse, argmax) per row."""
    logits = np.asarray(logits)
    n = logits.shape[0]
    m = np.empty(n)
    lse = np.empty(n)
    am = np.empty(n, dtype=np.int64)
    for u in range(n):
        m[u], lse[u], am[u] = row_stats(logits[u], temperature)
    return m, lse, am


def drafted_token_prob(logits, lse, parent, tokens, temperature: float = 1.0) -> np.ndarray:
    """p_c = softmax(x[parent(c)] / T)[tok c] = exp(x[parent(c)][tok c] / T - lse[parent(c)]).

    Entry 0 (the root, not a draft) and padding rows (parent -1) are NaN.
    """
    n = len(parent)
    out = np.full(n, np.nan)
    for c in range(1, n):
        u = int(parent[c])
        if u < 0:
            continue
        out[c] = math.exp(float(logits[u][int(tokens[c])]) / temperature - float(lse[u]))
    return out
