"""Committing the accepted path's keys and values (oracle).

What it restates
  * Speculative-decoding blog, "KV cache handling": verifying the drafted tokens writes
    a cache entry for every candidate; the entries of accepted tokens are kept in the
    target cache, those of rejected candidates (and everything after a rejection) are
    dropped, so that the next round continues from the accepted context only.

Readings (not fixed by the pages)
  * Layout as in ``attention``: cache rows [0, P) are the committed prefix, row P + t
    holds tree node t, the root (node 0, the last committed token) sits at row P.
  * A round accepts a root path a_1, ..., a_L (parent[a_1] = 0, parent[a_k] = a_{k-1}).
    Committing it moves node a_k's row to row P + k, so that rows [0, P + L] become the
    cache of the plain sequence prefix, root, a_1, ..., a_L.  Rows outside
    [P + 1, P + L] keep their contents.
"""
from __future__ import annotations

import numpy as np

from .tree import validate


def check_path(parent, accepted, length: int) -> None:
    """Raise unless accepted[:length] is a root path of the tree."""
    validate(parent)
    prev = 0
    for k in range(length):
        a = int(accepted[k])
        if not (0 < a < len(parent)) or int(parent[a]) != prev:
            raise ValueError(f"accepted[{k}] = {a} does not continue the root path")
        prev = a


def commit_accepted(k_cache, v_cache, parent, accepted, accept_len, prefix_len: int):
    """Return copies of the caches with each sequence's accepted path compacted.

    k_cache, v_cache [B][Hkv][S][D]; parent [B][N]; accepted [B][N] (node ids, then
    padding); accept_len [B].
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    for b in range(k_out.shape[0]):
        length = int(accept_len[b])
        check_path(parent[b], accepted[b], length)
        for k in range(1, length + 1):
            src = prefix_len + int(accepted[b][k - 1])
            k_out[b, :, prefix_len + k, :] = k_cache[b, :, src, :]
            v_out[b, :, prefix_len + k, :] = v_cache[b, :, src, :]
    return k_out, v_out
