"""Philox4x32-10 counter-based generator (oracle copy).

Written from the published definition: J. K. Salmon, M. A. Moraes, R. O. Dror,
D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11, Philox-4x32 with
10 rounds.  Each round multiplies words 0 and 2 by the two Philox multipliers, takes
(hi, lo) halves of the 64-bit products, and mixes the other two words and the round
key in with XOR; the key is bumped by the two Weyl constants between rounds.

Use in verification (reading; the pages require reproducible random acceptance but fix
no generator): key = the 64-bit seed split into (low, high) 32-bit words; counter =
(round mod 2^32, sequence b, node u, 2*k + kind); the uniform is (x0 >> 8) * 2^-24,
exactly representable in fp32 and in [0, 1).
"""
from __future__ import annotations

import numpy as np

MUL0 = 0xD2511F53
MUL1 = 0xCD9E8D57
WEYL0 = 0x9E3779B9
WEYL1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """counter: (..., 4) uint32-like, key: (2,) uint32-like.  Returns (..., 4) uint32."""
    c = np.asarray(counter, dtype=np.uint64).copy()
    k0 = np.uint64(int(key[0]) & MASK32)
    k1 = np.uint64(int(key[1]) & MASK32)
    m0 = np.uint64(MUL0)
    m1 = np.uint64(MUL1)
    mask = np.uint64(MASK32)
    sh = np.uint64(32)
    for rnd in range(10):
        if rnd > 0:
            k0 = np.uint64((int(k0) + WEYL0) & MASK32)
            k1 = np.uint64((int(k1) + WEYL1) & MASK32)
        prod0 = m0 * c[..., 0]          # < 2^64, exact in uint64
        prod1 = m1 * c[..., 2]
        hi0, lo0 = prod0 >> sh, prod0 & mask
        hi1, lo1 = prod1 >> sh, prod1 & mask
        n0 = hi1 ^ c[..., 1] ^ k0
        n2 = hi0 ^ c[..., 3] ^ k1
        c[..., 0] = n0
        c[..., 1] = lo1
        c[..., 2] = n2
        c[..., 3] = lo0
    return c.astype(np.uint32)


def seed_key(seed: int):
    return (seed & MASK32, (seed >> 32) & MASK32)


def counter(rnd: int, b: int, u: int, k: int, kind: int):
    return (rnd & MASK32, b & MASK32, u & MASK32, (2 * k + kind) & MASK32)


def uniform(seed: int, rnd: int, b: int, u: int, k: int, kind: int) -> float:
    """U in [0, 1) for the draw (round, b, u, k, kind); 24 significant bits."""
    x0 = int(philox4x32_10(np.array(counter(rnd, b, u, k, kind)), seed_key(seed))[0])
    return (x0 >> 8) * (1.0 / 16777216.0)
