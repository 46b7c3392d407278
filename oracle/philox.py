"""Philox4x32-10, written from its published definition.

TEST INFRASTRUCTURE ONLY.  Reference: J. K. Salmon, M. A. Moraes, R. O. Dror,
D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11, section 4
(the Philox S-box: two 32x32->64 multiplies per round, the Weyl key schedule,
N=4 words of W=32 bits, 10 rounds).

The sampler draws one Philox block per (output row, round).  The mapping of the
pages' "seed + offset, advanced on every call" and "independent stream per output
instance" ([explainer] seed/offset and RNG ownership sections) onto counter and
key is this library's reading:
    key     = (seed & 0xffffffff, seed >> 32)
    counter = (round, output_row, offset & 0xffffffff, offset >> 32)
    u       = (word0 >> 8) * 2**-24          (24 random bits, exact in float32)
"""
from __future__ import annotations

import numpy as np

MASK = 0xFFFFFFFF
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85


def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: 4 counter words, 2 key words -> 4 output words."""
    x0, x1, x2, x3 = (int(c) & MASK for c in ctr)
    k0, k1 = (int(k) & MASK for k in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & MASK
            k1 = (k1 + PHILOX_W1) & MASK
        p0 = PHILOX_M0 * x0
        p1 = PHILOX_M1 * x2
        hi0, lo0 = p0 >> 32, p0 & MASK
        hi1, lo1 = p1 >> 32, p1 & MASK
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return (x0, x1, x2, x3)


def philox4x32_10_np(ctr: np.ndarray, key: np.ndarray) -> np.ndarray:
    """Vectorised form over rows of ``ctr`` [n,4] and ``key`` [n,2] (uint32)."""
    x = [np.asarray(ctr[:, i], dtype=np.uint64) for i in range(4)]
    k0 = np.asarray(key[:, 0], dtype=np.uint64)
    k1 = np.asarray(key[:, 1], dtype=np.uint64)
    m = np.uint64(MASK)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & m
            k1 = (k1 + np.uint64(PHILOX_W1)) & m
        p0 = np.uint64(PHILOX_M0) * x[0]
        p1 = np.uint64(PHILOX_M1) * x[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & m
        hi1, lo1 = p1 >> np.uint64(32), p1 & m
        x = [hi1 ^ x[1] ^ k0, lo1, hi0 ^ x[3] ^ k1, lo0]
    return np.stack(x, axis=1).astype(np.uint32)


def sampler_counter(seed: int, offset: int, row: int, rnd: int):
    """(counter, key) of the block drawn by output row ``row`` in round ``rnd``."""
    ctr = (rnd, row, offset & MASK, (offset >> 32) & MASK)
    key = (seed & MASK, (seed >> 32) & MASK)
    return ctr, key


def uniform_from_word(w: int) -> float:
    """Top 24 bits of a 32-bit word as a float in [0, 1)."""
    return float((int(w) & MASK) >> 8) * 2.0 ** -24


def sampler_uniform(seed: int, offset: int, row: int, rnd: int) -> float:
    ctr, key = sampler_counter(seed, offset, row, rnd)
    return uniform_from_word(philox4x32_10(ctr, key)[0])
