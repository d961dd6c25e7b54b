"""Philox4x32-10 counter-based generator (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Written from the published definition: J. Salmon, M. Moraes, R. Dror,
D. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11, section on the
Philox family.  One round maps the 4-word counter (c0, c1, c2, c3) with key
(k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with the multipliers M0 = 0xD2511F53, M1 = 0xCD9E8D57; between rounds the key
is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85).  Ten rounds.

The verification method draws one uniform per decision ("r ~ Uniform(0, 1)",
exactness rule of "投机解码与 EAGLE").  Where the pages leave the generator
open we use: key = (seed low 32 bits, seed high 32 bits), counter =
(b, i, slot, offset) and u = (word0 >> 8) * 2^-24 in [0, 1).  This integer
formula is exact in float32 and float64, so both sides see identical u.

Slots: slot 0 = accept test of drafted token i, slot 1 = residual / bonus draw
at target row i.
"""

from __future__ import annotations

import numpy as np

MASK32 = 0xFFFFFFFF
M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85

SLOT_ACCEPT = 0
SLOT_SAMPLE = 1


def philox_round(c, k):
    """One Philox4x32 round on Python integers (exact)."""
    p0 = M0 * c[0]
    p1 = M1 * c[2]
    hi0, lo0 = p0 >> 32, p0 & MASK32
    hi1, lo1 = p1 >> 32, p1 & MASK32
    return (hi1 ^ c[1] ^ k[0], lo1, hi0 ^ c[3] ^ k[1], lo0)


def philox4x32_10(counter, key):
    """Ten rounds; returns four 32-bit words."""
    c = tuple(int(x) & MASK32 for x in counter)
    k0, k1 = (int(key[0]) & MASK32, int(key[1]) & MASK32)
    for _ in range(10):
        c = philox_round(c, (k0, k1))
        k0 = (k0 + W0) & MASK32
        k1 = (k1 + W1) & MASK32
    return c


def seed_key(seed: int):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return (seed & MASK32, seed >> 32)


def uniform(seed: int, b: int, i: int, slot: int, offset: int = 0) -> float:
    """u(b, i, slot) in [0, 1) with 24-bit resolution."""
    w = philox4x32_10((b, i, slot, offset), seed_key(seed))
    return float(w[0] >> 8) * (2.0 ** -24)


def philox4x32_10_np(c0, c1, c2, c3, seed: int):
    """Vectorised variant for Monte-Carlo tests (uint64 lanes, same rounds)."""
    m = np.uint64(MASK32)
    c = [np.asarray(x, dtype=np.uint64) & m for x in (c0, c1, c2, c3)]
    c = np.broadcast_arrays(*c)
    c = [x.copy() for x in c]
    k0, k1 = seed_key(seed)
    for _ in range(10):
        p0 = np.uint64(M0) * c[0]
        p1 = np.uint64(M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & m
        hi1, lo1 = p1 >> np.uint64(32), p1 & m
        c = [hi1 ^ c[1] ^ np.uint64(k0), lo1, hi0 ^ c[3] ^ np.uint64(k1), lo0]
        k0 = (k0 + W0) & MASK32
        k1 = (k1 + W1) & MASK32
    return c


def uniform_np(seed: int, b, i, slot, offset=0):
    w = philox4x32_10_np(b, i, slot, offset, seed)
    return (w[0] >> np.uint64(8)).astype(np.float64) * (2.0 ** -24)
