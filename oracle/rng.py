"""Counter-based random numbers for the stochastic re-encoding (oracle side).

Test infrastructure only; see the package docstring.

piper-offload docs, "LoRA merge": the stochastic re-encoding of a quantised merge draws its
samples from backend-local randomness keyed by a scalar seed, "keyed by logical element
index, so launch geometry does not change the result"; the pages name no generator and
promise no identical bytes across backends.  The one used on both sides here is
Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC 2011), written from that definition: a 128-bit counter
(four 32-bit words) and a 64-bit key (two words) go through ten rounds; a round multiplies
words 0 and 2 by the two Philox constants into 64-bit products, and the new words are
(high product of word 2) ^ word 1 ^ key 0, (low product of word 2), (high product of word 0)
^ word 3 ^ key 1, (low product of word 0); between rounds the key words advance by the two
Weyl constants (the golden ratio's and sqrt(3) - 1's 32-bit fractions).

The element stream: element e (its logical row-major index in the weight) takes word e % 4
of Philox(counter = (e // 4 as two 32-bit words, 0, 0), key = the seed's two 32-bit
words), and its uniform integer U = word >> 9 (23 bits).

Pinned by ``tests/test_oracle_stochastic.py`` through properties a correct generator of
this family has and a slip in it loses (no known-answer vectors are used): uniform bytes and
23-bit draws (chi-square), full avalanche of one flipped counter or key bit over the ten
rounds, no correlation between neighbouring counters, and a bijective round for a fixed key.
"""
from __future__ import annotations

import numpy as np

MUL0 = np.uint64(0xD2511F53)
MUL1 = np.uint64(0xCD9E8D57)
WEYL0 = np.uint32(0x9E3779B9)
WEYL1 = np.uint32(0xBB67AE85)
ROUNDS = 10
_MASK32 = np.uint64(0xFFFFFFFF)


def philox_round(c0, c1, c2, c3, k0, k1):
    """One round on uint32 arrays (broadcast); returns the four new words."""
    p0 = c0.astype(np.uint64) * MUL0
    p1 = c2.astype(np.uint64) * MUL1
    hi0, lo0 = (p0 >> np.uint64(32)).astype(np.uint32), (p0 & _MASK32).astype(np.uint32)
    hi1, lo1 = (p1 >> np.uint64(32)).astype(np.uint32), (p1 & _MASK32).astype(np.uint32)
    return hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0


def philox4x32(c0, c1, c2, c3, k0, k1, rounds: int = ROUNDS):
    """Philox4x32-`rounds` of counters (c0..c3) under keys (k0, k1), uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint32) for c in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint32)
    k1 = np.asarray(k1, dtype=np.uint32)
    with np.errstate(over="ignore"):
        for i in range(rounds):
            if i > 0:
                k0 = (k0 + WEYL0).astype(np.uint32)
                k1 = (k1 + WEYL1).astype(np.uint32)
            c0, c1, c2, c3 = philox_round(c0, c1, c2, c3, k0, k1)
    return c0, c1, c2, c3


def seed_words(seed: int):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return np.uint32(seed & 0xFFFFFFFF), np.uint32(seed >> 32)


def element_uniform23(e: np.ndarray, seed: int) -> np.ndarray:
    """U (uint32 in [0, 2^23)) of the logical elements e (int64 array) under `seed`."""
    e = np.asarray(e, dtype=np.int64)
    q = (e >> 2).astype(np.uint64)
    k0, k1 = seed_words(seed)
    c0 = (q & _MASK32).astype(np.uint32)
    c1 = (q >> np.uint64(32)).astype(np.uint32)
    z = np.zeros_like(c0)
    w = philox4x32(c0, c1, z, z, k0, k1)
    word = np.choose((e & 3).astype(np.int64), w)
    return (word >> np.uint32(9)).astype(np.uint32)
