"""Philox4x32-10 counter-based generator, written from its published definition.

Reference: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11 -- the Philox-4x32 bijection: each round
multiplies counter words 0 and 2 by two fixed odd constants, keeps the 64-bit
products' high and low halves, mixes the high halves with the other two counter
words and the key, and permutes; the 2-word key is bumped by two Weyl constants
between rounds; 10 rounds.

The FORGE summary asks for stochastic rounding of the weight write-back (§2
Precision and fidelity, second low-precision point) but names no generator.  We
read the RNG as Philox4x32-10 keyed by the seed, with the counter made from the
element index and the optimizer step -- see ``sr_bits``.

Pinned by: a published known-answer vector, bijectivity on a sampled counter
set, and uniformity of the 16-bit outputs (tests/test_oracle_philox.py).
"""
from __future__ import annotations

import numpy as np

_MASK = np.uint64(0xFFFFFFFF)
# Multipliers and Weyl key increments of Philox-4x32 (Salmon et al., SC'11, Table 2 / §4).
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)
ROUNDS = 10


def philox4x32(ctr, key, rounds: int = ROUNDS) -> np.ndarray:
    """Philox4x32-R of counters ``ctr`` (shape (4, n), uint32) under ``key`` ((2,) or (2, n)).

    Returns a (4, n) uint32 array.
    """
    c = [np.asarray(w, dtype=np.uint64) & _MASK for w in ctr]
    k0 = np.asarray(key[0], dtype=np.uint64) & _MASK
    k1 = np.asarray(key[1], dtype=np.uint64) & _MASK
    for r in range(rounds):
        if r:
            k0 = (k0 + PHILOX_W0) & _MASK
            k1 = (k1 + PHILOX_W1) & _MASK
        p0 = PHILOX_M0 * c[0]          # < 2^64: exact in uint64
        p1 = PHILOX_M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack([w.astype(np.uint32) for w in c])


STREAM_W, STREAM_M, STREAM_V = 0, 1, 2


def sr_bits(seed: int, step: int, e, stream: int = STREAM_W) -> np.ndarray:
    """16 random bits for element ``e`` (row-major flat index) of tensor ``stream`` at optimizer
    step ``step``.

    Reading of the summary's unspecified stream (stated in the design notes):
      key     = (seed mod 2^32, seed div 2^32)
      counter = (j mod 2^32, (j div 2^32) + stream * 2^30, step mod 2^32, step div 2^32),
                j = e div 8; stream 0 is the weight, 1 and 2 the BF16 first and second moments
                (j div 2^32 < 2^30 for every layer the library accepts, so the streams never meet)
      element e takes output word (e div 2) mod 4, its low half when e is even and
      its high half when e is odd -- one Philox call serves 8 consecutive elements.
    """
    assert stream in (STREAM_W, STREAM_M, STREAM_V)
    e = np.asarray(e, dtype=np.uint64)
    j = e >> np.uint64(3)
    step = np.uint64(step)
    seed = np.uint64(seed)
    n = e.shape[0]
    ctr = np.stack([j & _MASK, (j >> np.uint64(32)) + np.uint64(stream << 30),
                    np.full(n, step & _MASK, dtype=np.uint64),
                    np.full(n, step >> np.uint64(32), dtype=np.uint64)])
    out = philox4x32(ctr, (seed & _MASK, seed >> np.uint64(32))).astype(np.uint64)
    word = ((e >> np.uint64(1)) & np.uint64(3)).astype(np.intp)
    chosen = out[word, np.arange(n)]
    shift = (e & np.uint64(1)) * np.uint64(16)
    return ((chosen >> shift) & np.uint64(0xFFFF)).astype(np.uint32)
