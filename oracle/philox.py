"""Philox4x32-10 and the verify step's uniform draws (oracle side).

Test infrastructure only (see the package docstring).

Philox4x32-10 follows the published definition (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11): a 128-bit counter of
four 32-bit words and a 64-bit key of two words; ten rounds, each multiplying
words 0 and 2 by two fixed 32-bit constants and mixing the high halves with
the other words and the key; the key is bumped by two Weyl constants between
rounds.

Stream layout used by the verify step (the pages fix only that r and u are
uniform on [0, 1]; this layout is the reading both the oracle and the CUDA
library implement):

* key     = (seed mod 2^32, seed >> 32)
* counter = (b, i, purpose, 0): sequence b, draft position i, purpose
  ACCEPT (0) for the acceptance draw r_i, SAMPLE (1) for the replacement /
  bonus draw at the position where it happens.
* k = (output word 0) >> 8, a 24-bit integer, so the value is exact in fp32.
* r = (k + 1) / 2^24 in (0, 1]  -- acceptance ("r <= p/q" keeps the draft).
* u = k / 2^24 in [0, 1)        -- inverse-CDF position for sampling.
"""
from __future__ import annotations

import numpy as np

MASK32 = 0xFFFFFFFF

# Round multipliers and key increments of Philox4x32 (Salmon et al. 2011).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10

PURPOSE_ACCEPT = 0
PURPOSE_SAMPLE = 1

TWO_M24 = 2.0 ** -24


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Apply Philox4x32-10 to counters (c0..c3) under key (k0, k1).

    All arguments are integers or integer arrays holding values in
    [0, 2^32); they broadcast together. Returns four uint64 arrays with the
    four 32-bit output words.
    """
    c0, c1, c2, c3, k0, k1 = (np.asarray(x, dtype=np.uint64) & np.uint64(MASK32)
                              for x in (c0, c1, c2, c3, k0, k1))
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    w0 = np.uint64(PHILOX_W0)
    w1 = np.uint64(PHILOX_W1)
    mask = np.uint64(MASK32)
    s32 = np.uint64(32)
    for rnd in range(PHILOX_ROUNDS):
        if rnd > 0:
            k0 = (k0 + w0) & mask
            k1 = (k1 + w1) & mask
        prod0 = m0 * c0          # < 2^64: exact in uint64
        prod1 = m1 * c2
        hi0, lo0 = prod0 >> s32, prod0 & mask
        hi1, lo1 = prod1 >> s32, prod1 & mask
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def uniform24(seed: int, b, i, purpose: int):
    """The 24-bit integer k for (seed, sequence b, position i, purpose)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    w0, _, _, _ = philox4x32_10(b, i, purpose, 0, seed & MASK32, seed >> 32)
    return w0 >> np.uint64(8)


def accept_uniform(seed: int, b, i):
    """r_i in (0, 1] for the acceptance test at draft position i."""
    k = uniform24(seed, b, i, PURPOSE_ACCEPT)
    return (k.astype(np.float64) + 1.0) * TWO_M24


def sample_uniform(seed: int, b, i):
    """u in [0, 1) for the replacement or bonus draw made at position i."""
    k = uniform24(seed, b, i, PURPOSE_SAMPLE)
    return k.astype(np.float64) * TWO_M24
