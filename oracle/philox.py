"""Philox-4x32-10 counter-based generator.

Test infrastructure (see ``oracle/__init__``).  Restated from Salmon, Moraes,
Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11),
section 3.3 (the Philox S-box built from one 32x32->64-bit multiply per
word pair) with the round multipliers and Weyl key increments given there
for the 4x32 variant, 10 rounds.

The method uses it in two places (format-aware fusion article, MXFP4 recipe):
the stochastic-rounding draw (key = the caller's seed, counter = the element
index) and the 32 fixed Hadamard signs (key = the sign seed, counter = 0).
``sr_draw4`` is the four-draws-per-call option of the stochastic-rounding
draw (counter = index >> 2, word = index & 3).
"""

from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK = 0xFFFFFFFF


def _mulhilo(m: int, x: np.ndarray):
    p = np.uint64(m) * x.astype(np.uint64)
    return (p >> np.uint64(32)).astype(np.uint32), (p & np.uint64(MASK)).astype(np.uint32)


def philox4x32_10(ctr, key):
    """Vectorised Philox-4x32-10.

    ``ctr``: array [..., 4] of uint32 counter words (c0, c1, c2, c3).
    ``key``: pair (k0, k1) of uint32 key words, or array [..., 2].
    Returns uint32 array [..., 4].

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
    the key is bumped by (W0, W1) between rounds.
    """
    c = np.asarray(ctr, dtype=np.uint32)
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k = np.asarray(key, dtype=np.uint64)
    k0 = (k[..., 0] & np.uint64(MASK)).astype(np.uint32)
    k1 = (k[..., 1] & np.uint64(MASK)).astype(np.uint32)
    for r in range(10):
        if r:
            k0 = (k0.astype(np.uint64) + np.uint64(W0)).astype(np.uint64) & np.uint64(MASK)
            k1 = (k1.astype(np.uint64) + np.uint64(W1)).astype(np.uint64) & np.uint64(MASK)
            k0 = k0.astype(np.uint32)
            k1 = k1.astype(np.uint32)
        hi0, lo0 = _mulhilo(M0, c0)
        hi1, lo1 = _mulhilo(M1, c2)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1)


def split64(v: int):
    """64-bit integer -> (low 32 bits, high 32 bits)."""
    v = int(v) & 0xFFFFFFFFFFFFFFFF
    return v & MASK, v >> 32


def sr_draw(seed: int, idx: np.ndarray) -> np.ndarray:
    """Stochastic-rounding draw for element indices ``idx`` (int64): word 0 of
    Philox-4x32-10 with key = (seed_lo, seed_hi) and counter =
    (idx_lo, idx_hi, 0, 0)."""
    idx = np.asarray(idx, dtype=np.uint64)
    ctr = np.zeros(idx.shape + (4,), dtype=np.uint32)
    ctr[..., 0] = (idx & np.uint64(MASK)).astype(np.uint32)
    ctr[..., 1] = (idx >> np.uint64(32)).astype(np.uint32)
    return philox4x32_10(ctr, split64(seed))[..., 0]


def sr_draw4(seed: int, idx: np.ndarray) -> np.ndarray:
    """Stochastic-rounding draw, four draws per generator call: word
    (idx & 3) of Philox-4x32-10 with key = (seed_lo, seed_hi) and counter =
    (c_lo, c_hi, 0, 0), c = idx >> 2.  Four consecutive indices 4c .. 4c + 3
    share one call and take its words 0 .. 3 in order.  This is an explicit
    option of the implementation (the pages fix only that the draws come from
    Philox keyed by the seed and counted by the element index); with it one
    generator call serves four elements."""
    idx = np.asarray(idx, dtype=np.uint64)
    c = idx >> np.uint64(2)
    ctr = np.zeros(idx.shape + (4,), dtype=np.uint32)
    ctr[..., 0] = (c & np.uint64(MASK)).astype(np.uint32)
    ctr[..., 1] = (c >> np.uint64(32)).astype(np.uint32)
    words = philox4x32_10(ctr, split64(seed))
    w = (idx & np.uint64(3)).astype(np.int64)
    return np.take_along_axis(words, w[..., None], axis=-1)[..., 0]


def hadamard_signs(seed: int) -> np.ndarray:
    """The 32 fixed signs (+1/-1, float64) of the Hadamard preconditioner:
    bit j of word 0 of Philox-4x32-10(key = (seed_lo, seed_hi),
    counter = 0); a set bit means -1."""
    w = int(philox4x32_10(np.zeros(4, dtype=np.uint32), split64(seed))[0])
    return np.array([-1.0 if (w >> j) & 1 else 1.0 for j in range(32)])
