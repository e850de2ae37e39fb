"""Philox4x32-10 counter-based generator, written from its published definition
(Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11,
section 4: the Philox S-box built from two 32x32->64 multiplications, a Weyl key
schedule, ten rounds).

Oracle-side implementation (test infrastructure).  The CUDA path carries its own,
written independently from the same definition; the two are compared bit for bit.

Stream layout used by the method (the pages only say the uniforms come from a seeded Philox):
key = (seed & 0xffffffff, seed >> 32); counter = (step t, purpose, 0, 0).
Purposes: 0 draft sample, 1 accept test, 2 target / residual sample,
3 forced-draft coin, 4 forced-draft alternative id.  The prefill's first sample is t = 0.
A uniform in [0,1) is (word0 >> 8) * 2^-24, exact in binary floating point.
"""
from __future__ import annotations

from typing import Sequence, Tuple

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK = 0xFFFFFFFF

PURPOSE_DRAFT = 0
PURPOSE_ACCEPT = 1
PURPOSE_TARGET = 2
PURPOSE_COIN = 3
PURPOSE_ALT = 4


def _round(c: Sequence[int], k: Sequence[int]) -> Tuple[int, int, int, int]:
    p0 = M0 * c[0]
    p1 = M1 * c[2]
    hi0, lo0 = p0 >> 32, p0 & MASK
    hi1, lo1 = p1 >> 32, p1 & MASK
    return ((hi1 ^ c[1] ^ k[0]) & MASK, lo1, (hi0 ^ c[3] ^ k[1]) & MASK, lo0)


def philox4x32_10(counter: Sequence[int], key: Sequence[int]) -> Tuple[int, int, int, int]:
    c = tuple(int(x) & MASK for x in counter)
    k = [int(key[0]) & MASK, int(key[1]) & MASK]
    for r in range(10):
        if r:
            k = [(k[0] + W0) & MASK, (k[1] + W1) & MASK]
        c = _round(c, k)
    return c


def word(seed: int, t: int, purpose: int) -> int:
    key = (seed & MASK, (seed >> 32) & MASK)
    return philox4x32_10((t & MASK, purpose, 0, 0), key)[0]


def uniform(seed: int, t: int, purpose: int) -> float:
    return (word(seed, t, purpose) >> 8) * (1.0 / 16777216.0)


def u24(seed: int, t: int, purpose: int) -> int:
    """The 24-bit integer behind ``uniform`` (uniform = u24 / 2^24)."""
    return word(seed, t, purpose) >> 8
