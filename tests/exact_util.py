"""Brute-force rounding for the oracle's pins: the fp32 or bf16 value nearest an
exact rational, ties to the even bit pattern, found by comparing the exact
distances of the neighbouring patterns (no floating-point rounding involved
in the choice). Independent of the oracle: nothing here imports it."""
from fractions import Fraction

import numpy as np


def _bf16_value(bits: int) -> float:
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


def nearest_bf16(v: Fraction) -> float:
    """The bf16 value nearest the exact rational v (ties to the even pattern)."""
    base = int(np.float32(float(v)).view(np.uint32) >> 16)
    cands = []
    for d in (-2, -1, 0, 1, 2):
        b = (base + d) & 0xFFFF
        val = _bf16_value(b)
        if np.isfinite(val):
            cands.append((abs(Fraction(val) - v), b % 2, val))
    cands.sort()
    return cands[0][2]


def nearest_f32(v: Fraction) -> Fraction:
    """The fp32 value nearest the exact rational v (ties to the even pattern), as a Fraction."""
    c0 = np.float32(float(v))
    cands = []
    for c in (np.nextafter(c0, np.float32(-np.inf)), c0, np.nextafter(c0, np.float32(np.inf))):
        if np.isfinite(c):
            cands.append((abs(Fraction(float(c)) - v), int(np.array(c).view(np.uint32)) & 1, float(c)))
    cands.sort()
    return Fraction(cands[0][2])
