"""bfloat16 storage helpers for the oracle (numpy, bit level).

A bf16 value is the upper 16 bits of an IEEE binary32. Widening is exact;
narrowing rounds to nearest, ties to even, which is what ``.astype(bf16)``
does in the Grok-1 code quoted by the pages (ch. 4 "model.py close reading I",
§4.3.1 RotaryEmbedding, the final cast back to the input dtype; §4.5.3, the cast
of the softmax weights).

Test infrastructure only: nothing in the CUDA library or its binding imports this.
"""
from __future__ import annotations

import numpy as np


def to_f32(u16: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    u16 = np.asarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(u16: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    return to_f32(u16).astype(np.float64)


def from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        sign = ((u >> np.uint64(16)) & np.uint64(0x8000)).astype(np.uint16)
        r = np.where(nan, sign | np.uint16(0x7FC0), r)
    return r


def from_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values straight to bf16 (nearest, ties to even): one rounding.

    Going through float32 first would round twice and can land on the wrong
    side of a bf16 tie, so the significand is rounded here directly: bf16 keeps
    8 significant bits, so x = m * 2**e with 0.5 <= |m| < 1 becomes
    rint(m * 2**8) * 2**(e - 8) (``np.rint`` rounds half to even, exactly).
    Below the smallest normal (2**-126) the spacing is fixed at 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    normal = np.abs(x) >= 2.0 ** -126
    r_norm = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    r_sub = np.ldexp(np.rint(np.ldexp(x, 133)), -133)
    r = np.where(normal, r_norm, r_sub)
    big = np.abs(r) >= 2.0 ** 128
    r = np.where(big, np.copysign(np.inf, x), r)
    r = np.where(np.isnan(x), np.nan, r)
    # r is now exactly representable in bf16, hence in float32: narrowing is exact
    return from_f32(r.astype(np.float32))
