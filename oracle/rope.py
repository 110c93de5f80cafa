"""Oracle: rotary position embedding of Q and K, and the KV-cache append.

Follows, step by step and in the same order, the Grok-1 code quoted in the
code-reading guide, ch. 4 "model.py close reading I: RMSNorm, RoPE, GQA
Attention" (yingwang.github.io/grok-1/04-model-1/):

* §4.3 ``rotate_half``: split the last axis in halves x1, x2 and return
  concat(-x2, x1) (GPT-NeoX pairing: feature i is paired with i + d/2, not i+1).
* §4.3.1 ``RotaryEmbedding.__call__``: exponents = arange(0, d, 2) in fp32;
  inv_freq = 1 / base**(exponents/d) in fp32; t = arange(T) + offset[b];
  phase = einsum("bi,j->bij", t, inv_freq), tiled twice along the feature
  axis; x' = x*cos(phase) + rotate_half(x)*sin(phase); cast back to bf16.
* §4.4 (RoPE placement): K and Q are rotated with offset = the cache step
  *before* the cache write, so the cache stores rotated keys; V is not rotated.
  ``update_into`` writes the new rows at step[b] of each sequence
  (``dynamic_update_slice_in_dim`` under vmap) and leaves every other row alone.

Readings where the pages leave rounding open (each one fixes a bit pattern):

* 10000**(j/64) is evaluated in fp64 and rounded once to fp32; the division
  1/that is an fp32 division. (j/64 is exact in fp32.)
* phase is one fp32 multiply of the fp32 position by inv_freq[j]; positions
  below 2**24 are exact in fp32.
* cos and sin of the fp32 phase are evaluated in fp64 and rounded once to fp32.
  For positions below 65536 every such value lies at least 59 fp64 ulps from an
  fp32 rounding midpoint (``check_no_near_ties`` re-verifies the margin used),
  so any fp64 evaluation within a few ulps gives the same fp32 bits.
* x*cos + rotate_half(x)*sin: bf16 x is widened exactly; each product and the
  sum are separate fp32 operations rounded to nearest (no fused multiply-add).

Test infrastructure only: nothing in the CUDA library or its binding imports this.
"""
from __future__ import annotations

import numpy as np

from . import bf16

ROPE_BASE = 10000
MAX_POSITION = 65536  # exclusive bound of positions the rounding argument covers


def rotate_half(x: np.ndarray) -> np.ndarray:
    """concat(-x2, x1) over the last axis (§4.3)."""
    x1, x2 = np.split(x, 2, axis=-1)
    return np.concatenate((-x2, x1), axis=-1)


def inv_freq(dim: int = 128, base: int = ROPE_BASE) -> np.ndarray:
    """fp32 [dim/2]: 1 / base**(2i/dim) (§4.3.1, frequency table)."""
    exponents = np.arange(0, dim, 2, dtype=np.float32)
    ratio = (exponents / np.float32(dim)).astype(np.float32)
    power = np.power(np.float64(base), ratio.astype(np.float64)).astype(np.float32)
    return (np.float32(1.0) / power).astype(np.float32)


def positions(offset: np.ndarray, T: int) -> np.ndarray:
    """fp32 [B, T]: t = arange(T) + offset[b] (§4.3.1)."""
    offset = np.asarray(offset, dtype=np.int64)
    if offset.min() < 0 or offset.max() + T > MAX_POSITION:
        raise ValueError("positions outside [0, 65536)")
    t = np.arange(T, dtype=np.float32)[None, :] + offset.astype(np.float32)[:, None]
    return t.astype(np.float32)


def phase(t: np.ndarray, freqs: np.ndarray) -> np.ndarray:
    """fp32 [B, T, dim/2]: einsum("bi,j->bij"), a single fp32 product per entry."""
    return (t[:, :, None] * freqs[None, None, :]).astype(np.float32)


def cos_sin(ph: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 cos and sin of an fp32 phase: fp64 evaluation, one rounding to fp32."""
    p64 = ph.astype(np.float64)
    c = np.cos(p64)
    s = np.sin(p64)
    check_no_near_ties(c)
    check_no_near_ties(s)
    return c.astype(np.float32), s.astype(np.float32)


def check_no_near_ties(y: np.ndarray, margin_ulps: float = 16.0) -> None:
    """Raise if an fp64 value lies within ``margin_ulps`` fp64 ulps of an fp32 midpoint.

    Such a value could round to either neighbour depending on the last bits of
    the fp64 evaluation; outside that margin the fp32 result is fixed.
    """
    y = np.asarray(y, dtype=np.float64)
    nz = y != 0
    if not nz.any():
        return
    y = y[nz]
    r = y.astype(np.float32)
    ulp32 = np.spacing(np.abs(r)).astype(np.float64)
    dist = 0.5 * ulp32 - np.abs(y - r.astype(np.float64))
    if (dist < margin_ulps * np.spacing(np.abs(y))).any():
        raise ArithmeticError("cos/sin value too close to an fp32 rounding midpoint")


def rotary_embedding(x_bits: np.ndarray, offset: np.ndarray) -> np.ndarray:
    """Rotate bf16 x [B, T, H, dim] (uint16 bits) with per-sequence offsets (§4.3.1).

    Returns the rotated tensor as bf16 bits.
    """
    B, T, H, dim = x_bits.shape
    x = bf16.to_f32(x_bits)
    t = positions(offset, T)
    half = phase(t, inv_freq(dim))                       # [B, T, dim/2]
    full = np.concatenate((half, half), axis=-1)         # tile reps=(1, 2)
    full = full[:, :, None, :]                           # [B, T, 1, dim]
    c, s = cos_sin(full)
    a = (x * c).astype(np.float32)
    b = (rotate_half(x) * s).astype(np.float32)
    y = (a + b).astype(np.float32)
    return bf16.from_f32(y)


def update_into(mem_bits: np.ndarray, start: np.ndarray, update_bits: np.ndarray) -> np.ndarray:
    """Per-sequence dynamic update slice along the position axis (§4.4).

    mem [B, Tmax, H, dim], update [B, T, H, dim]; rows [start[b], start[b]+T)
    of sequence b are replaced, every other row is kept. Returns a new array.
    """
    out = np.array(mem_bits, copy=True)
    T = update_bits.shape[1]
    for b in range(mem_bits.shape[0]):
        s = int(start[b])
        if s < 0 or s + T > mem_bits.shape[1]:
            raise ValueError("update slice out of range")
        out[b, s:s + T] = update_bits[b]
    return out


def rope_kv_append(q_bits, k_bits, v_bits, start, cache_k_bits, cache_v_bits):
    """The whole first step of the attention call (§4.4 execution order).

    Returns (q_rot, new_cache_k, new_cache_v), all bf16 bits: K and Q rotated
    with offset = start, rotated K and raw V written into the caches at start.
    """
    k_rot = rotary_embedding(k_bits, start)
    q_rot = rotary_embedding(q_bits, start)
    new_k = update_into(cache_k_bits, start, k_rot)
    new_v = update_into(cache_v_bits, start, v_bits)
    return q_rot, new_k, new_v
