"""Oracle: Grok-1 grouped-query attention over the KV cache (prefill and decode).

Plain definition, evaluated in fp64 from the bf16 tensors, following the Grok-1
code quoted in the code-reading guide:

* ch. 4 "model.py close reading I", §4.5.2 GQA reshape and attention: query
  heads are reshaped to [B, T, kv_heads, q_per_kv, d], so query head h uses
  KV head h // q_per_kv (48 query heads, 8 KV heads, 6 per group); logits =
  einsum("...thHd,...Thd->...hHtT") cast to fp32; logits *=
  attn_output_multiplier (1/sqrt(128), ch. 3 "Config and hyper-parameters",
  §3.3.2); logits = 30 * tanh(logits / 30) (soft cap).
* §4.5.3 mask and softmax: jnp.where(mask, logits, -1e30), softmax over keys in
  fp32, weights cast to the query dtype (bf16).
* §4.5.4: einsum("...hHtT,...Thd->...thHd") with V, heads flattened back in the
  order g*6 + r = h.
* Masks: ch. 6 "model.py close reading II", §6.4.2 (causal tril times key
  padding, [B,1,T,T]) and ch. 4 §4.4 / ch. 6 §6.4.2 (memory mask: cache rows
  below step + T). In decode the causal mask is all ones and the memory mask
  does the work (ch. 4 §4.4.1).

Two modes:

* ``exact`` (the oracle): dot products, scale, cap, softmax and the weighted
  sum in fp64; masked keys get weight exactly 0 (the limit of exp(-1e30 - max));
  the output is rounded once to bf16.
* ``chain`` (diagnostic, used only to measure the error floor of the pages' own
  dtype chain): logits rounded to fp32, fp32 scale and cap, fp32 softmax,
  weights rounded to bf16, weighted sum accumulated in fp64, output to bf16.

Readings where the pages are silent or garbled:

* Position convention: query i of sequence b sits at cache position
  start[b] + i; key (cache row) j is visible to it iff j <= start[b] + i
  (causal), j < start[b] + valid[b] (key padding of the new tokens; cached rows
  below start[b] are never padding) and j < start[b] + T (memory mask). For an
  empty cache (start = 0, T = Tmax) this is exactly tril x padding; for a decode
  step (T = 1) it is j <= step; for a chunk on a warm cache it is the
  [B,1,T,start+T] mask "causal within the chunk".
* Rows at or beyond start[b] + T lie outside the memory mask and take no part
  (the pages multiply their zero weight by a zero-initialised cache; here those
  rows hold junk and are simply not read).
* Padding query rows (i >= valid[b]) are computed like any other row: the
  pages' padding mask acts on keys only.
* Logits are fp32 or better (the prose of §4.5.3 and ch. 3 §3.3.2), not bf16.

Test infrastructure only: nothing in the CUDA library or its binding imports this.
"""
from __future__ import annotations

import numpy as np

from . import bf16

ATTN_OUTPUT_MULTIPLIER = 0.08838834764831845  # 1/sqrt(128), ch. 3 §3.3.2
MAX_ATTN_VAL = 30.0                            # soft cap, ch. 4 §4.5.2
MASK_FILL = -1e30                              # ch. 4 §4.5.3
ROW_BLOCK = 256


def visible(start: int, valid: int, T: int, i: np.ndarray, n_keys: int) -> np.ndarray:
    """bool [len(i), n_keys]: memory mask x causal mask x key padding for one sequence."""
    j = np.arange(n_keys)[None, :]
    i = np.asarray(i)[:, None]
    memory_mask = j < start + T
    causal_mask = j <= start + i
    padding_mask = ~((j >= start) & (j - start >= valid))
    return memory_mask & causal_mask & padding_mask


def soft_cap(x, cap=MAX_ATTN_VAL):
    """cap * tanh(x / cap) in the dtype of x."""
    return cap * np.tanh(x / cap)


def _softmax64(logits: np.ndarray) -> np.ndarray:
    m = logits.max(axis=-1, keepdims=True)
    e = np.exp(logits - m)
    return e / e.sum(axis=-1, keepdims=True)


def _attend_exact(q: np.ndarray, K: np.ndarray, V: np.ndarray, mask: np.ndarray,
                  cap=MAX_ATTN_VAL) -> np.ndarray:
    """fp64 rows: softmax(cap(q K^T * mult), masked) V for q [n, d], K, V [L, d].

    ``cap=None`` leaves the logits uncapped (used only to reduce the method to
    plain scaled dot-product attention in a test).
    """
    logits = q @ K.T
    logits = logits * ATTN_OUTPUT_MULTIPLIER
    if cap is not None:
        logits = soft_cap(logits, cap)
    logits = np.where(mask, logits, MASK_FILL)
    w = _softmax64(logits)
    return w @ V


def _attend_chain(q: np.ndarray, K: np.ndarray, V: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """The pages' dtype chain: fp32 logits/cap/softmax, bf16 weights; fp64 rows out."""
    logits = (q @ K.T).astype(np.float32)
    logits = (logits * np.float32(ATTN_OUTPUT_MULTIPLIER)).astype(np.float32)
    cap = np.float32(MAX_ATTN_VAL)
    logits = (cap * np.tanh((logits / cap).astype(np.float32))).astype(np.float32)
    logits = np.where(mask, logits, np.float32(MASK_FILL)).astype(np.float32)
    m = logits.max(axis=-1, keepdims=True)
    e = np.exp((logits - m).astype(np.float32)).astype(np.float32)
    w = (e / e.sum(axis=-1, keepdims=True, dtype=np.float32)).astype(np.float32)
    w = bf16.to_f64(bf16.from_f32(w))
    return w @ V


def _kv_heads(q_rot_bits: np.ndarray, cache_k_bits: np.ndarray) -> tuple[int, int]:
    n_q, n_kv = q_rot_bits.shape[2], cache_k_bits.shape[2]
    if n_q % n_kv:
        raise ValueError("query heads must be a multiple of KV heads")
    return n_q, n_q // n_kv


def attention(q_rot_bits, cache_k_bits, cache_v_bits, start, valid=None, mode="exact",
              return_f64=False, cap=MAX_ATTN_VAL):
    """Attention of all T new queries of every sequence over the (already appended) cache.

    q_rot [B, T, Hq, d] and cache_k/v [B, Tmax, Hkv, d] are bf16 bits; start [B]
    is the cache position of each sequence's first new token; valid [B] the
    number of non-padding new tokens (None: all T). Returns bf16 bits
    [B, T, Hq, d] (and the unrounded fp64 values when ``return_f64``).
    """
    B, T, n_q, d = q_rot_bits.shape
    _, group = _kv_heads(q_rot_bits, cache_k_bits)
    valid = np.full(B, T) if valid is None else np.asarray(valid)
    if mode == "exact":
        def attend(q, K, V, m):
            return _attend_exact(q, K, V, m, cap)
    else:
        attend = _attend_chain
    out = np.zeros((B, T, n_q, d), dtype=np.float64)
    for b in range(B):
        s, n = int(start[b]), int(valid[b])
        L = s + T                                  # rows inside the memory mask
        for h in range(n_q):
            g = h // group
            K = bf16.to_f64(cache_k_bits[b, :L, g, :])
            V = bf16.to_f64(cache_v_bits[b, :L, g, :])
            for i0 in range(0, T, ROW_BLOCK):
                rows = np.arange(i0, min(T, i0 + ROW_BLOCK))
                q = bf16.to_f64(q_rot_bits[b, rows, h, :])
                out[b, rows, h, :] = attend(q, K, V, visible(s, n, T, rows, L))
    bits = bf16.from_f64(out)
    return (bits, out) if return_f64 else bits


def attention_rows(q_rot_bits, cache_k_bits, cache_v_bits, start, valid, T, rows,
                   mode="exact"):
    """The same definition for selected outputs only: rows = [(b, i, h), ...].

    Returns (bf16 bits [n, d], fp64 [n, d]). Used for spot checks at sizes
    where the full output is too slow on the CPU.
    """
    _, group = _kv_heads(q_rot_bits, cache_k_bits)
    attend = _attend_exact if mode == "exact" else _attend_chain
    B = q_rot_bits.shape[0]
    valid = np.full(B, T) if valid is None else np.asarray(valid)
    d = q_rot_bits.shape[-1]
    out = np.zeros((len(rows), d), dtype=np.float64)
    for n, (b, i, h) in enumerate(rows):
        s, nv = int(start[b]), int(valid[b])
        L = s + T
        g = h // group
        K = bf16.to_f64(cache_k_bits[b, :L, g, :])
        V = bf16.to_f64(cache_v_bits[b, :L, g, :])
        q = bf16.to_f64(q_rot_bits[b, [i], h, :])
        out[n] = attend(q, K, V, visible(s, nv, T, np.array([i]), L))[0]
    return bf16.from_f64(out), out


def attention_block(q_rot_bits, cache_k_bits, cache_v_bits, start, valid, T, b, i0, i1):
    """The same definition for query rows [i0, i1) of sequence b, every head.

    Returns bf16 bits [i1 - i0, Hq, d]. Used to check whole query tiles at sizes
    where the full output is too slow on the CPU.
    """
    n_q, group = _kv_heads(q_rot_bits, cache_k_bits)
    B = q_rot_bits.shape[0]
    valid = np.full(B, T) if valid is None else np.asarray(valid)
    s, n = int(start[b]), int(valid[b])
    L = s + T
    rows = np.arange(i0, i1)
    mask = visible(s, n, T, rows, L)
    out = np.zeros((len(rows), n_q, q_rot_bits.shape[-1]), dtype=np.float64)
    for h in range(n_q):
        g = h // group
        K = bf16.to_f64(cache_k_bits[b, :L, g, :])
        V = bf16.to_f64(cache_v_bits[b, :L, g, :])
        q = bf16.to_f64(q_rot_bits[b, rows, h, :])
        out[:, h, :] = _attend_exact(q, K, V, mask)
    return bf16.from_f64(out)


def decode(q_rot_bits, cache_k_bits, cache_v_bits, kv_len, mode="exact", return_f64=False):
    """One decode step: q_rot [B, Hq, d] at position kv_len[b]-1 over cache rows < kv_len[b].

    This is ``attention`` with T = 1 and start = kv_len - 1 (the new token's
    own row was appended at position step = kv_len - 1).
    """
    kv_len = np.asarray(kv_len)
    r = attention(q_rot_bits[:, None], cache_k_bits, cache_v_bits, kv_len - 1, None, mode,
                  return_f64)
    if return_f64:
        return r[0][:, 0], r[1][:, 0]
    return r[:, 0]
