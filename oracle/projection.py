"""Oracle: the Q/K/V projections in front of the attention call, and the fused
projection + RoPE + cache append.

Follows the Grok-1 code quoted in the code-reading guide, ch. 4 "model.py close
reading I: RMSNorm, RoPE, GQA Attention" (yingwang.github.io/grok-1/04-model-1/):

* §4.1 ``Linear.__call__``: the weight parameter has shape [input_size,
  output_size]; the output is ``jnp.dot(inputs, w.astype(fprop_dtype))`` plus
  an optional bias.
* §4.5.1 Q/K/V projection and ``_linear_projection``: three ``Linear`` layers
  with ``with_bias=False``: query to 48 x 128 features, key and value to
  8 x 128 each, each output reshaped to [..., num_heads, head_size].
* §4.4 (RoPE placement): the projected query and key are then rotated with
  offset = the cache step and the rotated key and raw value written into the
  cache (``rope.rope_kv_append``).
* §4.1 Linear with ``QuantizedWeight8bit`` and §4.1.1: when the weight carries
  ``scales``, the weight is dequantized as ``weight.astype(scales.dtype) *
  scales`` (int8 weight [input, output], one fp32 scale per output channel,
  broadcast along the input axis) and then cast to the input dtype before the
  dot. Reading: the product is an fp32 multiply rounded to fp32, then rounded
  to bf16 (two roundings, in the pages' order).
* §4.5.4 final projection: the attention output [B, T, 48, 128] is reshaped
  to [B, T, 48 * 128] (heads in order h = 6g + r, features within a head
  contiguous) and multiplied by a bias-free Linear to model_size 6144. The
  Linear's weights are sharded along their input dimension (each model shard
  holds the rows of its heads), so under tensor parallelism every shard
  computes a partial product and the partials are summed.

Readings where the pages leave details open:

* The three projections are one product with the weights side by side:
  W = [W_query | W_key | W_value], shape [6144, 8192]; output column
  h*128 + d is query head h, 6144 + g*128 + d key head g, 7168 + g*128 + d
  value head g (the reshape to [..., heads, 128] splits columns head-major).
* The dot of bf16 inputs with bf16 weights returns bf16: here the exact sum
  (fp64; each bf16 x bf16 product is exact in fp64 and 6144 terms add far
  below bf16 resolution) rounded once to bf16, round to nearest even.
* The fused step feeds those bf16 q, k, v into the RoPE + append oracle
  unchanged.

Test infrastructure only: nothing in the CUDA library or its binding imports this.
"""
from __future__ import annotations

import numpy as np

from . import bf16, rope

MODEL_SIZE = 6144
N_Q_HEADS = 48
N_KV_HEADS = 8
HEAD_DIM = 128
QKV_COLUMNS = (N_Q_HEADS + 2 * N_KV_HEADS) * HEAD_DIM  # 8192


def linear_exact(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """The sum of §4.1's dot before its rounding to bf16, in fp64: x [..., K] . w [K, N]."""
    lead = x_bits.shape[:-1]
    x = bf16.to_f64(x_bits).reshape(-1, x_bits.shape[-1])
    return (x @ bf16.to_f64(w_bits)).reshape(*lead, w_bits.shape[1])


def linear(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """§4.1 Linear without bias: bf16 x [..., K] times bf16 w [K, N], exact sum rounded to bf16."""
    return bf16.from_f64(linear_exact(x_bits, w_bits))


def qkv_projection(x_bits: np.ndarray, w_bits: np.ndarray):
    """§4.5.1: x [B, T, 6144] and the side-by-side weights [6144, 8192] -> q [B,T,48,128], k, v [B,T,8,128]."""
    y = linear(x_bits, w_bits)
    B, T = x_bits.shape[0], x_bits.shape[1]
    nq = N_Q_HEADS * HEAD_DIM
    nk = N_KV_HEADS * HEAD_DIM
    q = y[..., :nq].reshape(B, T, N_Q_HEADS, HEAD_DIM)
    k = y[..., nq:nq + nk].reshape(B, T, N_KV_HEADS, HEAD_DIM)
    v = y[..., nq + nk:].reshape(B, T, N_KV_HEADS, HEAD_DIM)
    return q, k, v


def qkv_rope_append(x_bits, w_bits, start, cache_k_bits, cache_v_bits):
    """Projection, then §4.4's RoPE and cache append: returns (q_rot, new_cache_k, new_cache_v) bits."""
    q, k, v = qkv_projection(x_bits, w_bits)
    return rope.rope_kv_append(q, k, v, start, cache_k_bits, cache_v_bits)


def output_projection(attn_bits: np.ndarray, w_o_bits: np.ndarray) -> np.ndarray:
    """§4.5.4: attention output [B, T, 48, 128] flattened head-major, times W_o [6144, 6144] -> [B, T, 6144]."""
    B, T = attn_bits.shape[0], attn_bits.shape[1]
    return linear(attn_bits.reshape(B, T, N_Q_HEADS * HEAD_DIM), w_o_bits)


def output_projection_partial(attn_bits: np.ndarray, w_o_bits: np.ndarray, rank: int, ranks: int) -> np.ndarray:
    """One model shard's exact (fp64, unrounded) share: its heads' features times its rows of W_o."""
    B, T = attn_bits.shape[0], attn_bits.shape[1]
    width = N_Q_HEADS * HEAD_DIM // ranks
    x = attn_bits.reshape(B, T, N_Q_HEADS * HEAD_DIM)[..., rank * width:(rank + 1) * width]
    return linear_exact(x, w_o_bits[rank * width:(rank + 1) * width])


def dequant_int8(w8: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """§4.1: int8 weight [K, N] times fp32 per-output-channel scales [N], rounded to fp32, then to bf16."""
    prod = (w8.astype(np.float32) * scales.astype(np.float32)[None, :]).astype(np.float32)
    return bf16.from_f32(prod)


def linear_int8(x_bits: np.ndarray, w8: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """§4.1 Linear with a QuantizedWeight8bit weight: dequantize, then the bf16 dot."""
    return linear(x_bits, dequant_int8(w8, scales))
