"""Planted mistakes in the oracle, on the CPU: every mutant below is one plausible
slip in one oracle function (a dropped term, a wrong sign, index, pairing or
axis, a swapped operand, an off-by-one mask, a rounding taken once where the
pages take two). Each is applied by editing that function's source text and
rebinding it in its module; then the oracle's pins run, and at least one of
them must fail. A pin set that a mutant passed would not pin that part of the
oracle. The mutants are edits of the oracle only: no CUDA code is involved.
"""
import inspect

import numpy as np
import pytest

from oracle import attention as A
from oracle import bf16 as BF
from oracle import projection as P
from oracle import rope as R
from oracle import slots as S
from tests import (test_oracle_attention, test_oracle_bf16, test_oracle_projection, test_oracle_rope,
                   test_oracle_slots)
from tests.conftest import golden_path

# the exhaustive 65536-position table check takes ~17 s and pins the near-tie guard, not a formula
SLOW = {"test_cos_sin_table_rounding_is_decided_for_every_supported_position"}

PIN_FILES = {
    A: test_oracle_attention,
    BF: test_oracle_bf16,
    P: test_oracle_projection,
    R: test_oracle_rope,
    S: test_oracle_slots,
}


def _pins(oracle_module):
    first = PIN_FILES[oracle_module]  # the mutated module's own pins run first
    mods = [first] + [m for m in PIN_FILES.values() if m is not first]
    for mod in mods:
        for name, fn in list(vars(mod).items()):
            if name.startswith("test_") and inspect.isfunction(fn) and name not in SLOW:
                yield f"{mod.__name__.rsplit('.', 1)[-1]}::{name}", fn


def _first_failing_pin(oracle_module):
    for name, fn in _pins(oracle_module):
        kwargs = {"golden": golden_path} if "golden" in inspect.signature(fn).parameters else {}
        try:
            with np.errstate(all="ignore"):
                fn(**kwargs)
        except Exception:  # an assertion, or an error the mistake provokes: either way the pin fails
            return name
    return None


def _mutant(module, func, edits):
    """func of module with each (old, new) snippet replaced once in its source."""
    src = inspect.getsource(getattr(module, func))
    for old, new in edits:
        assert src.count(old) == 1, f"{module.__name__}.{func}: {old!r} does not occur exactly once"
        src = src.replace(old, new)
    ns = dict(vars(module))
    exec(compile(src, f"<mutant of {module.__name__}.{func}>", "exec"), ns)
    return ns[func]


# (id, module, function, [(old, new), ...])
MUTANTS = [
    # RoPE and the cache append
    ("rotate_half_sign", R, "rotate_half", [("np.concatenate((-x2, x1)", "np.concatenate((x2, -x1)")]),
    ("rotate_half_interleaved_pairs", R, "rotate_half",
     [("x1, x2 = np.split(x, 2, axis=-1)\n    return np.concatenate((-x2, x1), axis=-1)",
       "y = np.empty_like(x)\n    y[..., 0::2], y[..., 1::2] = -x[..., 1::2], x[..., 0::2]\n    return y")]),
    ("frequencies_repeated_not_tiled", R, "rotary_embedding",
     [("np.concatenate((half, half), axis=-1)", "np.repeat(half, 2, axis=-1)")]),
    ("inv_freq_exponent_i_over_d", R, "inv_freq",
     [("np.arange(0, dim, 2, dtype=np.float32)", "np.arange(0, dim // 2, dtype=np.float32)")]),
    ("inv_freq_base_not_inverted", R, "inv_freq",
     [("return (np.float32(1.0) / power)", "return (np.float32(1.0) * power)")]),
    ("offset_dropped", R, "positions",
     [("+ offset.astype(np.float32)[:, None]", "+ 0 * offset.astype(np.float32)[:, None]")]),
    ("positions_start_at_one", R, "positions",
     [("np.arange(T, dtype=np.float32)", "np.arange(1, T + 1, dtype=np.float32)")]),
    ("cos_and_sin_swapped", R, "rotary_embedding",
     [("a = (x * c)", "a = (x * s)"), ("b = (rotate_half(x) * s)", "b = (rotate_half(x) * c)")]),
    ("cos_sin_left_in_fp64", R, "cos_sin", [("return c.astype(np.float32), s.astype(np.float32)", "return c, s")]),
    ("phase_in_fp64", R, "phase",
     [("(t[:, :, None] * freqs[None, None, :]).astype(np.float32)",
       "t[:, :, None].astype(np.float64) * freqs[None, None, :].astype(np.float64)")]),
    ("products_and_sum_rounded_once", R, "rotary_embedding",
     [("a = (x * c).astype(np.float32)", "a = x.astype(np.float64) * c.astype(np.float64)"),
      ("b = (rotate_half(x) * s).astype(np.float32)", "b = rotate_half(x).astype(np.float64) * s.astype(np.float64)"),
      ("y = (a + b).astype(np.float32)\n    return bf16.from_f32(y)", "return bf16.from_f64(a + b)")]),
    ("update_one_row_late", R, "update_into",
     [("out[b, s:s + T] = update_bits[b]", "out[b, s + 1:s + T + 1] = update_bits[b][:T - 1 if s + T == out.shape[1] else T]")]),
    ("cache_stores_unrotated_k", R, "rope_kv_append",
     [("update_into(cache_k_bits, start, k_rot)", "update_into(cache_k_bits, start, k_bits)")]),
    ("cache_stores_rotated_v", R, "rope_kv_append",
     [("update_into(cache_v_bits, start, v_bits)", "update_into(cache_v_bits, start, rotary_embedding(v_bits, start))")]),
    # attention
    ("scale_dropped", A, "_attend_exact", [("logits = logits * ATTN_OUTPUT_MULTIPLIER", "logits = logits * 1.0")]),
    ("scale_one_over_d", A, "_attend_exact",
     [("logits = logits * ATTN_OUTPUT_MULTIPLIER", "logits = logits * ATTN_OUTPUT_MULTIPLIER ** 2")]),
    ("cap_dropped", A, "_attend_exact", [("logits = soft_cap(logits, cap)", "logits = logits")]),
    ("cap_before_scale", A, "_attend_exact",
     [("logits = logits * ATTN_OUTPUT_MULTIPLIER\n    if cap is not None:\n        logits = soft_cap(logits, cap)",
       "if cap is not None:\n        logits = soft_cap(logits, cap)\n    logits = logits * ATTN_OUTPUT_MULTIPLIER")]),
    ("cap_without_inner_division", A, "soft_cap", [("cap * np.tanh(x / cap)", "cap * np.tanh(x)")]),
    ("masked_logit_zero", A, "_attend_exact",
     [("np.where(mask, logits, MASK_FILL)", "np.where(mask, logits, 0.0)")]),
    ("causal_strict", A, "visible", [("causal_mask = j <= start + i", "causal_mask = j < start + i")]),
    ("causal_ignores_start", A, "visible", [("causal_mask = j <= start + i", "causal_mask = j <= i")]),
    ("padding_on_absolute_rows", A, "visible",
     [("padding_mask = ~((j >= start) & (j - start >= valid))", "padding_mask = j < valid")]),
    ("memory_mask_one_short", A, "visible", [("memory_mask = j < start + T", "memory_mask = j < start + T - 1")]),
    ("softmax_unnormalised", A, "_softmax64", [("return e / e.sum(axis=-1, keepdims=True)", "return e")]),
    ("softmax_over_queries", A, "_softmax64",
     [("return e / e.sum(axis=-1, keepdims=True)", "return e / e.sum(axis=0, keepdims=True)")]),
    ("values_replaced_by_keys", A, "_attend_exact", [("return w @ V", "return w @ K")]),
    ("gqa_head_modulo", A, "attention", [("g = h // group", "g = h % (n_q // group)")]),
    ("gqa_head_modulo_rows", A, "attention_rows", [("g = h // group", "g = h % (q_rot_bits.shape[2] // group)")]),
    ("valid_len_ignored", A, "attention",
     [("valid = np.full(B, T) if valid is None else np.asarray(valid)", "valid = np.full(B, T)")]),
    ("decode_at_kv_len", A, "decode", [("kv_len - 1, None, mode", "kv_len, None, mode")]),
    ("row_block_skips_its_last_row", A, "attention",
     [("np.arange(i0, min(T, i0 + ROW_BLOCK))", "np.arange(i0, min(T, i0 + ROW_BLOCK - 1))")]),
    ("block_ignores_start", A, "attention_block", [("s, n = int(start[b]), int(valid[b])", "s, n = 0, int(valid[b])")]),
    ("block_head_modulo", A, "attention_block", [("g = h // group", "g = h % (n_q // group)")]),
    ("rows_ignore_start", A, "attention_rows", [("s, nv = int(start[b]), int(valid[b])", "s, nv = 0, int(valid[b])")]),
    ("group_is_kv_head_count", A, "_kv_heads", [("return n_q, n_q // n_kv", "return n_q, n_kv")]),
    # the pages' dtype chain (diagnostic mode)
    ("chain_logits_in_bf16", A, "_attend_chain",
     [("logits = (q @ K.T).astype(np.float32)", "logits = bf16.to_f32(bf16.from_f64(q @ K.T))")]),
    ("chain_weights_not_rounded_to_bf16", A, "_attend_chain",
     [("w = bf16.to_f64(bf16.from_f32(w))", "w = w.astype(np.float64)")]),
    # projections
    ("k_and_v_columns_swapped", P, "qkv_projection",
     [("k = y[..., nq:nq + nk].reshape(B, T, N_KV_HEADS, HEAD_DIM)\n    v = y[..., nq + nk:]",
       "v = y[..., nq:nq + nk].reshape(B, T, N_KV_HEADS, HEAD_DIM)\n    k = y[..., nq + nk:]")]),
    ("q_columns_feature_major", P, "qkv_projection",
     [("q = y[..., :nq].reshape(B, T, N_Q_HEADS, HEAD_DIM)",
       "q = y[..., :nq].reshape(B, T, HEAD_DIM, N_Q_HEADS).swapaxes(-1, -2)")]),
    ("fused_step_rotates_at_next_position", P, "qkv_rope_append",
     [("rope.rope_kv_append(q, k, v, start,", "rope.rope_kv_append(q, k, v, start + 1,")]),
    ("output_projection_heads_reversed", P, "output_projection",
     [("linear(attn_bits.reshape(", "linear(attn_bits[:, :, ::-1].reshape(")]),
    ("shard_takes_wrong_rows", P, "output_projection_partial",
     [("w_o_bits[rank * width:(rank + 1) * width]", "w_o_bits[(ranks - 1 - rank) * width:(ranks - rank) * width]")]),
    ("dequant_scales_per_input_row", P, "dequant_int8",
     [("scales.astype(np.float32)[None, :]", "scales.astype(np.float32)[:w8.shape[1], None][:w8.shape[0]]")]),
    ("dequant_rounded_once", P, "dequant_int8",
     [("prod = (w8.astype(np.float32) * scales.astype(np.float32)[None, :]).astype(np.float32)\n"
       "    return bf16.from_f32(prod)",
       "return bf16.from_f64(w8.astype(np.float64) * scales.astype(np.float64)[None, :])")]),
    # bf16 rounding
    ("bf16_truncates", BF, "from_f32",
     [("r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16))", "r = (u >> np.uint64(16))")]),
    ("bf16_ties_away", BF, "from_f32", [("+ np.uint64(0x7FFF) + lsb)", "+ np.uint64(0x8000))")]),
    ("bf16_from_f64_rounds_twice", BF, "from_f64",
     [("x = np.asarray(x, dtype=np.float64)\n", "return from_f32(np.asarray(x, dtype=np.float64).astype(np.float32))\n")]),
    # slot insertion
    ("slot_one_row_too_many", S, "insert_slot",
     [("out[slot, :n_rows] = single_bits[0, :n_rows]", "out[slot, :n_rows + 1] = single_bits[0, :n_rows + 1]")]),
    ("slot_written_into_every_sequence", S, "insert_slot",
     [("out[slot, :n_rows] = single_bits[0, :n_rows]", "out[:, :n_rows] = single_bits[0, :n_rows]")]),
    ("step_updated_in_place", S, "insert_step", [("out = np.array(steps, copy=True)", "out = steps")]),
]


def test_unmutated_oracle_passes_every_pin():
    assert _first_failing_pin(A) is None


@pytest.mark.parametrize("mid,module,func,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_every_planted_mistake_fails_a_pin(monkeypatch, mid, module, func, edits):
    monkeypatch.setattr(module, func, _mutant(module, func, edits))
    caught = _first_failing_pin(module)
    assert caught is not None, f"mutant {mid} of {module.__name__}.{func} passes every pin"
