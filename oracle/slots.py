"""Oracle: continuous-batching slot insertion into the KV cache.

Follows the code-reading guide, ch. 6 "model.py close reading II", §6.6.1
(step field / continuous batching): every sequence of a batch carries its own
int32 step, so a finished sequence's slot can be handed to a new request; the
runner inserts the new sequence's memory into batch slot i with
``dynamic_update_index_in_dim(m, u[0], i, axis=0)`` on every memory tensor
(the k and v caches and the step).

Reading where the pages leave it open: attention never reads cache rows at or
beyond a sequence's step (the memory mask of ch. 4 §4.4), so replacing rows
[0, n_rows) of the slot, n_rows >= the new sequence's step, gives every later
result the pages' whole-slot replacement gives. Rows >= n_rows keep their
previous contents here.

Test infrastructure only: nothing in the CUDA library or its binding imports this.
"""
from __future__ import annotations

import numpy as np


def insert_slot(mem_bits: np.ndarray, slot: int, single_bits: np.ndarray, n_rows: int) -> np.ndarray:
    """mem [B, Tmax, H, d] with rows [0, n_rows) of slot replaced by single [1, L, H, d] (L >= n_rows)."""
    if not (0 <= slot < mem_bits.shape[0]) or not (0 <= n_rows <= min(mem_bits.shape[1], single_bits.shape[1])):
        raise ValueError("slot or row count out of range")
    out = np.array(mem_bits, copy=True)
    out[slot, :n_rows] = single_bits[0, :n_rows]
    return out


def insert_step(steps: np.ndarray, slot: int, step: int) -> np.ndarray:
    """The per-sequence step vector [B] with entry slot replaced."""
    out = np.array(steps, copy=True)
    out[slot] = step
    return out
