"""Pins for the slot-insertion oracle (ch. 6 §6.6.1): element-by-element brute
force, and the properties the insertion must have (other slots and the rows
past n_rows untouched, the step of the slot replaced, insertion idempotent)."""
import numpy as np
import pytest

from oracle import slots as S


def _rand(shape, seed):
    return np.random.default_rng(seed).integers(0, 1 << 16, size=shape, dtype=np.uint16)


def test_insert_matches_elementwise_brute_force():
    mem, single = _rand((3, 10, 2, 4), 1), _rand((1, 7, 2, 4), 2)
    out = S.insert_slot(mem, 1, single, 5)
    for b in range(3):
        for t in range(10):
            for h in range(2):
                for d in range(4):
                    want = single[0, t, h, d] if (b == 1 and t < 5) else mem[b, t, h, d]
                    assert out[b, t, h, d] == want


def test_insert_properties():
    mem, single = _rand((4, 16, 8, 8), 3), _rand((1, 16, 8, 8), 4)
    out = S.insert_slot(mem, 2, single, 9)
    assert np.array_equal(np.delete(out, 2, axis=0), np.delete(mem, 2, axis=0))  # other slots untouched
    assert np.array_equal(out[2, 9:], mem[2, 9:])                                # rows past n_rows untouched
    assert np.array_equal(out[2, :9], single[0, :9])
    assert np.array_equal(S.insert_slot(out, 2, single, 9), out)                # idempotent
    assert np.array_equal(S.insert_slot(mem, 0, single, 0), mem)                # zero rows: no change
    assert not np.shares_memory(out, mem)


def test_insert_step_and_ranges():
    steps = np.array([5, 7, 9], dtype=np.int32)
    assert S.insert_step(steps, 1, 42).tolist() == [5, 42, 9]
    assert steps.tolist() == [5, 7, 9]
    with pytest.raises(ValueError):
        S.insert_slot(_rand((2, 4, 1, 1), 5), 2, _rand((1, 4, 1, 1), 6), 1)
    with pytest.raises(ValueError):
        S.insert_slot(_rand((2, 4, 1, 1), 5), 0, _rand((1, 3, 1, 1), 6), 4)
