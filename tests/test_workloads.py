"""The seeded input generator: shapes, determinism and the junk fill of unused rows."""
import numpy as np

import workloads as W


def test_shapes_and_determinism():
    a = W.generate("prefill_b1_t128")
    b = W.generate("prefill_b1_t128")
    assert tuple(a.q.shape) == (1, 128, 48, 128)
    assert tuple(a.cache_k.shape) == (1, 128, 8, 128)
    assert np.array_equal(W.bits(a.q), W.bits(b.q))
    assert np.array_equal(W.bits(a.cache_v), W.bits(b.cache_v))


def test_decode_lengths_and_junk():
    inp = W.generate("decode_b32_ctx8192", batch=4)
    L = inp.start_pos.numpy()
    assert np.all((L >= 1) & (L <= 8191))
    ck = inp.cache_k.float().numpy()
    for b in range(4):
        assert np.all(np.abs(ck[b, L[b]:]) == 9984.0)        # bf16(1e4) junk from the new row on
        assert np.all(np.abs(ck[b, :L[b]]) < 100)


def test_ragged_valid_lengths():
    inp = W.generate("ragged_prefill_b8_t2048")
    n = inp.valid_len.numpy()
    assert n.shape == (8,) and np.all((n >= 256) & (n <= 2048))


def test_nan_poison():
    inp = W.custom(B=1, T=4, Tmax=16, start_pos=[3], junk="nan")
    ck = inp.cache_k.float().numpy()
    assert np.all(np.isnan(ck[0, 3:])) and not np.any(np.isnan(ck[0, :3]))
