"""The seeded input generator: shapes, determinism and the junk fill of unused rows."""
import numpy as np
import torch

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


def test_page_table_is_a_scattered_injection():
    table, n_pages = W.page_table(3, 6, [2, 6, 0], spare=4, seed=9)
    assert table.shape == (3, 6) and table.dtype == torch.int32 and n_pages == 12
    used = table[table >= 0].tolist()
    assert len(used) == 8 and len(set(used)) == 8 and all(0 <= x < n_pages for x in used)  # distinct, in range
    assert (table[0, 2:] == -1).all() and (table[2] == -1).all()                         # entries past need
    assert W.pages_needed([0, 1, 128, 129, 8192]).tolist() == [0, 1, 1, 2, 64]


def test_to_pages_and_from_pages_round_trip():
    B, Tmax = 2, 300  # Tmax not a multiple of the page size: the last page is partly filler
    cache = torch.arange(B * Tmax * 8 * 128, dtype=torch.float32).remainder(997).to(torch.bfloat16)
    cache = cache.view(B, Tmax, 8, 128)
    table, n_pages = W.page_table(B, 3, [3, 3], spare=2, seed=10)
    pool = W.to_pages(cache, table, n_pages, seed=11)
    assert pool.shape == (n_pages, W.PAGE_TOKENS, 8, 128)
    for b in range(B):
        assert torch.equal(W.from_pages(pool, table, b, Tmax), cache[b])
        assert torch.equal(pool[table[b, 1]], cache[b, 128:256])   # a page holds its 128 consecutive rows
