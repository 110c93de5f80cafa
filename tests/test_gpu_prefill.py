"""K2 parity: prefill attention against the exact fp64 oracle."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as A
from tests.gpu_util import cached_inputs, oracle_append, run_prefill
from tests.parity_util import assert_close

pytestmark = pytest.mark.gpu

SMALL_CASES = {
    "t128": lambda: W.generate("prefill_b1_t128"),
    "ragged_tail_padding": lambda: W.custom(B=2, T=300, Tmax=384, start_pos=[0, 0], valid_len=[300, 217], seed=11),
    "chunk_unaligned_start": lambda: W.custom(B=2, T=200, Tmax=512, start_pos=[100, 37], seed=12),
    "single_token": lambda: W.custom(B=1, T=1, Tmax=8, start_pos=[0], seed=13),
    "valid_len_edges": lambda: W.custom(B=3, T=130, Tmax=1000, start_pos=[0, 500, 870], valid_len=[1, 130, 64],
                                        seed=14),
    "many_tiles": lambda: W.custom(B=1, T=1000, Tmax=1100, start_pos=[100], valid_len=[999], seed=15),
    # more sequences than the kernel stages in shared memory (512): the rest are read from global memory
    "many_sequences": lambda: W.custom(B=520, T=8, Tmax=24, start_pos=[(7 * b) % 17 for b in range(520)],
                                       valid_len=[1 + (5 * b) % 8 for b in range(520)], seed=16),
}


def _full_check(inp, what):
    oq, ok_, ov, out, status = run_prefill(inp)
    assert status == 0
    rq, rk, rv = oracle_append(inp)
    assert np.array_equal(oq, rq) and np.array_equal(ok_, rk) and np.array_equal(ov, rv)
    valid = None if inp.valid_len is None else inp.valid_len.numpy()
    ref = A.attention(rq, rk, rv, inp.start_pos.numpy(), valid)
    return assert_close(out, ref, what)


@pytest.mark.parametrize("case", list(SMALL_CASES))
def test_prefill_matches_oracle_elementwise(case):
    _full_check(SMALL_CASES[case](), case)


def _sample_rows(B, T, n, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(B):
        for i in (0, 1, 127, 128, T - 1, T // 2):
            if 0 <= i < T:
                rows.add((b, i, int(rng.integers(48))))
    while len(rows) < n:
        rows.add((int(rng.integers(B)), int(rng.integers(T)), int(rng.integers(48))))
    return sorted(rows)


def _whole_tiles(name, inp):
    """(b, first row) of the 128-row query tiles checked in full, every head:
    the first, a middle and the last tile of the long prefill; for the ragged
    batch the tile holding each sequence's last valid row (where its key padding
    starts); for the chunk on a warm cache both tiles of the first and last
    sequence."""
    w = inp.workload
    if name == "prefill_b1_t8192":
        return [(0, 0), (0, (w.T // 256) * 128), (0, w.T - 128)]
    if name == "ragged_prefill_b8_t2048":
        return [(b, ((int(n) - 1) // 128) * 128) for b, n in enumerate(inp.valid_len.numpy())]
    return [(b, i0) for b in (0, w.B - 1) for i0 in range(0, w.T, 128)]


@pytest.mark.parametrize("name", ["prefill_b1_t8192", "ragged_prefill_b8_t2048", "chunked_prefill_b4_t256_at6144"])
def test_prefill_full_size_whole_tiles_and_sampled_rows(name):
    inp = cached_inputs(name)
    oq, ok_, ov, out, status = run_prefill(inp)
    assert status == 0
    rq, rk, rv = oracle_append(inp)
    assert np.array_equal(oq, rq) and np.array_equal(ok_, rk) and np.array_equal(ov, rv)
    w = inp.workload
    valid = None if inp.valid_len is None else inp.valid_len.numpy()
    start = inp.start_pos.numpy()
    for b, i0 in _whole_tiles(name, inp):
        i1 = min(i0 + 128, w.T)
        ref = A.attention_block(rq, rk, rv, start, valid, w.T, b, i0, i1)
        assert_close(out[b, i0:i1], ref, f"{name} tile b={b} rows {i0}..{i1 - 1}")
    rows = _sample_rows(w.B, w.T, 160, seed=1)
    ref, _ = A.attention_rows(rq, rk, rv, start, valid, w.T, rows)
    got = np.stack([out[b, i, h] for (b, i, h) in rows])
    assert_close(got, ref, name)
    vals = W.from_bits(out).float()
    assert bool(vals.isfinite().all())


def test_prefill_never_reads_rows_beyond_the_memory_mask():
    """NaN in every cache row at or beyond start + T gives the same bits as finite junk."""
    a = W.custom(B=2, T=200, Tmax=512, start_pos=[100, 37], valid_len=[200, 150], seed=21, junk="finite")
    b = W.custom(B=2, T=200, Tmax=512, start_pos=[100, 37], valid_len=[200, 150], seed=21, junk="nan")
    oa = run_prefill(a)[3]
    ob = run_prefill(b)[3]
    assert np.array_equal(oa, ob)


def test_prefill_saturated_logits():
    """Large inputs push |logits| far past the cap: weights span exp(-60)..1."""
    inp = W.custom(B=1, T=256, Tmax=256, start_pos=[0], seed=22, scale=12.0)
    _full_check(inp, "saturated")


def test_prefill_all_weights_tiny():
    """Small inputs with all logits near zero: every weight near exp(-30) relative to the fixed reference."""
    inp = W.custom(B=1, T=192, Tmax=256, start_pos=[0], seed=23, scale=0.05)
    _full_check(inp, "tiny logits")


def test_prefill_one_visible_key_copies_v():
    """valid_len = 1: every row sees only key 0, so the output is v[0] exactly."""
    inp = W.custom(B=1, T=64, Tmax=64, start_pos=[0], valid_len=[1], seed=24)
    oq, ok_, ov, out, status = run_prefill(inp)
    assert status == 0
    want = np.repeat(ov[0, 0], 6, axis=0)     # [48, 128]: head h reads kv head h // 6
    for i in range(64):
        assert np.array_equal(out[0, i], want)


def test_prefill_bad_integers_set_status():
    import grok_gqa_attention_gb300 as G
    inp = W.custom(B=2, T=16, Tmax=32, start_pos=[0, 8], valid_len=[16, 0], seed=25)
    *_, status = run_prefill(inp)
    assert status & G.DEV_BAD_VALID
