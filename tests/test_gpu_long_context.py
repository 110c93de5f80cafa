"""Parity at the largest supported cache: 65536 positions (GROK_MAX_POSITION).

A chunked prefill whose last token sits at the final position, a decode step
over a full 65536-row cache (64 splits), and the same prefill through a
512-page block table. Outputs are compared with the exact oracle: every
output of the decode step, sampled rows of the prefill (each one a dot
product against up to 65536 keys).
"""
import numpy as np
import pytest
import torch

import grok_gqa_attention_gb300 as G
import workloads as W
from oracle import attention as A
from tests.gpu_util import oracle_append, run_decode, run_prefill
from tests.parity_util import assert_close

pytestmark = pytest.mark.gpu

TMAX = G.MAX_POSITION  # 65536


def _rows(B, T, valid, n, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(B):
        for i in (0, 1, 127, 128, T - 1, int(valid[b]) - 1):
            rows.add((b, i, int(rng.integers(48))))
    while len(rows) < n:
        rows.add((int(rng.integers(B)), int(rng.integers(T)), int(rng.integers(48))))
    return sorted(rows)


def _check_rows(inp, out, what, n=40):
    rq, rk, rv = oracle_append(inp)
    B, T = inp.workload.B, inp.workload.T
    valid = np.full(B, T) if inp.valid_len is None else inp.valid_len.numpy()
    rows = _rows(B, T, valid, n, seed=5)
    ref, _ = A.attention_rows(rq, rk, rv, inp.start_pos.numpy(), valid, T, rows)
    got = np.stack([out[b, i, h] for b, i, h in rows])
    return assert_close(got, ref, what), (rq, rk, rv)


def test_prefill_chunk_ending_at_the_position_limit():
    # sequence 0's last token is position 65535; sequence 1 is a padded chunk mid-cache
    inp = W.custom(B=2, T=256, Tmax=TMAX, start_pos=[TMAX - 256, 30001], valid_len=[256, 200], seed=91)
    oq, ok_, ov, out, status = run_prefill(inp)
    assert status == 0
    _, (rq, rk, rv) = _check_rows(inp, out, "prefill at the position limit")
    assert np.array_equal(oq, rq)
    assert np.array_equal(ok_, rk) and np.array_equal(ov, rv)


def test_decode_over_a_full_65536_row_cache():
    inp = W.custom(B=2, T=1, Tmax=TMAX, start_pos=[TMAX - 1, 40000], seed=92)
    oq, ok_, ov, out, status = run_decode(inp)
    assert status == 0
    rq, rk, rv = oracle_append(inp)
    assert np.array_equal(ok_, rk) and np.array_equal(ov, rv)
    assert_close(out, A.decode(rq[:, 0], rk, rv, inp.start_pos.numpy() + 1), "decode at 65536")


def test_paged_prefill_at_the_position_limit():
    inp = W.custom(B=1, T=384, Tmax=TMAX, start_pos=[TMAX - 384], seed=93)
    _, _, _, ref_out, status = run_prefill(inp)  # contiguous
    assert status == 0
    max_pages = TMAX // W.PAGE_TOKENS
    table, n_pages = W.page_table(1, max_pages, [max_pages], spare=3, seed=94)
    kp = W.to_pages(inp.cache_k, table, n_pages, seed=95).cuda()
    vp = W.to_pages(inp.cache_v, table, n_pages, seed=96).cuda()
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    start, tab = inp.start_pos.cuda(), table.cuda()
    status_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot, out = torch.empty_like(q), torch.empty_like(q)
    G.rope_kv_append_paged(q, k, v, start, q_rot, kp, vp, tab, status_t)
    G.prefill_paged(q_rot, kp, vp, tab, start, None, out, status_t)
    torch.cuda.synchronize()
    assert int(status_t.item()) == 0
    assert np.array_equal(W.bits(out.cpu()), ref_out)
