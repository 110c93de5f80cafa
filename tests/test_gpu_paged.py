"""Paged KV cache: the paged calls give the bits of the contiguous calls.

A contiguous cache [B, Tmax, 8, 128] is scattered into a page pool through a
seeded random block table (pages in random order, spare pages in the pool,
table entries past what a sequence needs set to -1). The paged append, prefill
and decode must then reproduce the contiguous calls' results bit for bit, and
the pool, read back through the table, the contiguous caches. The contiguous
calls are held to the oracle by the other parity tests; one case per kernel
here also compares with the oracle directly.
"""
import numpy as np
import pytest
import torch

import grok_gqa_attention_gb300 as G
import workloads as W
from oracle import attention as A
from tests.gpu_util import oracle_append, run_append, run_prefill
from tests.parity_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
P = W.PAGE_TOKENS


def _paged_setup(inp, max_pages, need, seed, spare=3):
    table, n_pages = W.page_table(inp.workload.B, max_pages, need, spare=spare, seed=seed)
    kp = W.to_pages(inp.cache_k, table, n_pages, seed=seed + 1)
    vp = W.to_pages(inp.cache_v, table, n_pages, seed=seed + 2)
    return table, n_pages, kp, vp


def _run_append_paged(inp, table, kp, vp):
    q, k, v = (x.to(DEV) for x in (inp.q, inp.k, inp.v))
    kp, vp, tab = kp.to(DEV), vp.to(DEV), table.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q_rot = torch.empty_like(q)
    G.rope_kv_append_paged(q, k, v, inp.start_pos.to(DEV), q_rot, kp, vp, tab, status)
    torch.cuda.synchronize()
    return q_rot, kp, vp, tab, int(status.item())


def _gathered(pool, table, b, n_rows):
    return W.bits(W.from_pages(pool.cpu(), table, b, n_rows))


PREFILL_CASES = {
    # chunked prefill at unaligned starts, a padded tail, a sequence that ends mid-page
    "chunks": dict(B=3, T=200, Tmax=512, start_pos=[0, 130, 312], valid_len=[200, 150, 1], seed=61),
    # many pages per sequence, a start on a page boundary
    "long": dict(B=2, T=640, Tmax=1280, start_pos=[128, 500], valid_len=None, seed=62),
}


@pytest.mark.parametrize("case", list(PREFILL_CASES))
def test_paged_append_and_prefill_match_contiguous(case):
    c = PREFILL_CASES[case]
    inp = W.custom(**c)
    B, T, Tmax = c["B"], c["T"], c["Tmax"]
    max_pages = Tmax // P
    end = inp.start_pos.numpy() + T
    table, n_pages, kp0, vp0 = _paged_setup(inp, max_pages, W.pages_needed(end), seed=c["seed"])

    oq, ok_, ov, out, status = run_prefill(inp)  # contiguous
    assert status == 0

    q_rot, kp, vp, tab, st = _run_append_paged(inp, table, kp0, vp0)
    assert st == 0
    assert np.array_equal(W.bits(q_rot.cpu()), oq)
    for b in range(B):
        n = int(end[b])
        assert np.array_equal(_gathered(kp, table, b, n), ok_[b, :n]), f"k pages of sequence {b}"
        assert np.array_equal(_gathered(vp, table, b, n), ov[b, :n]), f"v pages of sequence {b}"
    used = set(int(x) for x in table.flatten() if x >= 0)
    for pg in range(n_pages):  # spare pages are never written
        if pg not in used:
            assert np.array_equal(W.bits(kp[pg].cpu()), W.bits(kp0[pg])) and np.array_equal(
                W.bits(vp[pg].cpu()), W.bits(vp0[pg]))

    start = inp.start_pos.to(DEV)
    valid = None if inp.valid_len is None else inp.valid_len.to(DEV)
    pout = torch.empty_like(q_rot)
    status_t = torch.zeros(1, dtype=torch.int32, device=DEV)
    G.prefill_paged(q_rot, kp, vp, tab, start, valid, pout, status_t)
    torch.cuda.synchronize()
    assert int(status_t.item()) == 0
    got = W.bits(pout.cpu())
    assert np.array_equal(got, out)
    if case == "chunks":  # and directly against the oracle
        rq, rk, rv = oracle_append(inp)
        vl = None if inp.valid_len is None else inp.valid_len.numpy()
        assert_close(got, A.attention(rq, rk, rv, inp.start_pos.numpy(), vl), "paged prefill")


WS_CASES = {
    "chunks": PREFILL_CASES["chunks"],
    # few items over long caches: the key-range split pass runs (48 items, 25-tile units)
    "split": dict(B=2, T=128, Tmax=4096, start_pos=[1500, 3000], valid_len=[128, 77], seed=64),
}


@pytest.mark.parametrize("case", list(WS_CASES))
def test_paged_fp16_prefill_matches_contiguous(case):
    """grok_attn_prefill_ws_paged reads K through the table and makes its fp16 copy of V
    through it: the bits equal grok_attn_prefill_ws over the contiguous caches, also when
    the second call of a chunked prefill reuses the copy (reuse_v_half)."""
    c = WS_CASES[case]
    inp = W.custom(**c)
    B, T, Tmax = c["B"], c["T"], c["Tmax"]
    max_pages = Tmax // P
    end = inp.start_pos.numpy() + T
    table, n_pages, kp0, vp0 = _paged_setup(inp, max_pages, W.pages_needed(end), seed=c["seed"])
    q_rot, ck, cv, st = run_append(inp, DEV)
    assert st == 0
    start = inp.start_pos.to(DEV)
    valid = None if inp.valid_len is None else inp.valid_len.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = G.alloc_prefill_workspace(B, Tmax, DEV)
    want = torch.empty_like(q_rot)
    G.prefill_ws(q_rot, ck, cv, start, valid, want, ws, status)
    q_rot_p, kp, vp, tab, st = _run_append_paged(inp, table, kp0, vp0)
    assert st == 0
    wsp = G.alloc_prefill_workspace(B, Tmax, DEV)
    got = torch.empty_like(q_rot)
    for reuse in (False, True):
        got.zero_()
        G.prefill_ws_paged(q_rot_p, kp, vp, tab, start, valid, got, wsp, status, reuse_v_half=reuse)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(W.bits(got.cpu()), W.bits(want.cpu())), f"reuse_v_half={reuse}"
    rq, rk, rv = oracle_append(inp)
    vl = None if inp.valid_len is None else inp.valid_len.numpy()
    assert_close(W.bits(got.cpu()), A.attention(rq, rk, rv, inp.start_pos.numpy(), vl), f"paged fp16 prefill {case}")


def test_paged_fp16_prefill_reports_a_bad_page():
    """A table entry outside the pool sets GROK_DEV_BAD_PAGE (the V copy and the K loads read
    page 0 in its place); the other sequence's rows keep the contiguous call's bits."""
    c = WS_CASES["chunks"]
    inp = W.custom(**c)
    B, T, Tmax = c["B"], c["T"], c["Tmax"]
    end = inp.start_pos.numpy() + T
    table, n_pages, kp0, vp0 = _paged_setup(inp, Tmax // P, W.pages_needed(end), seed=c["seed"])
    q_rot, ck, cv, st = run_append(inp, DEV)
    start = inp.start_pos.to(DEV)
    valid = inp.valid_len.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    want = torch.empty_like(q_rot)
    G.prefill_ws(q_rot, ck, cv, start, valid, want, G.alloc_prefill_workspace(B, Tmax, DEV), status)
    q_rot_p, kp, vp, tab, st = _run_append_paged(inp, table, kp0, vp0)
    assert st == 0
    tab[2, 0] = n_pages + 7   # sequence 2's first page id leaves the pool
    got = torch.empty_like(q_rot)
    G.prefill_ws_paged(q_rot_p, kp, vp, tab, start, valid, got, G.alloc_prefill_workspace(B, Tmax, DEV), status)
    torch.cuda.synchronize()
    assert int(status.item()) & G.DEV_BAD_PAGE
    assert np.array_equal(W.bits(got[:2].cpu()), W.bits(want[:2].cpu()))


def _decode(q_rot, ck, cv, kv_len, Tmax, table=None):
    B = q_rot.shape[0]
    ws = G.alloc_decode_workspace(B, Tmax, DEV)
    out = torch.empty((B, 48, 128), dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv = torch.as_tensor(np.asarray(kv_len, dtype=np.int32)).to(DEV)
    if table is None:
        G.decode(q_rot, ck, cv, kv, ws, status)
    else:
        G.decode_paged(q_rot, ck, cv, table.to(DEV), kv, ws, status)
    G.combine(ws, kv, out, Tmax, status)
    torch.cuda.synchronize()
    return W.bits(out.cpu()), int(status.item())


def test_paged_decode_matches_contiguous_and_oracle():
    # kv_len: one key, a full page, one past a page, a 512-key split edge, the whole capacity
    kv_len = [1, 128, 129, 513, 1024]
    Tmax = 1024
    inp = W.custom(B=5, T=1, Tmax=Tmax, start_pos=[k - 1 for k in kv_len], seed=63)
    q_rot, ck, cv, st = run_append(inp, DEV)
    assert st == 0
    q1 = q_rot[:, 0].contiguous()
    ref, st = _decode(q1, ck, cv, kv_len, Tmax)
    assert st == 0

    table, n_pages = W.page_table(5, Tmax // P, W.pages_needed(kv_len), spare=4, seed=64)
    kp = W.to_pages(ck.cpu(), table, n_pages, seed=65).to(DEV)
    vp = W.to_pages(cv.cpu(), table, n_pages, seed=66).to(DEV)
    got, st = _decode(q1, kp, vp, kv_len, Tmax, table)
    assert st == 0
    assert np.array_equal(got, ref)
    rq, rk, rv = oracle_append(inp)
    assert_close(got, A.decode(rq[:, 0], rk, rv, np.asarray(kv_len)), "paged decode")


def test_paged_decode_shared_prefix_pages():
    """Two sequences that name the same physical pages for a common prefix."""
    Tmax, prefix = 768, 256
    kv_len = [700, 300, 40]
    inp = W.custom(B=3, T=1, Tmax=Tmax, start_pos=[k - 1 for k in kv_len], seed=67)
    inp.cache_k[1, :prefix] = inp.cache_k[0, :prefix]  # sequence 1 shares sequence 0's first two pages
    inp.cache_v[1, :prefix] = inp.cache_v[0, :prefix]
    q_rot, ck, cv, st = run_append(inp, DEV)
    assert st == 0
    q1 = q_rot[:, 0].contiguous()
    ref, st = _decode(q1, ck, cv, kv_len, Tmax)
    assert st == 0
    table, n_pages = W.page_table(3, Tmax // P, W.pages_needed(kv_len), spare=2, seed=68)
    table[1, :prefix // P] = table[0, :prefix // P]
    kp = W.to_pages(ck.cpu(), table, n_pages, seed=69).to(DEV)
    vp = W.to_pages(cv.cpu(), table, n_pages, seed=70).to(DEV)
    got, st = _decode(q1, kp, vp, kv_len, Tmax, table)
    assert st == 0
    assert np.array_equal(got, ref)


def test_bad_page_ids_are_reported():
    Tmax = 512
    kv_len = [300, 200]
    inp = W.custom(B=2, T=1, Tmax=Tmax, start_pos=[k - 1 for k in kv_len], seed=71)
    q_rot, ck, cv, st = run_append(inp, DEV)
    q1 = q_rot[:, 0].contiguous()
    ref, _ = _decode(q1, ck, cv, kv_len, Tmax)
    table, n_pages = W.page_table(2, Tmax // P, W.pages_needed(kv_len), spare=0, seed=72)
    kp = W.to_pages(ck.cpu(), table, n_pages, seed=73).to(DEV)
    vp = W.to_pages(cv.cpu(), table, n_pages, seed=74).to(DEV)
    bad = table.clone()
    bad[1, 1] = n_pages  # a page sequence 1 reads
    got, st = _decode(q1, kp, vp, kv_len, Tmax, bad)
    assert st & G.DEV_BAD_PAGE
    assert np.array_equal(got[0], ref[0])  # the other sequence is unaffected
    bad[1, 1] = table[1, 1]
    bad[1, 3] = 12345  # past kv_len: never read
    got, st = _decode(q1, kp, vp, kv_len, Tmax, bad)
    assert st == 0 and np.array_equal(got, ref)

    # append: a bad page skips that token's cache write, still rotates q, reports
    pin = W.custom(B=2, T=150, Tmax=Tmax, start_pos=[0, 100], seed=75)
    end = pin.start_pos.numpy() + 150
    table, n_pages, kp0, vp0 = _paged_setup(pin, Tmax // P, W.pages_needed(end), seed=76, spare=0)
    qc, _, _, _ = run_append(pin, DEV)
    bad = table.clone()
    bad[0, 1] = -7  # rows 128..149 of sequence 0
    q_rot, kp, vp, tab, st = _run_append_paged(pin, bad, kp0, vp0)
    assert st & G.DEV_BAD_PAGE
    assert np.array_equal(W.bits(q_rot.cpu()), W.bits(qc.cpu()))
    assert np.array_equal(W.bits(kp[table[0, 1]].cpu()), W.bits(kp0[table[0, 1]]))  # untouched

    # prefill over a table with a bad page
    out = torch.empty_like(q_rot)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    G.prefill_paged(q_rot, kp, vp, tab, pin.start_pos.to(DEV), None, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) & G.DEV_BAD_PAGE


def test_paged_argument_errors():
    q_rot = torch.zeros((1, 48, 128), dtype=torch.bfloat16, device=DEV)
    kp = torch.zeros((2, P, 8, 128), dtype=torch.bfloat16, device=DEV)
    table = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    kv = torch.ones(1, dtype=torch.int32, device=DEV)
    ws = G.alloc_decode_workspace(1, P, DEV)
    lib = G.load()
    p = G._ptr
    s = G._stream(None)
    # null block table, zero pages, oversized capacity, short workspace
    assert lib.grok_attn_decode_paged(p(q_rot), p(kp), p(kp), 2, None, 1, p(kv), 1, p(ws), ws.numel(), None, s) == 1
    assert lib.grok_attn_decode_paged(p(q_rot), p(kp), p(kp), 0, p(table), 1, p(kv), 1, p(ws), ws.numel(), None, s) == 1
    assert lib.grok_attn_decode_paged(p(q_rot), p(kp), p(kp), 2, p(table), 1 << 20, p(kv), 1, p(ws), ws.numel(),
                                      None, s) == 1
    assert lib.grok_attn_decode_paged(p(q_rot), p(kp), p(kp), 2, p(table), 1, p(kv), 1, p(ws), 16, None, s) == 1
    q = torch.zeros((1, 4, 48, 128), dtype=torch.bfloat16, device=DEV)
    assert lib.grok_attn_prefill_paged(p(q), p(kp), p(kp), 2, p(table), 0, p(kv), None, 1, 4, p(q), None, s) == 1
    k = torch.zeros((1, 4, 8, 128), dtype=torch.bfloat16, device=DEV)
    qr = torch.empty_like(q)
    assert lib.grok_rope_kv_append_paged(p(q), p(k), p(k), p(kv), 1, 4, p(qr), p(kp), p(kp), 2, None, 1, None,
                                         s) == 1
    with pytest.raises(ValueError):
        G.decode_paged(q_rot, kp, kp[:1], table, kv, ws)  # pools of different sizes


def test_paged_fused_projection_matches_contiguous():
    """The projection + RoPE + append epilogue writes the same rows through the table."""
    B, T, Tmax = 2, 200, 512
    pin = W.projection(B=B, T=T, Tmax=Tmax, start_pos=[0, 130], seed=81)
    x, w = pin.x.to(DEV), pin.w.to(DEV)
    start = pin.start_pos.to(DEV)
    ws = G.alloc_qkv_workspace(B, T, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ck, cv = pin.cache_k.to(DEV), pin.cache_v.to(DEV)
    q_c = torch.empty((B, T, 48, 128), dtype=torch.bfloat16, device=DEV)
    G.qkv_rope_append(x, w, start, q_c, ck, cv, ws, status)

    end = pin.start_pos.numpy() + T
    table, n_pages = W.page_table(B, Tmax // P, W.pages_needed(end), spare=2, seed=82)
    kp0 = W.to_pages(pin.cache_k, table, n_pages, seed=83)
    vp0 = W.to_pages(pin.cache_v, table, n_pages, seed=84)
    kp, vp, tab = kp0.to(DEV), vp0.to(DEV), table.to(DEV)
    q_p = torch.empty_like(q_c)
    G.qkv_rope_append_paged(x, w, start, q_p, kp, vp, tab, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(W.bits(q_p.cpu()), W.bits(q_c.cpu()))
    rk, rv = W.bits(ck.cpu()), W.bits(cv.cpu())
    for b in range(B):
        n = int(end[b])
        assert np.array_equal(_gathered(kp, table, b, n), rk[b, :n]), f"k pages of sequence {b}"
        assert np.array_equal(_gathered(vp, table, b, n), rv[b, :n]), f"v pages of sequence {b}"

    bad = table.clone()
    bad[1, 2] = -1  # positions 256..329 of sequence 1
    kp, vp = kp0.to(DEV), vp0.to(DEV)
    G.qkv_rope_append_paged(x, w, start, q_p, kp, vp, bad.to(DEV), ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) & G.DEV_BAD_PAGE
    assert np.array_equal(W.bits(q_p.cpu()), W.bits(q_c.cpu()))  # q_rot is still written
    assert np.array_equal(W.bits(kp[table[1, 2]].cpu()), W.bits(kp0[table[1, 2]]))  # the page is untouched
