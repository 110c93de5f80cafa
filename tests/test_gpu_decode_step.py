"""The chained decode step (grok_attn_decode_step): append + decode + combine as
programmatic dependents must give the bits of the three separate calls.

Positions cover the cases where the stage holding the new row is loaded after
the wait: row 0 (kv_len 1), the last row of the first stage, the first row of a
stage, split edges and a full cache. Several steps are queued back to back with
no synchronisation in between (each step's decode overwrites the partial sums
the previous step's combine reads), and the chain is also captured in a CUDA
graph. One case is compared with the oracle directly.
"""
import numpy as np
import pytest
import torch

import grok_gqa_attention_gb300 as G
import workloads as W
from oracle import attention as A
from tests.gpu_util import oracle_append
from tests.parity_util import assert_close

pytestmark = pytest.mark.gpu

TMAX = 2048
POS = [0, 63, 64, 511, 512, 1023, 1500, TMAX - 1]


def _separate(inp, ck, cv, start):
    B = inp.workload.B
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    q_rot = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.rope_kv_append(q, k, v, start, q_rot, ck, cv, st)
    ws = G.alloc_decode_workspace(B, ck.shape[1])
    out = torch.empty((B, 48, 128), dtype=torch.bfloat16, device="cuda")
    G.decode_step(q_rot[:, 0].contiguous(), ck, cv, (start + 1).to(torch.int32), ws, out, st)
    return out, st


def test_chained_step_matches_separate_calls_and_oracle():
    inp = W.custom(B=len(POS), T=1, Tmax=TMAX, start_pos=POS, seed=111)
    start = inp.start_pos.cuda()
    ck1, cv1 = inp.cache_k.cuda(), inp.cache_v.cuda()
    ref, st1 = _separate(inp, ck1, cv1, start)
    ck2, cv2 = inp.cache_k.cuda(), inp.cache_v.cuda()
    ws = G.alloc_decode_step_workspace(len(POS), TMAX)
    out = torch.empty_like(ref)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.decode_step_chained(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), start, ck2, cv2, ws, out, st2)
    torch.cuda.synchronize()
    assert int(st1.item()) == 0 and int(st2.item()) == 0
    assert np.array_equal(W.bits(out.cpu()), W.bits(ref.cpu()))
    assert np.array_equal(W.bits(ck2.cpu()), W.bits(ck1.cpu())) and np.array_equal(W.bits(cv2.cpu()), W.bits(cv1.cpu()))
    rq, rk, rv = oracle_append(inp)
    assert_close(W.bits(out.cpu()), A.decode(rq[:, 0], rk, rv, np.asarray(POS) + 1), "chained decode step")


def _steps(n, B, seed):
    return [W.custom(B=B, T=1, Tmax=TMAX, start_pos=[100 + s, 700 + 3 * s, 63 + 64 * s], seed=seed + s)
            for s in range(n)]


def test_back_to_back_steps_and_graph_replay():
    B, n = 3, 4
    steps = _steps(n, B, 120)
    base = W.custom(B=B, T=1, Tmax=TMAX, start_pos=[0, 0, 0], seed=119, junk="finite")
    # reference: separate calls, synchronised after every step
    ck, cv = base.cache_k.cuda(), base.cache_v.cuda()
    ref = []
    for inp in steps:
        out, st = _separate(inp, ck, cv, inp.start_pos.cuda())
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref.append(W.bits(out.cpu()))
    ref_k, ref_v = W.bits(ck.cpu()), W.bits(cv.cpu())

    ins = [(s.q.cuda(), s.k.cuda(), s.v.cuda(), s.start_pos.cuda()) for s in steps]
    ws = G.alloc_decode_step_workspace(B, TMAX)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    # chained calls queued back to back on one stream, one workspace
    ck, cv = base.cache_k.cuda(), base.cache_v.cuda()
    outs = [torch.empty((B, 48, 128), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    for (q, k, v, sp), o in zip(ins, outs):
        G.decode_step_chained(q, k, v, sp, ck, cv, ws, o, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for s in range(n):
        assert np.array_equal(W.bits(outs[s].cpu()), ref[s]), f"step {s}"
    assert np.array_equal(W.bits(ck.cpu()), ref_k) and np.array_equal(W.bits(cv.cpu()), ref_v)

    # the same chain captured once in a CUDA graph and replayed
    ck, cv = base.cache_k.cuda(), base.cache_v.cuda()
    outs = [torch.zeros((B, 48, 128), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for (q, k, v, sp), o in zip(ins, outs):
            G.decode_step_chained(q, k, v, sp, ck, cv, ws, o, st)
    graph.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for s in range(n):
        assert np.array_equal(W.bits(outs[s].cpu()), ref[s]), f"graph step {s}"


def test_chained_step_status_and_arguments():
    inp = W.custom(B=2, T=1, Tmax=256, start_pos=[5, 9], seed=131)
    ck, cv = inp.cache_k.cuda(), inp.cache_v.cuda()
    ws = G.alloc_decode_step_workspace(2, 256)
    out = torch.empty((2, 48, 128), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([5, 256], dtype=torch.int32, device="cuda")  # position 256 does not fit Tmax 256
    G.decode_step_chained(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), bad, ck, cv, ws, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) & G.DEV_BAD_START
    with pytest.raises(G.GrokError):
        G.decode_step_chained(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.start_pos.cuda(), ck, cv, ws[:64], out)
