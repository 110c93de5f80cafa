"""Continuous-batching slot insertion against the oracle (ch. 6 §6.6.1).

A sequence prefilled on its own is inserted into a slot of a batch cache; the
batch cache must equal the oracle's insertion bit for bit, the slot's step must
be set, and a decode step over the whole batch must give, for that slot, the
oracle's decode of the inserted sequence.
"""
import numpy as np
import pytest
import torch

import grok_gqa_attention_gb300 as G
import workloads as W
from oracle import attention as A
from oracle import slots as S
from tests.gpu_util import oracle_append, run_append
from tests.parity_util import assert_close

pytestmark = pytest.mark.gpu


def test_insert_slot_matches_oracle_and_decodes():
    B, Tmax, L = 3, 1024, 600
    batch = W.custom(B=B, T=1, Tmax=Tmax, start_pos=[100, 900, 300], seed=101)
    single = W.custom(B=1, T=L, Tmax=L, start_pos=[0], seed=102)
    # the new request: prefill-append its L tokens on its own
    _, sk, sv, st = run_append(single)
    assert st == 0
    ck, cv = batch.cache_k.cuda(), batch.cache_v.cuda()
    step = torch.tensor([100, 900, 300], dtype=torch.int32, device="cuda")
    G.kv_insert_slot(ck, cv, 1, sk[0], sv[0], L, step, L)
    torch.cuda.synchronize()
    want_k = S.insert_slot(W.bits(batch.cache_k), 1, W.bits(sk.cpu()), L)
    want_v = S.insert_slot(W.bits(batch.cache_v), 1, W.bits(sv.cpu()), L)
    assert np.array_equal(W.bits(ck.cpu()), want_k) and np.array_equal(W.bits(cv.cpu()), want_v)
    assert step.cpu().tolist() == S.insert_step(np.array([100, 900, 300]), 1, L).tolist()

    # the next decode step of the whole batch: slot 1 continues the inserted sequence at position L
    q = W.custom(B=B, T=1, Tmax=Tmax, start_pos=[100, L, 300], seed=103)
    qd, kd, vd = (x.cuda() for x in (q.q, q.k, q.v))
    q_rot = torch.empty_like(qd)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.rope_kv_append(qd, kd, vd, step, q_rot, ck, cv, status)
    kv_len = step + 1
    ws = G.alloc_decode_workspace(B, Tmax)
    out = torch.empty((B, 48, 128), dtype=torch.bfloat16, device="cuda")
    G.decode_step(q_rot[:, 0].contiguous(), ck, cv, kv_len, ws, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle: append the new token into the oracle's inserted caches, decode slot 1
    q.cache_k[:] = W.from_bits(want_k)
    q.cache_v[:] = W.from_bits(want_v)
    rq, rk, rv = oracle_append(q)
    ref = A.decode(rq[:, 0], rk, rv, np.array([101, L + 1, 301]))
    assert_close(W.bits(out.cpu())[1], ref[1], "decode after slot insertion")


def test_insert_slot_argument_checks_and_no_op():
    ck = torch.zeros((2, 64, 8, 128), dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    src = torch.ones((32, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G.GrokError):
        G.kv_insert_slot(ck, cv, 2, src, src, 8)          # slot out of range
    with pytest.raises(G.GrokError):
        G.kv_insert_slot(ck, cv, 0, src, src, 33)         # more rows than the source holds
    with pytest.raises(G.GrokError):
        G.kv_insert_slot(ck, cv, 0, ck[0], cv[0], 8)      # source overlaps the slot
    step = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(G.GrokError):
        G.kv_insert_slot(ck, cv, 0, src, src, 8, step, 65)  # step beyond Tmax
    G.kv_insert_slot(ck, cv, 1, src, src, 0)              # nothing to do: no launch
    G.kv_insert_slot(ck, cv, 1, src, src, 0, step, 7)     # only the step
    torch.cuda.synchronize()
    assert step.cpu().tolist() == [0, 7] and int(ck.abs().sum()) == 0
