"""The host-buffer prefill pipeline gives the same bits as the device entry points.

Several chunked-prefill steps are queued back to back (their copies overlap
each other's kernels); each step's output and the final caches must equal, bit
for bit, those of grok_rope_kv_append + grok_attn_prefill_ws called step by
step on device tensors, which the other parity tests hold to the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import grok_gqa_attention_gb300 as G
import workloads as W

pytestmark = pytest.mark.gpu

B, T, TMAX, STEPS = 2, 160, 640, 4


def _steps():
    out = []
    for s in range(STEPS):
        start = [s * T, s * T]
        valid = None if s % 2 == 0 else [T, 97 + 13 * s]
        inp = W.custom(B=B, T=T, Tmax=TMAX, start_pos=start, valid_len=valid, seed=40 + s)
        out.append(inp)
    return out


def _caches():
    base = W.custom(B=B, T=T, Tmax=TMAX, start_pos=[0, 0], seed=39, junk="finite")
    return base.cache_k, base.cache_v


def _host_out(kind):
    """Host output buffer: page-locked (copies overlap the kernels) or pageable
    (copies serialise)."""
    shape = (B, T, 48, 128)
    if kind == "pinned":
        return torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    return torch.empty(shape, dtype=torch.bfloat16)


@pytest.mark.parametrize("out_kind", ["pinned", "pageable"])
def test_pipeline_matches_step_by_step_device_calls(out_kind):
    steps = _steps()
    ck0, cv0 = _caches()
    # reference: device entry points, one step after another
    ck, cv = ck0.cuda(), cv0.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = []
    for inp in steps:
        q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
        start = inp.start_pos.cuda()
        valid = None if inp.valid_len is None else inp.valid_len.cuda()
        q_rot = torch.empty_like(q)
        out = torch.empty_like(q)
        G.rope_kv_append(q, k, v, start, q_rot, ck, cv, status)
        G.prefill_ws(q_rot, ck, cv, start, valid, out, G.alloc_prefill_workspace(B, TMAX), status)
        ref.append(W.bits(out.cpu()))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_k, ref_v = W.bits(ck.cpu()), W.bits(cv.cpu())

    # pipeline: every step queued before one wait
    pk, pv = ck0.cuda(), cv0.cuda()
    pipe = G.prefill_pipe_create(B, T, TMAX, pk, pv)
    try:
        host_in, host_out = [], []
        for inp in steps:
            hin = [inp.q.pin_memory(), inp.k.pin_memory(), inp.v.pin_memory(), inp.start_pos.pin_memory(),
                   None if inp.valid_len is None else inp.valid_len.pin_memory()]
            hout = _host_out(out_kind)
            host_in.append(hin)
            host_out.append(hout)
            G.prefill_pipe_submit(pipe, B, T, *hin, hout)
        assert G.prefill_pipe_wait(pipe) == 0
    finally:
        G.prefill_pipe_destroy(pipe)
    for s in range(STEPS):
        assert np.array_equal(W.bits(host_out[s]), ref[s]), f"step {s}"
    assert np.array_equal(W.bits(pk.cpu()), ref_k) and np.array_equal(W.bits(pv.cpu()), ref_v)


def test_pipeline_reports_and_clears_device_status():
    ck0, cv0 = _caches()
    ck, cv = ck0.cuda(), cv0.cuda()
    pipe = G.prefill_pipe_create(B, T, TMAX, ck, cv)
    try:
        inp = _steps()[0]
        hq, hk, hv = inp.q.pin_memory(), inp.k.pin_memory(), inp.v.pin_memory()
        out = torch.empty((B, T, 48, 128), dtype=torch.bfloat16).pin_memory()
        bad_start = torch.tensor([0, TMAX - T + 1], dtype=torch.int32).pin_memory()  # start + T > Tmax
        G.prefill_pipe_submit(pipe, B, T, hq, hk, hv, bad_start, None, out)
        assert G.prefill_pipe_wait(pipe) & G.DEV_BAD_START
        good_start = torch.tensor([0, 0], dtype=torch.int32).pin_memory()
        G.prefill_pipe_submit(pipe, B, T, hq, hk, hv, good_start, None, out)
        assert G.prefill_pipe_wait(pipe) == 0
    finally:
        G.prefill_pipe_destroy(pipe)


def test_pipeline_argument_errors():
    ck0, cv0 = _caches()
    ck, cv = ck0.cuda(), cv0.cuda()
    with pytest.raises(G.GrokError):
        G.prefill_pipe_create(B, TMAX + 1, TMAX, ck, cv)  # T > Tmax (shapes of the caches still match)
    pipe = G.prefill_pipe_create(B, T, TMAX, ck, cv)
    try:
        lib = G.load()
        st = lib.grok_prefill_pipe_submit(pipe, None, None, None, None, None, None)
        assert st == 1  # GROK_ERR_INVALID_ARG, nothing queued
        assert G.prefill_pipe_wait(pipe) == 0
    finally:
        G.prefill_pipe_destroy(pipe)
    assert G.load().grok_prefill_pipe_destroy(ctypes.c_void_p()) == 0  # NULL is ignored
