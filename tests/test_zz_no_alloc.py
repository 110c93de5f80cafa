"""The decode step that allocates nothing (grok_attn_decode_step_static).

Some callers of this library cannot allocate device memory: a plugin whose host
framework owns every byte of device memory, or a serving loop with a fixed
memory plan that may not call cudaMalloc between steps. For them the library
keeps the decode partial sums in its own static device array. This test calls
that entry point through the C ABI twice in a row, with different shapes, and
checks each result against the ordinary decode + combine path with a
caller-owned workspace; the second call also shows that what the first call
left in the shared array does not leak into the next result.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _lib():
    from grok_gqa_attention_gb300 import build
    build.build()
    import grok_gqa_attention_gb300 as G
    return G, G.load()


def _inputs(inp, dev):
    import grok_gqa_attention_gb300 as G
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    q_rot = torch.empty_like(q)
    G.rope_kv_append(q, k, v, start, q_rot, ck, cv)
    kv_len = (start + 1).to(torch.int32)
    return q_rot[:, 0].contiguous(), ck, cv, kv_len


def _static_call(lib, q, ck, cv, kv_len, out, status):
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    B, Tmax = ck.shape[0], ck.shape[1]
    return lib.grok_attn_decode_step_static(p(q), p(ck), p(cv), p(kv_len), B, Tmax, p(out), p(status),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_workspace_decode_matches_workspace_decode_twice():
    G, lib = _lib()
    dev = "cuda"
    cases = [W.generate("decode_b32_ctx8192", seed=0),
             W.custom(B=5, T=1, Tmax=2048, start_pos=[0, 511, 512, 1500, 2047], seed=41)]
    for inp in cases:
        q, ck, cv, kv_len = _inputs(inp, dev)
        B, Tmax = ck.shape[0], ck.shape[1]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        got = torch.empty((B, 48, 128), dtype=torch.bfloat16, device=dev)
        assert _static_call(lib, q, ck, cv, kv_len, got, status) == 0, lib.grok_last_error()
        ws = G.alloc_decode_workspace(B, Tmax, dev)
        want = torch.empty_like(got)
        G.decode_step(q, ck, cv, kv_len, ws, want, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # the same kernels with the same arithmetic: the bits must be identical
        assert np.array_equal(W.bits(got.cpu()), W.bits(want.cpu())), f"static workspace B={B} Tmax={Tmax}"


def test_warm_static_call_allocates_no_device_memory():
    """After one warm-up call (which may load the library's device code and with it
    the static array), a further call leaves the device's free memory unchanged."""
    G, lib = _lib()
    dev = "cuda"
    inp = W.custom(B=4, T=1, Tmax=1024, start_pos=[0, 100, 511, 1023], seed=42)
    q, ck, cv, kv_len = _inputs(inp, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((4, 48, 128), dtype=torch.bfloat16, device=dev)
    assert _static_call(lib, q, ck, cv, kv_len, out, status) == 0, lib.grok_last_error()
    first = out.clone()   # torch allocates here, before the measurement
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    assert _static_call(lib, q, ck, cv, kv_len, out, status) == 0, lib.grok_last_error()
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert int(status.item()) == 0
    assert torch.equal(out, first)


def test_static_workspace_rejects_shapes_beyond_its_size():
    G, lib = _lib()
    nbytes, _ = G.decode_workspace(128, 8192)
    assert nbytes > 16 << 20
    n = ctypes.c_void_p(0)
    rc = lib.grok_attn_decode_step_static(n, n, n, n, 128, 8192, n, n, n)
    assert rc == 1
    assert b"static workspace" in lib.grok_last_error()
