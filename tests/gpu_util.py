"""GPU-side runners for the parity tests: copy seeded inputs to the device, call
the library through the binding (C ABI), bring the results back as bf16 bits."""
from __future__ import annotations

import functools

import numpy as np
import torch

import workloads as W


@functools.lru_cache(maxsize=4)
def cached_inputs(name: str, junk: str = "finite", seed: int = 0) -> W.Inputs:
    return W.generate(name, seed=seed, junk=junk)


def oracle_append(inp: W.Inputs):
    from oracle import rope as R
    return R.rope_kv_append(W.bits(inp.q), W.bits(inp.k), W.bits(inp.v), inp.start_pos.numpy(),
                            W.bits(inp.cache_k), W.bits(inp.cache_v))


def run_append(inp: W.Inputs, dev="cuda"):
    import grok_gqa_attention_gb300 as G
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    q_rot = torch.empty_like(q)
    G.rope_kv_append(q, k, v, start, q_rot, ck, cv, status)
    torch.cuda.synchronize()
    return q_rot, ck, cv, int(status.item())


PREFILL_IMPLS = ("bf16p", "f16p")  # grok_attn_prefill (P as bf16 hi + lo) and grok_attn_prefill_ws (fp16 P)


def run_prefill(inp: W.Inputs, dev="cuda", impl="bf16p"):
    """Append then prefill on the GPU; returns (q_rot, cache_k, cache_v, out) bits and status."""
    import grok_gqa_attention_gb300 as G
    q_rot, ck, cv, st = run_append(inp, dev)
    start = inp.start_pos.to(dev)
    valid = None if inp.valid_len is None else inp.valid_len.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q_rot)
    if impl == "f16p":
        ws = G.alloc_prefill_workspace(q_rot.shape[0], ck.shape[1], dev)
        G.prefill_ws(q_rot, ck, cv, start, valid, out, ws, status)
    else:
        G.prefill(q_rot, ck, cv, start, valid, out, status)
    torch.cuda.synchronize()
    return (W.bits(q_rot.cpu()), W.bits(ck.cpu()), W.bits(cv.cpu()), W.bits(out.cpu()),
            st | int(status.item()))


def run_decode(inp: W.Inputs, dev="cuda", kv_len=None):
    """Append the new token, then one decode step (decode + combine); returns bits and status."""
    import grok_gqa_attention_gb300 as G
    q_rot, ck, cv, st = run_append(inp, dev)
    B, Tmax = ck.shape[0], ck.shape[1]
    if kv_len is None:
        kv_len = inp.start_pos + 1
    kv = torch.as_tensor(np.asarray(kv_len, dtype=np.int32)).to(dev)
    ws = G.alloc_decode_workspace(B, Tmax, dev)
    out = torch.empty((B, 48, 128), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    G.decode_step(q_rot[:, 0].contiguous(), ck, cv, kv, ws, out, status)
    torch.cuda.synchronize()
    return (W.bits(q_rot[:, 0].contiguous().cpu()), W.bits(ck.cpu()), W.bits(cv.cpu()), W.bits(out.cpu()),
            st | int(status.item()))
