"""K1 parity: rotated Q and the appended KV cache must equal the oracle bit for bit."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import cached_inputs, oracle_append, run_append

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_append_bit_exact_at_full_size(name):
    inp = cached_inputs(name)
    q_rot, ck, cv, status = run_append(inp)
    assert status == 0
    oq, ok_, ov = oracle_append(inp)
    assert np.array_equal(W.bits(q_rot.cpu()), oq)
    assert np.array_equal(W.bits(ck.cpu()), ok_)   # written rows and untouched rows
    assert np.array_equal(W.bits(cv.cpu()), ov)


def test_append_positions_spread_over_supported_range():
    starts = [b * 4096 + (b * 37) % 256 for b in range(15)] + [65536 - 256]
    inp = W.custom(B=16, T=256, Tmax=65536, start_pos=starts, seed=3)
    q_rot, ck, cv, status = run_append(inp)
    assert status == 0
    oq, ok_, ov = oracle_append(inp)
    assert np.array_equal(W.bits(q_rot.cpu()), oq)
    assert np.array_equal(W.bits(ck.cpu()), ok_)
    assert np.array_equal(W.bits(cv.cpu()), ov)


def test_append_ragged_token_counts():
    for T in (1, 3, 129):
        inp = W.custom(B=3, T=T, Tmax=300, start_pos=[0, 7, 300 - T], seed=T)
        q_rot, ck, cv, status = run_append(inp)
        assert status == 0
        oq, ok_, ov = oracle_append(inp)
        assert np.array_equal(W.bits(q_rot.cpu()), oq)
        assert np.array_equal(W.bits(ck.cpu()), ok_)
        assert np.array_equal(W.bits(cv.cpu()), ov)


def test_append_invalid_start_sets_status_and_skips_sequence():
    import grok_gqa_attention_gb300 as G
    inp = W.custom(B=2, T=8, Tmax=16, start_pos=[4, 9], seed=5)   # 9 + 8 > 16
    q_rot, ck, cv, status = run_append(inp)
    assert status & G.DEV_BAD_START
    oq, ok_, ov = oracle_append(W.custom(B=2, T=8, Tmax=16, start_pos=[4, 0], seed=5))
    assert np.array_equal(W.bits(ck.cpu())[0], ok_[0])
    assert np.array_equal(W.bits(ck.cpu())[1], W.bits(inp.cache_k)[1])   # untouched
    assert np.array_equal(W.bits(cv.cpu())[1], W.bits(inp.cache_v)[1])


def test_append_host_argument_checks():
    import grok_gqa_attention_gb300 as G
    inp = W.custom(B=1, T=4, Tmax=8, start_pos=[0], seed=6)
    dev = "cuda"
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    with pytest.raises(G.GrokError):          # q_rot aliasing q is rejected by the library
        G.rope_kv_append(q, k, v, start, q, ck, cv)
    flat = torch.empty(q.numel() + 1, dtype=torch.bfloat16, device=dev)
    mis = flat[1:].view(q.shape)              # 2-byte offset: not 16-byte aligned
    with pytest.raises(G.GrokError):
        G.rope_kv_append(q, k, v, start, mis, ck, cv)


def test_cos_sin_table_bit_exact_for_every_supported_position():
    """All 65536 positions x 64 frequencies of the device table equal the oracle's fp32 values."""
    import grok_gqa_attention_gb300 as G
    from oracle import rope as R
    c, s = G.rope_cos_sin(0, R.MAX_POSITION)
    torch.cuda.synchronize()
    t = np.arange(R.MAX_POSITION, dtype=np.float32)[None, :]
    oc, os_ = R.cos_sin(R.phase(t, R.inv_freq(128)))
    assert np.array_equal(c.cpu().numpy().view(np.uint32), oc[0].view(np.uint32))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_[0].view(np.uint32))


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_append_from_table_bit_exact_at_full_size(name):
    """The table variant (cos/sin from a table of every position, filled once) writes the
    same bits as the oracle on every workload."""
    import grok_gqa_attention_gb300 as G
    inp = cached_inputs(name)
    dev = "cuda"
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    q_rot = torch.empty_like(q)
    ctab, stab = G.rope_cos_sin(0, inp.workload.Tmax)
    G.rope_kv_append_table(q, k, v, start, ctab, stab, q_rot, ck, cv, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    oq, ok_, ov = oracle_append(inp)
    assert np.array_equal(W.bits(q_rot.cpu()), oq)
    assert np.array_equal(W.bits(ck.cpu()), ok_)
    assert np.array_equal(W.bits(cv.cpu()), ov)


def test_append_from_table_positions_beyond_the_table_set_status():
    import grok_gqa_attention_gb300 as G
    inp = W.custom(B=2, T=8, Tmax=64, start_pos=[4, 40], seed=7)
    dev = "cuda"
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ctab, stab = G.rope_cos_sin(0, 32)          # covers positions [0, 32): sequence 1 needs 40..47
    G.rope_kv_append_table(q, k, v, start, ctab, stab, torch.empty_like(q), ck, cv, status)
    torch.cuda.synchronize()
    assert int(status.item()) & G.DEV_BAD_START
    assert np.array_equal(W.bits(ck.cpu())[1], W.bits(inp.cache_k)[1])   # untouched
