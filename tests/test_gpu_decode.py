"""K3 + K4 parity: split-K decode and combine against the exact fp64 oracle."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as A
from tests.gpu_util import cached_inputs, oracle_append, run_decode
from tests.parity_util import assert_close

pytestmark = pytest.mark.gpu


def _check(inp, what, kv_len=None):
    oq, ok_, ov, out, status = run_decode(inp, kv_len=kv_len)
    assert status == 0
    rq, rk, rv = oracle_append(inp)
    assert np.array_equal(oq, rq[:, 0]) and np.array_equal(ok_, rk) and np.array_equal(ov, rv)
    kv = inp.start_pos.numpy() + 1 if kv_len is None else np.asarray(kv_len)
    ref = A.decode(rq[:, 0], rk, rv, kv)
    return assert_close(out, ref, what)


def test_decode_full_size_every_output():
    _check(cached_inputs("decode_b32_ctx8192"), "decode_b32_ctx8192")


def test_decode_split_boundaries():
    # kv_len = 1, 2, 512, 513, 1023, 1024, 1025, 2048: one row, stage and split edges
    # (a split is GROK_DECODE_SPLIT = 1024 rows), a full cache
    inp = W.custom(B=8, T=1, Tmax=2048, start_pos=[0, 1, 511, 512, 1022, 1023, 1024, 2047], seed=31)
    _check(inp, "split edges")


def test_decode_never_reads_rows_beyond_kv_len():
    a = W.custom(B=4, T=1, Tmax=1024, start_pos=[0, 100, 600, 1000], seed=32, junk="finite")
    b = W.custom(B=4, T=1, Tmax=1024, start_pos=[0, 100, 600, 1000], seed=32, junk="nan")
    assert np.array_equal(run_decode(a)[3], run_decode(b)[3])


def test_decode_equals_prefill_row():
    """A decode step at position t reproduces row t of a prefill over the same cache."""
    from tests.gpu_util import run_prefill
    T = 700
    pre = W.custom(B=1, T=T, Tmax=T, start_pos=[0], seed=33)
    oq, ok_, ov, out, status = run_prefill(pre)
    assert status == 0
    import torch
    import grok_gqa_attention_gb300 as G
    dev = "cuda"
    ck, cv = W.from_bits(ok_).to(dev), W.from_bits(ov).to(dev)
    ws = G.alloc_decode_workspace(1, T, dev)
    for t in (0, 1, 511, 512, 699):
        q = W.from_bits(oq[:, t]).contiguous().to(dev)
        kv = torch.tensor([t + 1], dtype=torch.int32, device=dev)
        dout = torch.empty((1, 48, 128), dtype=torch.bfloat16, device=dev)
        G.decode_step(q, ck, cv, kv, ws, dout)
        torch.cuda.synchronize()
        got = W.bits(dout.cpu())[0]
        assert_close(got, out[0, t], f"decode vs prefill row {t}")


def test_decode_bad_kv_len_sets_status():
    import grok_gqa_attention_gb300 as G
    inp = W.custom(B=3, T=1, Tmax=256, start_pos=[5, 6, 7], seed=34)
    *_, status = run_decode(inp, kv_len=[6, 0, 300])
    assert status & G.DEV_BAD_KV_LEN


def test_workspace_query_and_small_workspace_rejected():
    import torch
    import grok_gqa_attention_gb300 as G
    nbytes, splits = G.decode_workspace(32, 8192)
    assert splits == 8192 // G.DECODE_SPLIT and nbytes >= 32 * 8 * splits * (6 * 128 + 6) * 4
    inp = W.custom(B=2, T=1, Tmax=1024, start_pos=[3, 4], seed=35)
    dev = "cuda"
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    q = inp.q[:, 0].contiguous().to(dev)
    kv = torch.tensor([4, 5], dtype=torch.int32, device=dev)
    small = torch.empty(256, dtype=torch.uint8, device=dev)
    with pytest.raises(G.GrokError):
        G.decode(q, ck, cv, kv, small)
