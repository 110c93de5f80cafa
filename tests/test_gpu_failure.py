"""Failure detection on the GPU without a fault: a bounded wait runs out on a
barrier nothing completes; the kernel reports GROK_DEV_TIMEOUT and returns, the
other waiting warp leaves through the abort flag, and the context stays usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    import grok_gqa_attention_gb300 as G
    dev = "cuda"
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flags = torch.zeros(2, dtype=torch.int32, device=dev)
    t0 = time.time()
    G.selftest_bounded_wait(status, flags, 2_000_000)       # ~1 ms of clock cycles
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert int(status.item()) & G.DEV_TIMEOUT
    assert flags.tolist() == [2, 2]
    # the context is still usable: a normal decode step runs afterwards
    x = torch.arange(10, device=dev).sum()
    assert int(x.item()) == 45


def test_selftest_rejects_bad_limits():
    import grok_gqa_attention_gb300 as G
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(G.GrokError):
        G.selftest_bounded_wait(status, flags, 0)
