#!/usr/bin/env python3
"""Benchmark of the Grok-1 GQA attention core on GB300: prints ONE JSON line.

A step is one pass of the prefill hot path over the long causal prefill
(B=1, T=8192, 48 query / 8 KV heads, d=128, bf16): RoPE + KV-cache append,
then soft-capped causal GQA attention (grok_attn_prefill_ws: fp16 softmax
weights, fp16 copy of V in a workspace). `value` is algorithmic attention
TFLOP/s (48 heads x visible keys x 4 x 128 FLOP per query row) over the whole
step, inputs resident in HBM. The decode hot path (B=32, cached lengths uniform
in [1, 8191]: append, split-K decode, combine) is measured in the same run and
reported under "decode" in KV-cache GB/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (exact fp64 NumPy) on a bounded sample
of the same workload and metric. Under torchrun (N > 1) each rank runs an
independent replica (the path shards by sequence and KV head with no
exchange), times are max-reduced, and rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

PREFILL_WORKLOAD = "prefill_b1_t8192"
DECODE_WORKLOAD = "decode_b32_ctx8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-qkv", action="store_true")
    ap.add_argument("--no-paged", action="store_true", help="skip the paged-cache timings")
    ap.add_argument("--only", choices=["prefill", "decode", "qkv"], default=None,
                    help="run one workload only (profiling); implies --no-cpu-baseline --no-e2e")
    return ap.parse_args()


def time_stats(ms_list) -> dict:
    """Mean, median, min and 90th percentile of per-step kernel times (ms)."""
    a = np.asarray(ms_list, dtype=np.float64)
    return {"mean": float(a.mean()), "median": float(np.median(a)), "min": float(a.min()),
            "p90": float(np.percentile(a, 90))}


# ----------------------------------------------------------------------------- work counts
def prefill_flops(start: np.ndarray, valid, T: int) -> float:
    """48 heads x sum over query rows of visible keys x (2 QK + 2 PV) x 128."""
    total = 0
    i = np.arange(T, dtype=np.int64)
    for b, s in enumerate(start):
        n = T if valid is None else int(valid[b])
        total += int((np.minimum(s + i, s + n - 1) + 1).sum())
    return 48.0 * 4 * 128 * total


def decode_bytes(kv_len: np.ndarray) -> float:
    """K and V rows read once (8 heads x 128 x 2 B each) + q read + out written."""
    B = len(kv_len)
    return float(kv_len.astype(np.int64).sum() * 8 * 128 * 2 * 2 + 2 * B * 48 * 128 * 2)


def append_bytes(B: int, T: int) -> float:
    """q, k, v read and q_rot, cache rows written: 2 x B x T x (48 + 8 + 8) x 128 x 2 B."""
    return 2.0 * B * T * 64 * 128 * 2


def source_digest(*paths: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


KERNEL_SOURCES = {
    "qkv_kernel": ("grok_gqa_attention_gb300/csrc/qkv.cu", "grok_gqa_attention_gb300/csrc/common.cuh"),
    "prefill_kernel": ("grok_gqa_attention_gb300/csrc/prefill.cu", "grok_gqa_attention_gb300/csrc/common.cuh"),
    "decode_kernel": ("grok_gqa_attention_gb300/csrc/decode.cu", "grok_gqa_attention_gb300/csrc/common.cuh",
                      "include/grok_attn.h"),  # (the header fixes the split size)
}


def measured_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu capture, or None if the kernel changed since."""
    p = os.path.join(ROOT, "profiles", "kernel_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("source_sha256") != source_digest(*KERNEL_SOURCES[kernel]):
        return None
    return rec["dram_bytes_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(values, dist=None, device="cpu"):
    """Elementwise maximum of per-rank timings (identity on one rank)."""
    values = [float(x) for x in values]
    if dist is None:
        return values
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(work_per_rank: float, world: int, ms_max: float, scale: float) -> float:
    """Weak scaling: every rank processes work_per_rank units; the job ends with the slowest rank."""
    return world * work_per_rank / (ms_max * 1e-3) / scale


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.lines: list[str] = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- CPU oracle
_STATE = {}


def _oracle_init(name: str):
    import workloads as W
    from oracle import rope as R
    inp = W.generate(name)
    q_rot, ck, cv = R.rope_kv_append(W.bits(inp.q), W.bits(inp.k), W.bits(inp.v), inp.start_pos.numpy(),
                                     W.bits(inp.cache_k), W.bits(inp.cache_v))
    valid = None if inp.valid_len is None else inp.valid_len.numpy()
    _STATE.update(q_rot=q_rot, ck=ck, cv=cv, start=inp.start_pos.numpy(), valid=valid, T=inp.workload.T)


def _oracle_rows(rows):
    from oracle import attention as A
    st = _STATE
    t0 = time.perf_counter()
    A.attention_rows(st["q_rot"], st["ck"], st["cv"], st["start"], st["valid"], st["T"], rows)
    return time.perf_counter() - t0


class OraclePool:
    """The exact fp64 oracle on every host core (spawned workers, one BLAS thread each)."""

    def __init__(self, name: str):
        import workloads as W
        self.name = name
        self.T = W.WORKLOADS[name].T
        self.cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_init, initargs=(name,))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def rate(self, n_tokens: int, seed: int):
        """TFLOP/s of the oracle's attention over n_tokens sampled query tokens x 48 heads.

        Time = the slowest worker's attention time (the workers run concurrently).
        """
        rng = np.random.default_rng(seed)
        toks = np.sort(rng.choice(self.T, size=n_tokens, replace=False))
        rows = [(0, int(i), h) for i in toks for h in range(48)]
        chunks = [c for c in (rows[k::self.cores] for k in range(self.cores)) if c]
        times = self.pool.map(_oracle_rows, chunks)
        flops = sum(4.0 * 128 * (i + 1) for (_, i, _) in rows)   # empty-cache causal: row i sees i+1 keys
        return flops / max(times) / 1e12, max(times), len(chunks)

    def close(self):
        self.pool.close()
        self.pool.join()


def _oracle_c1_single_thread():
    """The whole tiny causal prefill (B1, T128) through the oracle in one process with one
    BLAS thread: the RoPE + append chain, then exact attention; seconds for each."""
    import workloads as W
    from oracle import attention as A
    from oracle import rope as R
    inp = W.generate("prefill_b1_t128")
    t0 = time.perf_counter()
    q_rot, ck, cv = R.rope_kv_append(W.bits(inp.q), W.bits(inp.k), W.bits(inp.v), inp.start_pos.numpy(),
                                     W.bits(inp.cache_k), W.bits(inp.cache_v))
    t1 = time.perf_counter()
    A.attention(q_rot, ck, cv, inp.start_pos.numpy(), None)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def cpu_baseline(n_tokens: int = 512) -> dict:
    pool = OraclePool(PREFILL_WORKLOAD)
    try:
        r, wall, used = pool.rate(n_tokens, seed=0)
    finally:
        pool.close()
    # the tiny causal prefill on one core (one spawned process, one BLAS thread)
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(1) as p1:
            t_rope, t_attn = p1.apply(_oracle_c1_single_thread)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    c1_flops = prefill_flops(np.zeros(1, dtype=np.int64), None, 128)
    return {"value": r, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
            "sample": (f"{n_tokens} random query tokens x 48 heads of {PREFILL_WORKLOAD}, exact fp64 NumPy "
                       f"oracle, attention only (RoPE/append precomputed), {wall:.1f} s on {used} cores"),
            "c1_single_thread": {"workload": "prefill_b1_t128", "threads": 1, "rope_append_s": t_rope,
                                 "attention_s": t_attn, "attention_TFLOP/s": c1_flops / t_attn / 1e12,
                                 "algorithmic_gflop": c1_flops / 1e9}}


# ----------------------------------------------------------------------------- GPU arm
def run_ours(args, rank: int, world: int, dist):
    import torch

    import grok_gqa_attention_gb300 as G
    import workloads as W
    from grok_gqa_attention_gb300 import build as gbuild

    gbuild.build()
    G.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_kind = load_peaks()

    # ---------------- prefill workload
    inp = W.generate(PREFILL_WORKLOAD, seed=rank)
    w = inp.workload
    B, T, Tmax = w.B, w.T, w.Tmax
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    valid = None if inp.valid_len is None else inp.valid_len.to(dev)
    q_rot = torch.empty_like(q)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pf_ws = G.alloc_prefill_workspace(B, Tmax, dev)
    # cos/sin of every position, computed once (a model shares it across all layers and steps)
    cos_tab, sin_tab = G.rope_cos_sin(0, Tmax)
    flops = prefill_flops(inp.start_pos.numpy(), None if inp.valid_len is None else inp.valid_len.numpy(), T)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def step(e=None):
        if e is not None:
            e[0].record(stream)
        G.rope_kv_append_table(q, k, v, start, cos_tab, sin_tab, q_rot, ck, cv, status)
        if e is not None:
            e[1].record(stream)
        G.prefill_ws(q_rot, ck, cv, start, valid, out, pf_ws, status)
        if e is not None:
            e[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    time.sleep(0.5)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        step(ev[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end) / args.steps
    append_times = [e[0].elapsed_time(e[1]) for e in ev]
    prefill_times = [e[1].elapsed_time(e[2]) for e in ev]
    ms_append = float(np.mean(append_times))
    ms_prefill = float(np.mean(prefill_times))
    # context: the workspace-free prefill (softmax weights as bf16 hi + lo, two P V products)
    out_b = torch.empty_like(out)
    for _ in range(args.warmup):
        G.prefill(q_rot, ck, cv, start, valid, out_b, status)
    ev_b = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e in ev_b:
        e[0].record(stream)
        G.prefill(q_rot, ck, cv, start, valid, out_b, status)
        e[1].record(stream)
    torch.cuda.synchronize()
    bf16p_times = [a.elapsed_time(b_) for a, b_ in ev_b]
    # context: the append that evaluates its cos/sin per token instead of reading the table
    q_rot_e = torch.empty_like(q_rot)
    for _ in range(args.warmup):
        G.rope_kv_append(q, k, v, start, q_rot_e, ck, cv, status)
    ev_e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e in ev_e:
        e[0].record(stream)
        G.rope_kv_append(q, k, v, start, q_rot_e, ck, cv, status)
        e[1].record(stream)
    torch.cuda.synchronize()
    append_eval_times = [a.elapsed_time(b_) for a, b_ in ev_e]
    if not torch.equal(q_rot_e.view(torch.int16), q_rot.view(torch.int16)):
        raise RuntimeError("the table append and the evaluating append differ")
    del q_rot_e
    diff = (out.float() - out_b.float()).abs()
    bf16p = {"call": "grok_attn_prefill (no workspace; P as bf16 hi + lo)", "ms": float(np.mean(bf16p_times)),
             "stats": time_stats(bf16p_times), "TFLOP/s": flops / (float(np.mean(bf16p_times)) * 1e-3) / 1e12,
             "max_abs_diff_to_fp16_path": float(diff.max()), "mean_abs_diff_to_fp16_path": float(diff.mean())}
    del out_b, diff
    ms, ms_prefill, ms_append = max_over_ranks([ms, ms_prefill, ms_append], dist, dev)
    value = whole_job_rate(flops, world, ms, 1e12)
    prefill_tflops = flops / (ms_prefill * 1e-3) / 1e12
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    result = {
        "metric": "prefill attention TFLOP/s and decode KV-cache GB/s, % of GB300 roofline",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded randn*3 -> bf16, causal, empty cache)",
        "config": {"workload": PREFILL_WORKLOAD, "B": B, "T": T, "Tmax": Tmax, "q_heads": 48, "kv_heads": 8,
                   "head_dim": 128, "algorithmic_gflop_per_step": flops / 1e9,
                   "l2": "inputs larger than L2 (q, q_rot, out 100 MB each + caches 34 MB)",
                   "parallelism": f"replicas x{world} (independent sequences, no exchange)"},
        "kernels_ms": {"rope_kv_append": ms_append, "prefill": ms_prefill},
        "kernels_ms_stats": {"rope_kv_append": time_stats(append_times), "prefill": time_stats(prefill_times)},
        "roofline": {"bound": "tensor",
                     "kernel": "prefill_kernel<fp16> (timed over the whole grok_attn_prefill_ws call: V pre-pass, "
                               "fp16 pass and the fallback pass)",
                     "achieved": prefill_tflops, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": prefill_tflops / peak_tf, "peak_source": f"bf16_tflops ({peak_kind})",
                     "frac_of_sustained": prefill_tflops / float(peaks.get("bf16_tflops_sustained",
                                                                          FALLBACK_PEAKS["bf16_tflops_sustained"])),
                     "traffic": measured_traffic("prefill_kernel"), "traffic_unit": "bytes per launch (ncu)"},
        "prefill_bf16_weights": bf16p,
        "append": {"call": "grok_rope_kv_append_table (cos/sin table of every position computed once "
                           "before timing, shared by all layers and steps)",
                   "GB/s": append_bytes(B, T) / (ms_append * 1e-3) / 1e9,
                   "frac_of_hbm": append_bytes(B, T) / (ms_append * 1e-3) / 1e9 / peak_bw,
                   "evaluating_cos_sin_per_token": {"call": "grok_rope_kv_append", "stats": time_stats(append_eval_times),
                                                    "GB/s": append_bytes(B, T) / (float(np.mean(append_eval_times)) * 1e-3) / 1e9}},
        "clocks": clk,
        # per step: append (table), V pre-pass, fp16 pass, fallback pass (the flag/list reset is a memset)
        "gpu_launches": 4 * args.steps,
    }

    # ---------------- end to end through the public API with host buffers
    if not args.no_e2e:
        qh = inp.q.pin_memory()
        kh = inp.k.pin_memory()
        vh = inp.v.pin_memory()
        sh = inp.start_pos.pin_memory()
        vlh = None if inp.valid_len is None else inp.valid_len.pin_memory()
        ohs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh, sh) + (() if vlh is None else (vlh,)))
        d2h = ohs[0].numel() * ohs[0].element_size()

        # (a) serial: copy in, both kernels, copy out, one step after another on one stream
        def e2e_serial_step():
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            start.copy_(sh, non_blocking=True)
            G.rope_kv_append_table(q, k, v, start, cos_tab, sin_tab, q_rot, ck, cv, status)
            G.prefill_ws(q_rot, ck, cv, start, valid, out, pf_ws, status)
            ohs[0].copy_(out, non_blocking=True)

        for _ in range(args.warmup):
            e2e_serial_step()
        torch.cuda.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            e2e_serial_step()
        b_.record(stream)
        torch.cuda.synchronize()
        ms_serial = a.elapsed_time(b_) / args.steps

        # (b) the library's host-buffer pipeline: each step's copy-in and copy-out
        # overlap the kernels of the neighbouring steps (three streams, double buffers)
        pipe = G.prefill_pipe_create(B, T, Tmax, ck, cv)
        try:
            for s_ in range(args.warmup):
                G.prefill_pipe_submit(pipe, B, T, qh, kh, vh, sh, vlh, ohs[s_ % 2])
            if G.prefill_pipe_wait(pipe) != 0:
                raise RuntimeError("device status set in the e2e pipeline")
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            for s_ in range(args.steps):
                G.prefill_pipe_submit(pipe, B, T, qh, kh, vh, sh, vlh, ohs[s_ % 2])
            pipe_status = G.prefill_pipe_wait(pipe)
            ms_pipe = (time.perf_counter() - t0) * 1e3 / args.steps
        finally:
            G.prefill_pipe_destroy(pipe)
        if pipe_status != 0:
            raise RuntimeError(f"device status {pipe_status} in the e2e pipeline")
        ms_pipe, ms_serial = max_over_ranks([ms_pipe, ms_serial], dist, dev)
        result["e2e"] = {"value": whole_job_rate(flops, world, ms_pipe, 1e12), "unit": "TFLOP/s",
                         "ms_per_step": ms_pipe, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "api": "grok_prefill_pipe_submit/_wait from page-locked host tensors (copies of one step "
                                "overlap the kernels of its neighbours; host wall clock over the K steps)",
                         "ms_per_step_serial": ms_serial,
                         "value_serial": whole_job_rate(flops, world, ms_serial, 1e12)}
        del qh, kh, vh, ohs
    del q, k, v, ck, cv, q_rot, out, pf_ws, cos_tab, sin_tab
    torch.cuda.empty_cache()

    # ---------------- the other prefill workloads: ragged batch and chunk on a warm cache
    result["other_prefill"] = run_other_prefill(args, rank, world, dist, dev, peaks, peak_kind)

    # ---------------- Q/K/V projection (the step in front of the attention call)
    if not args.no_qkv:
        result["qkv_projection"] = run_qkv(args, rank, world, dist, dev, peaks, peak_kind)

    # ---------------- decode workload
    if not args.no_decode:
        result["decode"] = run_decode(args, rank, world, dist, dev, peaks, peak_kind)

    # ---------------- paged KV cache: the same kernels through a shuffled block table
    if not args.no_paged:
        result["paged"] = run_paged(args, rank, dev)
    return result


def run_other_prefill(args, rank, world, dist, dev, peaks, peak_kind):
    """Append + prefill on the ragged batch (B8, T2048, valid lengths U[256, 2048]) and the
    chunk on a warm cache (B4, 256 tokens at 6144): CUDA events around each call."""
    import torch

    import grok_gqa_attention_gb300 as G
    import workloads as W
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    stream = torch.cuda.current_stream()
    res = {}
    for name in ("ragged_prefill_b8_t2048", "chunked_prefill_b4_t256_at6144"):
        inp = W.generate(name, seed=rank)
        w = inp.workload
        q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
        ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
        start = inp.start_pos.to(dev)
        valid = None if inp.valid_len is None else inp.valid_len.to(dev)
        valid_np = None if inp.valid_len is None else inp.valid_len.numpy()
        q_rot, out = torch.empty_like(q), torch.empty_like(q)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = G.alloc_prefill_workspace(w.B, w.Tmax, dev)
        flops = prefill_flops(inp.start_pos.numpy(), valid_np, w.T)
        cos_tab, sin_tab = G.rope_cos_sin(0, w.Tmax)
        calls = {"append": lambda: G.rope_kv_append_table(q, k, v, start, cos_tab, sin_tab, q_rot, ck, cv, status),
                 "prefill_ws": lambda: G.prefill_ws(q_rot, ck, cv, start, valid, out, ws, status),
                 "prefill_bf16_weights": lambda: G.prefill(q_rot, ck, cv, start, valid, out, status)}
        if name.startswith("chunked"):
            # steady state of a chunked prefill: the cached rows were converted by the calls
            # that appended them, so each call converts only its own 256 rows per sequence
            calls["prefill_ws_reusing_v_half"] = lambda: G.prefill_ws(q_rot, ck, cv, start, valid, out, ws, status,
                                                                      reuse_v_half=True)
        times = {}
        for key, fn in calls.items():
            for _ in range(args.warmup):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
            for e in evs:
                e[0].record(stream)
                fn()
                e[1].record(stream)
            torch.cuda.synchronize()
            times[key] = [a.elapsed_time(b_) for a, b_ in evs]
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in {name}")
        ms = {key: max_over_ranks([float(np.mean(t))], dist, dev)[0] for key, t in times.items()}
        entry = {"shape": {"B": w.B, "T": w.T, "Tmax": w.Tmax}, "algorithmic_gflop": flops / 1e9,
                 "ms": ms, "stats": {key: time_stats(t) for key, t in times.items()},
                 "prefill_TFLOP/s": flops / (ms["prefill_ws"] * 1e-3) / 1e12,
                 "roofline": {"bound": "tensor", "frac": flops / (ms["prefill_ws"] * 1e-3) / 1e12 / peak_tf,
                              "peak": peak_tf, "peak_source": f"bf16_tflops ({peak_kind})"},
                 "prefill_bf16_weights_TFLOP/s": flops / (ms["prefill_bf16_weights"] * 1e-3) / 1e12,
                 "step_TFLOP/s": whole_job_rate(flops, world, ms["append"] + ms["prefill_ws"], 1e12)}
        if valid_np is not None:
            # the padding query rows (i >= valid) are computed because the pages define them; without them:
            s0 = inp.start_pos.numpy()
            vis = sum(int((np.minimum(s0[b] + np.arange(int(n)), s0[b] + int(n) - 1) + 1).sum())
                      for b, n in enumerate(valid_np))
            entry["algorithmic_gflop_valid_rows_only"] = 48.0 * 4 * 128 * vis / 1e9
        if name.startswith("chunked"):
            entry["note"] = ("prefill_ws converts every cached V row [0, start + T) to fp16 each call (6400 rows "
                             "per sequence); prefill_ws_reusing_v_half converts only the chunk's rows, the rest "
                             "being in the workspace from the calls that appended them")
            entry["prefill_reusing_v_half_TFLOP/s"] = flops / (ms["prefill_ws_reusing_v_half"] * 1e-3) / 1e12
            entry["roofline_reusing_v_half"] = {"bound": "tensor", "frac": entry["prefill_reusing_v_half_TFLOP/s"] / peak_tf,
                                                "peak": peak_tf, "peak_source": f"bf16_tflops ({peak_kind})"}
        res[name] = entry
        del q, k, v, ck, cv, q_rot, out, ws, cos_tab, sin_tab
        torch.cuda.empty_cache()
    return res


def _to_pool(cache, table, n_pages):
    """Device-side scatter of a contiguous cache [B, Tmax, 8, 128] into pages (Tmax a multiple of 128)."""
    import torch
    B, Tmax = cache.shape[0], cache.shape[1]
    pages = cache.reshape(B * (Tmax // 128), 128, cache.shape[2], cache.shape[3])
    pool = torch.empty((n_pages, 128, cache.shape[2], cache.shape[3]), dtype=cache.dtype, device=cache.device)
    pool[table.reshape(-1).long().to(cache.device)] = pages
    return pool


def run_paged(args, rank, dev):
    """Kernel time of the paged calls against the contiguous calls on the same keys and values.

    Every page of the caches is placed at a random slot of a pool (a full random
    permutation), so consecutive key tiles of a sequence come from unrelated
    addresses. Eager launches alternate between the two layouts; CUDA events
    bracket each launch.
    """
    import torch

    import grok_gqa_attention_gb300 as G
    import workloads as W
    res = {}
    stream = torch.cuda.current_stream()
    n = max(4, min(args.steps, 20))

    def timed(fn):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b_.record(stream)
        return a, b_

    # prefill
    inp = W.generate(PREFILL_WORKLOAD, seed=rank)
    B, T, Tmax = inp.workload.B, inp.workload.T, inp.workload.Tmax
    q_rot = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=dev)
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    valid = None if inp.valid_len is None else inp.valid_len.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    G.rope_kv_append(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), start, q_rot, ck, cv, status)
    table, n_pages = W.page_table(B, Tmax // 128, [Tmax // 128] * B, spare=0, seed=100 + rank)
    kp, vp, tab = _to_pool(ck, table, n_pages), _to_pool(cv, table, n_pages), table.to(dev)
    out_c, out_p = torch.empty_like(q_rot), torch.empty_like(q_rot)
    for _ in range(2):
        G.prefill(q_rot, ck, cv, start, valid, out_c, status)
        G.prefill_paged(q_rot, kp, vp, tab, start, valid, out_p, status)
    ev_c, ev_p = [], []
    for _ in range(n):
        ev_c.append(timed(lambda: G.prefill(q_rot, ck, cv, start, valid, out_c, status)))
        ev_p.append(timed(lambda: G.prefill_paged(q_rot, kp, vp, tab, start, valid, out_p, status)))
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the paged prefill")
    same = bool(torch.equal(out_c.view(torch.int16), out_p.view(torch.int16)))
    mc = float(np.median([a.elapsed_time(b_) for a, b_ in ev_c]))
    mp = float(np.median([a.elapsed_time(b_) for a, b_ in ev_p]))
    res["prefill"] = {"workload": PREFILL_WORKLOAD, "pages": n_pages, "ms_contiguous": mc, "ms_paged": mp,
                      "paged_over_contiguous": mp / mc, "bit_identical": same, "calls": "grok_attn_prefill(_paged)"}
    # the fp16-weight calls (the bench step's prefill) on the same pages
    ws_c, ws_p = G.alloc_prefill_workspace(B, Tmax, dev), G.alloc_prefill_workspace(B, Tmax, dev)
    for _ in range(2):
        G.prefill_ws(q_rot, ck, cv, start, valid, out_c, ws_c, status)
        G.prefill_ws_paged(q_rot, kp, vp, tab, start, valid, out_p, ws_p, status)
    ev_c, ev_p = [], []
    for _ in range(n):
        ev_c.append(timed(lambda: G.prefill_ws(q_rot, ck, cv, start, valid, out_c, ws_c, status)))
        ev_p.append(timed(lambda: G.prefill_ws_paged(q_rot, kp, vp, tab, start, valid, out_p, ws_p, status)))
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the paged fp16 prefill")
    same = bool(torch.equal(out_c.view(torch.int16), out_p.view(torch.int16)))
    mc = float(np.median([a.elapsed_time(b_) for a, b_ in ev_c]))
    mp = float(np.median([a.elapsed_time(b_) for a, b_ in ev_p]))
    res["prefill_ws"] = {"workload": PREFILL_WORKLOAD, "pages": n_pages, "ms_contiguous": mc, "ms_paged": mp,
                         "paged_over_contiguous": mp / mc, "bit_identical": same,
                         "calls": "grok_attn_prefill_ws(_paged)"}
    del q_rot, ck, cv, kp, vp, out_c, out_p, ws_c, ws_p
    torch.cuda.empty_cache()

    # decode
    inp = W.generate(DECODE_WORKLOAD, seed=rank)
    B, Tmax = inp.workload.B, inp.workload.Tmax
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    kv_len = (inp.start_pos + 1).to(torch.int32).to(dev)
    q_rot = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=dev)
    G.rope_kv_append(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), start, q_rot, ck, cv, status)
    q1 = q_rot[:, 0].contiguous()
    table, n_pages = W.page_table(B, Tmax // 128, [Tmax // 128] * B, spare=0, seed=200 + rank)
    kp, vp, tab = _to_pool(ck, table, n_pages), _to_pool(cv, table, n_pages), table.to(dev)
    ws = G.alloc_decode_workspace(B, Tmax, dev)
    for _ in range(2):
        G.decode(q1, ck, cv, kv_len, ws, status)
        G.decode_paged(q1, kp, vp, tab, kv_len, ws, status)
    ev_c, ev_p = [], []
    for _ in range(n):
        ev_c.append(timed(lambda: G.decode(q1, ck, cv, kv_len, ws, status)))
        ev_p.append(timed(lambda: G.decode_paged(q1, kp, vp, tab, kv_len, ws, status)))
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the paged decode")
    mc = float(np.median([a.elapsed_time(b_) for a, b_ in ev_c]))
    mp = float(np.median([a.elapsed_time(b_) for a, b_ in ev_p]))
    nbytes = decode_bytes((inp.start_pos + 1).numpy())
    res["decode"] = {"workload": DECODE_WORKLOAD, "pages": n_pages, "ms_contiguous": mc, "ms_paged": mp,
                     "paged_over_contiguous": mp / mc, "GB/s_paged": nbytes / (mp * 1e-3) / 1e9}
    # prefill and decode: 2 kernels per pair of calls; the fp16 prefill: 3 per call (V copy, pass, fallback pass)
    res["gpu_launches"] = 4 * n + 8 + 3 * (2 * n + 4)
    return res


QKV_WORKLOAD = (1, 8192)  # B, T of the projection line: the prefill workload's tokens


def run_qkv(args, rank, world, dist, dev, peaks, peak_kind):
    """x [B,T,6144] . W [6144,8192] on tcgen05: plain (one launch) and fused with RoPE + append."""
    import torch
    import grok_gqa_attention_gb300 as G
    import workloads as W
    B, T = QKV_WORKLOAD
    Tmax = T
    inp = W.projection(B, T, Tmax, [0] * B, seed=rank)
    x, w = inp.x.to(dev), inp.w.to(dev)
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    M = B * T
    y = torch.empty((M, G.QKV_COLUMNS), dtype=torch.bfloat16, device=dev)
    q_rot = torch.empty((B, T, 48, 128), dtype=torch.bfloat16, device=dev)
    ws = G.alloc_qkv_workspace(B, T, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flops = 2.0 * M * G.MODEL_SIZE * G.QKV_COLUMNS
    stream = torch.cuda.current_stream()
    x2d = x.view(M, G.MODEL_SIZE)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for e in evs:
            e[0].record(stream)
            fn()
            e[1].record(stream)
        torch.cuda.synchronize()
        t = [a.elapsed_time(b) for a, b in evs]
        (m,) = max_over_ranks([float(np.mean(t))], dist, dev)
        return m, t

    ms_plain, t_plain = timed(lambda: G.qkv_project(x2d, w, y))
    ms_fused_step_table, t_fused_step_table = timed(lambda: G.qkv_rope_append(x, w, start, q_rot, ck, cv, ws, status))
    # the same with a cos/sin table of every position computed once (shared by all layers and steps)
    cos_tab, sin_tab = G.rope_cos_sin(0, Tmax)
    ms_fused, t_fused = timed(lambda: G.qkv_rope_append_table(x, w, start, cos_tab, sin_tab, q_rot, ck, cv, status))
    ms_cublas, _ = timed(lambda: torch.matmul(x2d, w))
    # output projection (the step after the attention call): [M, 6144] . W_o [6144, 6144]
    gen = torch.Generator().manual_seed(100 + rank)
    w_o = (torch.randn(G.MODEL_SIZE, G.MODEL_SIZE, generator=gen) / np.sqrt(G.MODEL_SIZE)).to(torch.bfloat16).to(dev)
    attn2d = q_rot.view(M, G.MODEL_SIZE)   # any [M, 6144] bf16 activation of the right scale
    y_o = torch.empty((M, G.MODEL_SIZE), dtype=torch.bfloat16, device=dev)
    ms_out, t_out = timed(lambda: G.linear(attn2d, w_o, y_o))
    flops_out = 2.0 * M * G.MODEL_SIZE * G.MODEL_SIZE
    # int8 weight-only Linear on the Q/K/V shape: dequantize (HBM-bound), then the bf16 product
    w8 = torch.randint(-127, 128, (G.MODEL_SIZE, G.QKV_COLUMNS), generator=gen, dtype=torch.int32).to(torch.int8).to(dev)
    scales = ((torch.rand(G.QKV_COLUMNS, generator=gen) + 0.5) * (3.0 / np.sqrt(G.MODEL_SIZE) / 73.0)).to(dev)
    w16 = torch.empty((G.MODEL_SIZE, G.QKV_COLUMNS), dtype=torch.bfloat16, device=dev)
    ms_deq, _ = timed(lambda: G.dequant_int8(w8, scales, w16))
    ms_i8, _ = timed(lambda: G.linear_int8(x2d, w8, scales, y, w16))
    deq_bytes = G.MODEL_SIZE * G.QKV_COLUMNS * 3 + G.QKV_COLUMNS * 4
    # decode-sized M (32 tokens): the one-pass int8 path against dequantize + bf16 product.
    # The 50 MB int8 weight fits in L2, so calls rotate over 5 distinct weights (250 MB,
    # as a decode step walks the layers), and 10 calls are replayed from a CUDA graph so
    # the device time is not hidden behind host launch overhead (a memset flush would
    # leave ~130 MB of dirty lines whose write-back the next call would pay for).
    xs, ys = x2d[:32], y[:32]
    w8r = [w8] + [torch.randint(-127, 128, w8.shape, generator=gen, dtype=torch.int32).to(torch.int8).to(dev)
                  for _ in range(4)]

    def timed_graph(fn_i):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for i in range(len(w8r)):
                fn_i(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(10):
                fn_i(i)
        ts = []
        for _ in range(max(3, min(args.steps, 10))):
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b_.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b_) / 10)
        del g
        (m,) = max_over_ranks([float(np.median(ts))], dist, dev)
        return m

    ms_i8s = timed_graph(lambda i: G.linear_int8(xs, w8r[i % len(w8r)], scales, ys, w16, stream=torch.cuda.current_stream()))
    ms_i8g = timed_graph(lambda i: (G.dequant_int8(w8r[i % len(w8r)], scales, w16, stream=torch.cuda.current_stream()),
                                    G.linear(xs, w16, ys, stream=torch.cuda.current_stream())))
    del w8r
    w8_bytes = G.MODEL_SIZE * G.QKV_COLUMNS
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the projection")
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tf_plain = flops / (ms_plain * 1e-3) / 1e12
    out = {
        "workload": f"qkv_b{B}_t{T}", "shape": {"M": M, "K": G.MODEL_SIZE, "N": G.QKV_COLUMNS},
        "metric": "Q/K/V projection TFLOP/s (2*M*K*N per step)",
        "value": whole_job_rate(flops, world, ms_fused, 1e12), "unit": "TFLOP/s", "ms_per_step": ms_fused,
        "step": ("grok_qkv_rope_append_table: projection GEMM with RoPE and cache-append epilogue, cos/sin from "
                 "a table of every position computed once before timing"),
        "plain": {"ms": ms_plain, "TFLOP/s": tf_plain, "stats": time_stats(t_plain)},
        "fused_stats": time_stats(t_fused),
        "fused_frac": flops / (ms_fused * 1e-3) / 1e12 / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
        "fused_with_per_call_table": {"call": "grok_qkv_rope_append (table kernel + GEMM, programmatic dependent)",
                                      "ms": ms_fused_step_table, "stats": time_stats(t_fused_step_table),
                                      "TFLOP/s": flops / (ms_fused_step_table * 1e-3) / 1e12},
        "roofline": {"bound": "tensor", "kernel": "qkv_kernel (plain epilogue, one launch)", "achieved": tf_plain,
                     "peak": peak_tf, "unit": "TFLOP/s", "frac": tf_plain / peak_tf,
                     "peak_source": f"bf16_tflops ({peak_kind})", "traffic": measured_traffic("qkv_kernel"),
                     "traffic_unit": "bytes per launch (ncu)"},
        "output_projection": {"shape": {"M": M, "K": G.MODEL_SIZE, "N": G.MODEL_SIZE}, "call": "grok_linear",
                              "ms": ms_out, "TFLOP/s": flops_out / (ms_out * 1e-3) / 1e12,
                              "frac": flops_out / (ms_out * 1e-3) / 1e12 / peak_tf, "stats": time_stats(t_out)},
        "int8_linear": {"call": "grok_linear_int8 (grok_dequant_int8 into a workspace, then grok_linear)",
                        "ms": ms_i8, "TFLOP/s": flops / (ms_i8 * 1e-3) / 1e12,
                        "dequant_ms": ms_deq, "dequant_GB/s": deq_bytes / (ms_deq * 1e-3) / 1e9,
                        "dequant_frac_of_hbm": deq_bytes / (ms_deq * 1e-3) / 1e9 / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                        "decode_sized": {"M": 32, "call": "grok_linear_int8 (one pass over the int8 weight)",
                                         "timing": "10 calls over 5 rotating 50 MB weights replayed from a CUDA graph "
                                                   "(inputs larger than L2), median over replays",
                                         "ms": ms_i8s, "weight_GB/s": w8_bytes / (ms_i8s * 1e-3) / 1e9,
                                         "weight_frac_of_hbm": w8_bytes / (ms_i8s * 1e-3) / 1e9 / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                                         "ms_dequant_then_linear": ms_i8g}},
        "cublas_context": {"op": "torch.matmul on the same bf16 product", "ms": ms_cublas,
                           "TFLOP/s": flops / (ms_cublas * 1e-3) / 1e12},
        "data": "synthetic (seeded randn -> bf16; weights randn*3/sqrt(6144))",
        "l2": "inputs larger than L2 (x 100 MB, W 100 MB, y 134 MB)",
        "gpu_launches": 10 * args.steps,
    }
    del x, w, ck, cv, y, q_rot, w_o, y_o, w8, w16
    torch.cuda.empty_cache()
    return out


def run_decode(args, rank, world, dist, dev, peaks, peak_kind):
    import torch

    import grok_gqa_attention_gb300 as G
    import workloads as W
    inp = W.generate(DECODE_WORKLOAD, seed=rank)
    B, Tmax = inp.workload.B, inp.workload.Tmax
    n_copies = 1 if args.only else 3  # rotate independent caches so every step reads from HBM, not L2
    caches = [(inp.cache_k.to(dev), inp.cache_v.to(dev)) for _ in range(n_copies)]
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    start = inp.start_pos.to(dev)
    kv_len = (inp.start_pos + 1).to(torch.int32).to(dev)
    q_rot = torch.empty_like(q)
    ws = G.alloc_decode_workspace(B, Tmax, dev)
    out = torch.empty((B, 48, 128), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    nbytes = decode_bytes((inp.start_pos + 1).numpy())
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def step(s, e=None):
        ck, cv = caches[s % n_copies]
        if e is not None:
            e[0].record(stream)
        G.rope_kv_append(q, k, v, start, q_rot, ck, cv, status)
        if e is not None:
            e[1].record(stream)
        G.decode(q_rot[:, 0], ck, cv, kv_len, ws, status)
        if e is not None:
            e[2].record(stream)
        G.combine(ws, kv_len, out, Tmax, status)
        if e is not None:
            e[3].record(stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    if dist:
        dist.barrier()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s in range(args.steps):
        step(s, ev[s])
    b_.record(stream)
    torch.cuda.synchronize()
    ms_eager = a.elapsed_time(b_) / args.steps
    dec_times = [e[1].elapsed_time(e[2]) for e in ev]
    comb_times = [e[2].elapsed_time(e[3]) for e in ev]
    app_times = [e[0].elapsed_time(e[1]) for e in ev]
    ms_dec, ms_comb, ms_app = (float(np.mean(x)) for x in (dec_times, comb_times, app_times))
    # The step as a serving loop runs it: the K steps captured once in a CUDA graph
    # and replayed, so the short launches per step cost no host round trips. The
    # timed graph uses the one-call step (grok_attn_decode_step: the three kernels
    # as programmatic dependents); the graph of three separate calls is timed too.
    step_ws = G.alloc_decode_step_workspace(B, Tmax, dev)

    def step_chained(s):
        ck, cv = caches[s % n_copies]
        G.decode_step_chained(q, k, v, start, ck, cv, step_ws, out, status)

    def graph_ms(fn):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for s in range(args.steps):
                fn(s)
        graph.replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        a.record(stream)
        graph.replay()
        b_.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b_) / args.steps

    ms_separate = graph_ms(step)
    ms = graph_ms(step_chained)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms, ms_dec = max_over_ranks([ms, ms_dec], dist, dev)
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs_step = whole_job_rate(nbytes, world, ms, 1e9)
    gbs_kernel = nbytes / (ms_dec * 1e-3) / 1e9
    return {
        "workload": DECODE_WORKLOAD, "value": gbs_step, "unit": "GB/s", "ms_per_step": ms,
        "timing": "K one-call steps (grok_attn_decode_step) replayed from one CUDA graph; kernel times from "
                  "events around eager launches of the three separate calls",
        "ms_per_step_eager": ms_eager,
        "ms_per_step_separate_calls_graph": ms_separate,
        "algorithmic_bytes_per_step": nbytes,
        "kernels_ms": {"rope_kv_append": ms_app, "decode": ms_dec, "combine": ms_comb},
        "kernels_ms_stats": {"rope_kv_append": time_stats(app_times), "decode": time_stats(dec_times),
                             "combine": time_stats(comb_times)},
        "l2": f"{n_copies} rotating cache copies of {nbytes / 1e6:.0f} MB used rows each",
        "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": gbs_kernel, "peak": peak_bw,
                     "unit": "GB/s", "frac": gbs_kernel / peak_bw, "peak_source": f"hbm_gbs ({peak_kind})",
                     "traffic": measured_traffic("decode_kernel"), "traffic_unit": "bytes per launch (ncu)"},
        "gpu_launches": 3 * args.steps,
        "api": "grok_attn_decode_step (append + decode + combine as programmatic dependents)",
    }


def run_reference(args):
    """The CPU oracle, as it stands, on a bounded sample of the prefill workload per step."""
    pool = OraclePool(PREFILL_WORKLOAD)
    n_tokens = 8
    try:
        rates, walls = [], []
        for s in range(args.steps):
            r, wall, cores = pool.rate(n_tokens, seed=1000 + s)
            rates.append(r)
            walls.append(wall)
    finally:
        pool.close()
    value = float(np.mean(rates))
    sample = (f"per step {n_tokens} random query tokens x 48 heads of {PREFILL_WORKLOAD}, exact fp64 NumPy oracle, "
              f"attention only (RoPE/append precomputed once)")
    return {
        "impl": "reference",
        "metric": "prefill attention TFLOP/s and decode KV-cache GB/s, % of GB300 roofline",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": float(np.mean(walls)) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded randn*3 -> bf16, causal, empty cache)",
        "config": {"workload": PREFILL_WORKLOAD, "B": 1, "T": 8192, "Tmax": 8192},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    if args.only:
        args.no_cpu_baseline = True
        args.no_e2e = True
        args.no_decode = args.only != "decode"
        args.no_qkv = args.only != "qkv"
        args.no_paged = True
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline()   # before any GPU work; the pool is spawned, never forked
    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    res = run_ours(args, rank, world, dist)
    if cpu is not None:
        res["cpu_baseline"] = cpu
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
