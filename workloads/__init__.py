"""Seeded synthetic inputs for the Grok-1 grouped-query attention core.

This module is the one piece shared by the CPU oracle's tests and by the CUDA
path's tests and benchmark. It holds shapes, seeds, value distributions and the
fill pattern of cache slots that no query may read, and none of the method's
arithmetic: no rotation, no logits, no softmax.

Recipe (the same for every workload): a ``torch.Generator`` seeded with ``seed``
draws, in this order, ``q [B,T,48,128]``, ``k [B,T,8,128]``, ``v [B,T,8,128]``,
``cache_k [B,Tmax,8,128]``, ``cache_v [B,Tmax,8,128]`` as ``randn * 3`` in fp32,
each rounded to bf16 (round to nearest even), then the per-sequence integers
(start positions for decode, valid lengths for ragged prefill) with
``torch.randint``. Warm cache rows stand for already-rotated keys. Every cache
row at or after ``start_pos[b]`` is then overwritten with junk (alternating
+-1e4, or NaN for a poison run): rows ``[start, start+T)`` must be written by the
append and rows beyond must never be read.

Projection inputs (``projection``): the same generator draws x [B,T,6144] as
``randn`` (std 1) and the side-by-side Q/K/V weights w [6144, 8192] as
``randn * 3 / sqrt(6144)`` (so projected q, k, v have std about 3, like the
attention inputs above), both rounded to bf16, then cache_k, cache_v and the
start positions as above.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

N_Q_HEADS = 48
N_KV_HEADS = 8
HEAD_DIM = 128

JUNK_VALUE = 1.0e4


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic attention workload.

    ``start`` is the per-sequence cache position of the first new token:
    ``("fixed", n)`` or ``("uniform", lo, hi)`` (inclusive, drawn per sequence).
    ``valid`` is the per-sequence count of non-padding new tokens:
    ``("full",)`` or ``("uniform", lo, hi)`` (inclusive).
    """

    name: str
    B: int
    T: int
    Tmax: int
    start: tuple
    valid: tuple
    description: str

    @property
    def is_decode(self) -> bool:
        return self.T == 1


WORKLOADS = {
    w.name: w
    for w in (
        Workload("prefill_b1_t128", 1, 128, 128, ("fixed", 0), ("full",),
                 "causal prefill, B=1, T=128, empty cache of 128 rows"),
        Workload("prefill_b1_t8192", 1, 8192, 8192, ("fixed", 0), ("full",),
                 "causal prefill, B=1, T=8192, cache of 8192 rows filled by the append"),
        Workload("decode_b32_ctx8192", 32, 1, 8192, ("uniform", 1, 8191), ("full",),
                 "one new token per sequence, B=32, cached lengths uniform in [1, 8191]"),
        Workload("ragged_prefill_b8_t2048", 8, 2048, 2048, ("fixed", 0), ("uniform", 256, 2048),
                 "causal plus key-padding prefill, B=8, padded T=2048, valid lengths uniform in [256, 2048]"),
        Workload("chunked_prefill_b4_t256_at6144", 4, 256, 8192, ("fixed", 6144), ("full",),
                 "256 new tokens at positions 6144..6399 over a warm cache, B=4, Tmax=8192"),
    )
}


@dataclasses.dataclass
class Inputs:
    """Host (CPU) tensors of one workload; bf16 tensors, int32 integer arrays."""

    workload: Workload
    q: torch.Tensor          # [B, T, 48, 128] bf16
    k: torch.Tensor          # [B, T, 8, 128] bf16
    v: torch.Tensor          # [B, T, 8, 128] bf16
    cache_k: torch.Tensor    # [B, Tmax, 8, 128] bf16
    cache_v: torch.Tensor    # [B, Tmax, 8, 128] bf16
    start_pos: torch.Tensor  # [B] int32
    valid_len: Optional[torch.Tensor]  # [B] int32, or None when every token is valid

    @property
    def kv_len(self) -> torch.Tensor:
        """Cache rows in use after the append: start_pos + T."""
        return (self.start_pos + self.workload.T).to(torch.int32)


def _randn_bf16(gen: torch.Generator, shape, scale: float) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    x.mul_(scale)
    return x.to(torch.bfloat16)


def _draw(gen: torch.Generator, spec: tuple, B: int) -> torch.Tensor:
    if spec[0] == "fixed":
        return torch.full((B,), spec[1], dtype=torch.int32)
    if spec[0] == "uniform":
        lo, hi = spec[1], spec[2]
        return torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64).to(torch.int32)
    raise ValueError(f"unknown spec {spec}")


def junk_rows_(cache: torch.Tensor, start_pos: torch.Tensor, kind: str = "finite") -> None:
    """Overwrite rows [start_pos[b], Tmax) of a [B,Tmax,8,128] bf16 cache in place."""
    if kind == "none":
        return
    B, Tmax = cache.shape[0], cache.shape[1]
    if kind == "finite":
        pattern = torch.tensor([JUNK_VALUE, -JUNK_VALUE], dtype=torch.float32).to(torch.bfloat16)
        fill = pattern.repeat(cache.shape[2] * cache.shape[3] // 2).view(cache.shape[2], cache.shape[3])
    elif kind == "nan":
        fill = torch.full((cache.shape[2], cache.shape[3]), float("nan"), dtype=torch.bfloat16)
    else:
        raise ValueError(kind)
    for b in range(B):
        s = int(start_pos[b])
        if s < Tmax:
            cache[b, s:] = fill


def generate(workload: Workload | str, seed: int = 0, junk: str = "finite",
             batch: Optional[int] = None, scale: float = 3.0) -> Inputs:
    """Draw the inputs of ``workload`` (see the module docstring for the recipe).

    ``batch`` overrides B (a smaller batch draws a different, still seeded,
    sample); ``junk`` is "finite", "nan" or "none".
    """
    w = WORKLOADS[workload] if isinstance(workload, str) else workload
    if batch is not None:
        w = dataclasses.replace(w, B=batch)
    B, T, Tmax = w.B, w.T, w.Tmax
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (B, T, N_Q_HEADS, HEAD_DIM), scale)
    k = _randn_bf16(gen, (B, T, N_KV_HEADS, HEAD_DIM), scale)
    v = _randn_bf16(gen, (B, T, N_KV_HEADS, HEAD_DIM), scale)
    cache_k = _randn_bf16(gen, (B, Tmax, N_KV_HEADS, HEAD_DIM), scale)
    cache_v = _randn_bf16(gen, (B, Tmax, N_KV_HEADS, HEAD_DIM), scale)
    start_pos = _draw(gen, w.start, B)
    valid_len = None if w.valid[0] == "full" else _draw(gen, w.valid, B)
    if int(start_pos.max()) + T > Tmax:
        raise ValueError(f"{w.name}: start_pos + T exceeds Tmax")
    junk_rows_(cache_k, start_pos, junk)
    junk_rows_(cache_v, start_pos, junk)
    return Inputs(w, q, k, v, cache_k, cache_v, start_pos, valid_len)


def custom(B: int, T: int, Tmax: int, start_pos, valid_len=None, seed: int = 0,
           junk: str = "finite", scale: float = 3.0) -> Inputs:
    """Inputs of arbitrary shape with explicit per-sequence integers (edge cases)."""
    start = torch.as_tensor(np.asarray(start_pos, dtype=np.int32))
    valid = None if valid_len is None else torch.as_tensor(np.asarray(valid_len, dtype=np.int32))
    w = Workload(f"custom_b{B}_t{T}_tmax{Tmax}", B, T, Tmax, ("given",), ("given",), "edge case")
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (B, T, N_Q_HEADS, HEAD_DIM), scale)
    k = _randn_bf16(gen, (B, T, N_KV_HEADS, HEAD_DIM), scale)
    v = _randn_bf16(gen, (B, T, N_KV_HEADS, HEAD_DIM), scale)
    cache_k = _randn_bf16(gen, (B, Tmax, N_KV_HEADS, HEAD_DIM), scale)
    cache_v = _randn_bf16(gen, (B, Tmax, N_KV_HEADS, HEAD_DIM), scale)
    junk_rows_(cache_k, start, junk)
    junk_rows_(cache_v, start, junk)
    return Inputs(w, q, k, v, cache_k, cache_v, start, valid)


def bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 storage of a bf16 tensor as a numpy array (no copy of values)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """A bf16 tensor whose storage is the given uint16 array."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)


MODEL_SIZE = 6144
QKV_COLUMNS = (N_Q_HEADS + 2 * N_KV_HEADS) * HEAD_DIM


@dataclasses.dataclass
class ProjectionInputs:
    """Host tensors for the Q/K/V projection: bf16 x, w, caches; int32 start positions."""

    x: torch.Tensor          # [B, T, 6144]
    w: torch.Tensor          # [6144, 8192]
    cache_k: torch.Tensor    # [B, Tmax, 8, 128]
    cache_v: torch.Tensor    # [B, Tmax, 8, 128]
    start_pos: torch.Tensor  # [B] int32


def projection(B: int, T: int, Tmax: int, start_pos, seed: int = 0, junk: str = "finite") -> ProjectionInputs:
    """Seeded projection inputs (recipe in the module docstring)."""
    gen = torch.Generator().manual_seed(seed)
    x = _randn_bf16(gen, (B, T, MODEL_SIZE), 1.0)
    w = _randn_bf16(gen, (MODEL_SIZE, QKV_COLUMNS), 3.0 / float(np.sqrt(MODEL_SIZE)))
    cache_k = _randn_bf16(gen, (B, Tmax, N_KV_HEADS, HEAD_DIM), 3.0)
    cache_v = _randn_bf16(gen, (B, Tmax, N_KV_HEADS, HEAD_DIM), 3.0)
    start = torch.as_tensor(np.asarray(start_pos, dtype=np.int32))
    junk_rows_(cache_k, start, junk)
    junk_rows_(cache_v, start, junk)
    return ProjectionInputs(x, w, cache_k, cache_v, start)


PAGE_TOKENS = 128


def page_table(B: int, max_pages: int, need, spare: int = 3, seed: int = 0, unused: int = -1):
    """A block table [B, max_pages] int32 over a pool of n_pages, and n_pages.

    Sequence b gets need[b] pages, drawn without replacement from the pool in a
    seeded random order (so logical neighbours are scattered); the pool holds
    `spare` pages that no sequence uses; table entries past need[b] hold `unused`.
    """
    need = np.asarray(need, dtype=np.int64)
    if need.shape != (B,) or (need < 0).any() or (need > max_pages).any():
        raise ValueError("need[b] must lie in [0, max_pages]")
    n_pages = int(need.sum()) + spare
    perm = np.random.default_rng(seed).permutation(n_pages)
    table = np.full((B, max_pages), unused, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, :need[b]] = perm[at:at + need[b]]
        at += need[b]
    return torch.from_numpy(table), n_pages


def pages_needed(end_positions) -> np.ndarray:
    """Pages that hold positions [0, end) for each end."""
    end = np.asarray(end_positions, dtype=np.int64)
    return (end + PAGE_TOKENS - 1) // PAGE_TOKENS


def to_pages(cache: torch.Tensor, table: torch.Tensor, n_pages: int, seed: int = 0) -> torch.Tensor:
    """Scatter a contiguous cache [B, Tmax, 8, 128] into a pool [n_pages, 128, 8, 128].

    Page table[b, j] receives rows [128 j, 128 j + 128) of sequence b (rows past
    Tmax stay as filler); pages no entry names are seeded random filler.
    """
    B, Tmax = cache.shape[0], cache.shape[1]
    gen = torch.Generator().manual_seed(seed)
    pool = _randn_bf16(gen, (n_pages, PAGE_TOKENS) + tuple(cache.shape[2:]), 3.0)
    for b in range(B):
        for j, pg in enumerate(table[b].tolist()):
            if 0 <= pg < n_pages:
                lo = j * PAGE_TOKENS
                hi = min(lo + PAGE_TOKENS, Tmax)
                if lo < hi:
                    pool[pg, :hi - lo] = cache[b, lo:hi]
    return pool


def from_pages(pool: torch.Tensor, table: torch.Tensor, b: int, n_rows: int) -> torch.Tensor:
    """Rows [0, n_rows) of sequence b gathered from a pool through the table."""
    rows = []
    for j in range((n_rows + PAGE_TOKENS - 1) // PAGE_TOKENS):
        pg = int(table[b, j])
        rows.append(pool[pg, :min(PAGE_TOKENS, n_rows - j * PAGE_TOKENS)])
    return torch.cat(rows, 0)
