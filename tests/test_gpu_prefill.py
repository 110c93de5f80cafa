"""K2 parity: prefill attention against the exact fp64 oracle, for both prefill
calls: grok_attn_prefill (softmax weights as bf16 hi + lo, no workspace) and
grok_attn_prefill_ws (fp16 weights with a lazily moved row maximum, fp16 copy
of V in a workspace, bf16 path for sequences whose V does not fit fp16)."""
import functools

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests.gpu_util import PREFILL_IMPLS, cached_inputs, oracle_append, run_prefill
from tests.parity_util import assert_close

pytestmark = pytest.mark.gpu

SMALL_CASES = {
    "t128": lambda: W.generate("prefill_b1_t128"),
    "ragged_tail_padding": lambda: W.custom(B=2, T=300, Tmax=384, start_pos=[0, 0], valid_len=[300, 217], seed=11),
    "chunk_unaligned_start": lambda: W.custom(B=2, T=200, Tmax=512, start_pos=[100, 37], seed=12),
    "single_token": lambda: W.custom(B=1, T=1, Tmax=8, start_pos=[0], seed=13),
    "valid_len_edges": lambda: W.custom(B=3, T=130, Tmax=1000, start_pos=[0, 500, 870], valid_len=[1, 130, 64],
                                        seed=14),
    "many_tiles": lambda: W.custom(B=1, T=1000, Tmax=1100, start_pos=[100], valid_len=[999], seed=15),
    # more sequences than the kernel stages in shared memory (512): the rest are read from global memory
    "many_sequences": lambda: W.custom(B=520, T=8, Tmax=24, start_pos=[(7 * b) % 17 for b in range(520)],
                                       valid_len=[1 + (5 * b) % 8 for b in range(520)], seed=16),
}


def _full_check(inp, what, impl):
    oq, ok_, ov, out, status = run_prefill(inp, impl=impl)
    assert status == 0
    rq, rk, rv = oracle_append(inp)
    assert np.array_equal(oq, rq) and np.array_equal(ok_, rk) and np.array_equal(ov, rv)
    valid = None if inp.valid_len is None else inp.valid_len.numpy()
    ref = A.attention(rq, rk, rv, inp.start_pos.numpy(), valid)
    return assert_close(out, ref, f"{what} [{impl}]")


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
@pytest.mark.parametrize("case", list(SMALL_CASES))
def test_prefill_matches_oracle_elementwise(case, impl):
    _full_check(SMALL_CASES[case](), case, impl)


def _sample_rows(B, T, n, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(B):
        for i in (0, 1, 127, 128, T - 1, T // 2):
            if 0 <= i < T:
                rows.add((b, i, int(rng.integers(48))))
    while len(rows) < n:
        rows.add((int(rng.integers(B)), int(rng.integers(T)), int(rng.integers(48))))
    return sorted(rows)


def _whole_tiles(name, inp):
    """(b, first row) of the 128-row query tiles checked in full, every head:
    the first, a middle and the last tile of the long prefill; for the ragged
    batch the tile holding each sequence's last valid row (where its key padding
    starts); for the chunk on a warm cache both tiles of the first and last
    sequence."""
    w = inp.workload
    if name == "prefill_b1_t8192":
        return [(0, 0), (0, (w.T // 256) * 128), (0, w.T - 128)]
    if name == "ragged_prefill_b8_t2048":
        return [(b, ((int(n) - 1) // 128) * 128) for b, n in enumerate(inp.valid_len.numpy())]
    return [(b, i0) for b in (0, w.B - 1) for i0 in range(0, w.T, 128)]


@functools.lru_cache(maxsize=1)
def _oracle_append_cached(name):
    return oracle_append(cached_inputs(name))


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
@pytest.mark.parametrize("name", ["prefill_b1_t8192", "ragged_prefill_b8_t2048", "chunked_prefill_b4_t256_at6144"])
def test_prefill_full_size_whole_tiles_and_sampled_rows(name, impl):
    inp = cached_inputs(name)
    oq, ok_, ov, out, status = run_prefill(inp, impl=impl)
    assert status == 0
    rq, rk, rv = _oracle_append_cached(name)
    assert np.array_equal(oq, rq) and np.array_equal(ok_, rk) and np.array_equal(ov, rv)
    w = inp.workload
    valid = None if inp.valid_len is None else inp.valid_len.numpy()
    start = inp.start_pos.numpy()
    for b, i0 in _whole_tiles(name, inp):
        i1 = min(i0 + 128, w.T)
        ref = A.attention_block(rq, rk, rv, start, valid, w.T, b, i0, i1)
        assert_close(out[b, i0:i1], ref, f"{name} tile b={b} rows {i0}..{i1 - 1} [{impl}]")
    rows = _sample_rows(w.B, w.T, 160, seed=1)
    ref, _ = A.attention_rows(rq, rk, rv, start, valid, w.T, rows)
    got = np.stack([out[b, i, h] for (b, i, h) in rows])
    assert_close(got, ref, f"{name} [{impl}]")
    vals = W.from_bits(out).float()
    assert bool(vals.isfinite().all())


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_never_reads_rows_beyond_the_memory_mask(impl):
    """NaN in every cache row at or beyond start + T gives the same bits as finite junk."""
    a = W.custom(B=2, T=200, Tmax=512, start_pos=[100, 37], valid_len=[200, 150], seed=21, junk="finite")
    b = W.custom(B=2, T=200, Tmax=512, start_pos=[100, 37], valid_len=[200, 150], seed=21, junk="nan")
    oa = run_prefill(a, impl=impl)[3]
    ob = run_prefill(b, impl=impl)[3]
    assert np.array_equal(oa, ob)


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_saturated_logits(impl):
    """Large inputs push |logits| far past the cap: weights span exp(-60)..1."""
    inp = W.custom(B=1, T=256, Tmax=256, start_pos=[0], seed=22, scale=12.0)
    _full_check(inp, "saturated", impl)


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_tanh_polynomial_range_split(impl):
    """The fp16 pass takes tanh from an FMA-pipe polynomial for half of a 32-key
    chunk's columns (pairs 0, 2, 4, ...: columns 0, 1, 4, 5, ...) when no logit
    of the warp's chunk in those columns exceeds 45 (|y| = 1.5) in magnitude,
    and tanh.approx otherwise. Keys per 32-key chunk: all small (logits within
    the range), one large key in a polynomial column, one in a tanh.approx
    column (the check ignores it), or all large."""
    inp = W.custom(B=1, T=512, Tmax=512, start_pos=[0], seed=27, scale=2.0)
    k = inp.k.float()
    for c in range(512 // 32):
        kind = c % 4
        if kind == 1:
            k[0, 32 * c] *= 10.0
        elif kind == 2:
            k[0, 32 * c + 2] *= 10.0
        elif kind == 3:
            k[0, 32 * c:32 * c + 32] *= 10.0
    inp.k.copy_(k.to(torch.bfloat16))
    _full_check(inp, "tanh polynomial range split", impl)


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_all_weights_tiny(impl):
    """Small inputs with all logits near zero: every weight near exp(-30) relative to the fixed reference."""
    inp = W.custom(B=1, T=192, Tmax=256, start_pos=[0], seed=23, scale=0.05)
    _full_check(inp, "tiny logits", impl)


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_row_maximum_rises_across_tiles(impl):
    """Keys of the first 128-key tile give logits near 0, later keys logits near +-30:
    a row's maximum rises by up to ~43 octaves after its first tile, far past the
    fp16 pass's headroom, so that pass lists the overflowing items and the bf16
    pass recomputes them (the middle tile rises only part of the way)."""
    inp = W.custom(B=1, T=400, Tmax=512, start_pos=[0], seed=26, scale=3.0)
    k = inp.k.float()
    k[:, :128] *= 0.02      # first tile: |logits| ~ 0.2 before the cap
    k[:, 128:256] *= 0.7    # second tile: part of the way up
    k[:, 256:] *= 4.0       # later tiles: saturated
    inp.k.copy_(k.to(torch.bfloat16))
    _full_check(inp, "rising maximum", impl)


def test_prefill_ws_hands_overflowing_items_to_the_bf16_pass():
    """In the rising-maximum case every row from 256 on sees keys whose capped logits reach
    about +-30 while its first tile's stay near 0: a rise of about 43 octaves, so its weights
    would overflow fp16, its item goes on the fallback list and the bf16 pass recomputes it:
    those rows equal grok_attn_prefill's output bit for bit. The first query tile (rows 0..127
    see only the small keys) stays on the fp16 path."""
    inp = W.custom(B=1, T=400, Tmax=512, start_pos=[0], seed=26, scale=3.0)
    k = inp.k.float()
    k[:, :128] *= 0.02
    k[:, 128:256] *= 0.7
    k[:, 256:] *= 4.0
    inp.k.copy_(k.to(torch.bfloat16))
    _, _, _, out16, st16 = run_prefill(inp, impl="f16p")
    _, _, _, outb, stb = run_prefill(inp, impl="bf16p")
    assert st16 == 0 and stb == 0
    assert np.array_equal(out16[0, 256:], outb[0, 256:])
    assert not np.array_equal(out16[0, :128], outb[0, :128])


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_values_beyond_fp16_range(impl):
    """V values above fp16's largest finite value (65504) in one sequence: the fp16
    path must run that sequence from the bf16 cache (the other sequence stays on
    fp16), with results matching the oracle."""
    inp = W.custom(B=2, T=300, Tmax=384, start_pos=[0, 20], valid_len=[300, 250], seed=27)
    v = inp.v.float()
    v[1, 5] *= 4e4           # |v| up to ~5e5 in sequence 1 (a visible row)
    inp.v.copy_(v.to(torch.bfloat16))
    assert float(inp.v[1].float().abs().max()) > 65504 and float(inp.v[0].float().abs().max()) < 65504
    oq, ok_, ov, out, status = run_prefill(inp, impl=impl)
    assert status == 0
    rq, rk, rv = oracle_append(inp)
    ref = A.attention(rq, rk, rv, inp.start_pos.numpy(), inp.valid_len.numpy())
    # sequence 0 keeps the usual absolute tolerance
    assert_close(out[0], ref[0], f"fp16-range sequence [{impl}]")
    # sequence 1's outputs reach ~1e5 where the big row has weight: errors relative to
    # each output row's scale (its largest |value|, at least 1)
    g = W.from_bits(out[1]).float().numpy()
    r = W.from_bits(ref[1]).float().numpy()
    row_scale = np.maximum(1.0, np.abs(r).max(axis=-1, keepdims=True))
    rel = np.abs(g - r) / row_scale
    assert np.isfinite(g).all()
    assert rel.max() <= 2.0 ** -7 and rel.mean() <= 1e-3, (float(rel.max()), float(rel.mean()))


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_one_visible_key_copies_v(impl):
    """valid_len = 1: every row sees only key 0, so the output is v[0] exactly."""
    inp = W.custom(B=1, T=64, Tmax=64, start_pos=[0], valid_len=[1], seed=24)
    oq, ok_, ov, out, status = run_prefill(inp, impl=impl)
    assert status == 0
    want = np.repeat(ov[0, 0], 6, axis=0)     # [48, 128]: head h reads kv head h // 6
    for i in range(64):
        assert np.array_equal(out[0, i], want)


@pytest.mark.parametrize("impl", PREFILL_IMPLS)
def test_prefill_bad_integers_set_status(impl):
    import grok_gqa_attention_gb300 as G
    inp = W.custom(B=2, T=16, Tmax=32, start_pos=[0, 8], valid_len=[16, 0], seed=25)
    *_, status = run_prefill(inp, impl=impl)
    assert status & G.DEV_BAD_VALID


def test_prefill_ws_reusing_the_fp16_copy_across_chunks():
    """A chunked prefill in two calls on one workspace: the second call converts only its
    own 300 rows of V (reuse_v_half) and must give the same bits as a call that converts
    every row, and match the oracle."""
    import grok_gqa_attention_gb300 as G
    dev = "cuda"
    B, Tmax = 2, 1024
    first = W.custom(B=B, T=300, Tmax=Tmax, start_pos=[0, 0], valid_len=[300, 300], seed=31)
    second = W.custom(B=B, T=300, Tmax=Tmax, start_pos=[300, 300], valid_len=[300, 211], seed=32)
    ck, cv = first.cache_k.to(dev), first.cache_v.to(dev)
    ws = G.alloc_prefill_workspace(B, Tmax, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = []
    for inp, reuse in ((first, False), (second, True)):
        q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
        start, valid = inp.start_pos.to(dev), inp.valid_len.to(dev)
        q_rot, out = torch.empty_like(q), torch.empty_like(q)
        G.rope_kv_append(q, k, v, start, q_rot, ck, cv, status)
        G.prefill_ws(q_rot, ck, cv, start, valid, out, ws, status, reuse_v_half=reuse)
        outs.append((q_rot, start, valid, out))
    q_rot, start, valid, out = outs[1]
    full = torch.empty_like(out)
    G.prefill_ws(q_rot, ck, cv, start, valid, full, G.alloc_prefill_workspace(B, Tmax, dev), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))
    ref = A.attention(W.bits(q_rot.cpu()), W.bits(ck.cpu()), W.bits(cv.cpu()), second.start_pos.numpy(),
                      second.valid_len.numpy())
    assert_close(W.bits(out.cpu()), ref, "second chunk, reused fp16 V")


def _append_then_prefill_ws(inp, ws_bytes, dev="cuda", calls=1):
    """Append, then grok_attn_prefill_ws `calls` times with a workspace of ws_bytes; output bits of each call."""
    import grok_gqa_attention_gb300 as G
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    start = inp.start_pos.to(dev)
    valid = None if inp.valid_len is None else inp.valid_len.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    q_rot = torch.empty_like(q)
    G.rope_kv_append(q, k, v, start, q_rot, ck, cv, status)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(calls):
        out = torch.empty_like(q_rot)
        G.prefill_ws(q_rot, ck, cv, start, valid, out, ws, status)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return [W.bits(o.cpu()) for o in outs], (W.bits(q_rot.cpu()), W.bits(ck.cpu()), W.bits(cv.cpu()))


def test_prefill_ws_key_split_matches_oracle():
    """Two 128-token chunks over long caches give 48 work items, fewer than the GPU's
    SMs, so grok_attn_prefill_ws runs them all in its split pass: sequence 1's items (25
    key tiles) are shared among three units each, whose partial outputs the item's last
    unit to finish adds; sequence 0's items (13 tiles, too few for two units of 8) run
    whole. The result must match the oracle, be the same bits on a second call
    (whichever unit finishes last), and differ from the unsplit call (a workspace of
    grok_attn_prefill_workspace_min bytes; other references, other fp16 roundings) while
    both stay within the tolerance."""
    import grok_gqa_attention_gb300 as G
    B, Tmax = 2, 4096
    inp = W.custom(B=B, T=128, Tmax=Tmax, start_pos=[1500, 3000], valid_len=[128, 77], seed=41)
    assert G.prefill_workspace(B, Tmax) > G.prefill_workspace_min(B, Tmax)
    (split, split2), (rq, rk, rv) = _append_then_prefill_ws(inp, G.prefill_workspace(B, Tmax), calls=2)
    (whole,), _ = _append_then_prefill_ws(inp, G.prefill_workspace_min(B, Tmax))
    assert np.array_equal(split, split2)
    assert not np.array_equal(split, whole)
    ref = A.attention(rq, rk, rv, inp.start_pos.numpy(), inp.valid_len.numpy())
    assert_close(split, ref, "key-range split")
    assert_close(whole, ref, "unsplit")


def test_prefill_ws_key_split_hands_overflowing_items_to_the_bf16_pass():
    """With the split active (24 items, each shared among three units over 25 key tiles),
    the first unit of every item sees a first tile of tiny logits and then saturated
    ones: its weights would overflow fp16, so every item goes to the bf16 pass, whose
    output equals grok_attn_prefill's bit for bit."""
    import grok_gqa_attention_gb300 as G
    Tmax = 4096
    inp = W.custom(B=1, T=128, Tmax=Tmax, start_pos=[3072], seed=42, scale=3.0)
    ck = inp.cache_k.float()
    ck[:, :128] *= 0.02
    ck[:, 128:3072] *= 4.0
    inp.cache_k.copy_(ck.to(torch.bfloat16))
    inp.k.copy_((inp.k.float() * 4.0).to(torch.bfloat16))
    (out16,), _ = _append_then_prefill_ws(inp, G.prefill_workspace(1, Tmax))
    _, _, _, outb, stb = run_prefill(inp, impl="bf16p")
    assert stb == 0
    assert np.array_equal(out16, outb)


def test_prefill_ws_key_split_skips_a_bad_sequence():
    """The split pass with one sequence whose start leaves the cache: its units are skipped
    (GROK_DEV_BAD_START, reported once), and the other sequence's split items still match
    the oracle."""
    import grok_gqa_attention_gb300 as G
    B, Tmax = 2, 4096
    good = W.custom(B=B, T=128, Tmax=Tmax, start_pos=[2000, 100], valid_len=[128, 128], seed=43)
    q_rot, ck, cv, st = run_append_dev(good)
    assert st == 0
    start = torch.tensor([2000, Tmax - 64], dtype=torch.int32, device="cuda")  # sequence 1: start + T > Tmax
    valid = good.valid_len.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q_rot)
    G.prefill_ws(q_rot, ck, cv, start, valid, out, G.alloc_prefill_workspace(B, Tmax, "cuda"), status)
    torch.cuda.synchronize()
    assert int(status.item()) == G.DEV_BAD_START
    rq, rk, rv = W.bits(q_rot.cpu()), W.bits(ck.cpu()), W.bits(cv.cpu())
    ref = A.attention(rq[:1], rk[:1], rv[:1], good.start_pos.numpy()[:1], good.valid_len.numpy()[:1])
    assert_close(W.bits(out[:1].cpu()), ref, "split pass beside a bad sequence")


def run_append_dev(inp, dev="cuda"):
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    ck, cv = inp.cache_k.to(dev), inp.cache_v.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    q_rot = torch.empty_like(q)
    import grok_gqa_attention_gb300 as G
    G.rope_kv_append(q, k, v, inp.start_pos.to(dev), q_rot, ck, cv, status)
    torch.cuda.synchronize()
    return q_rot, ck, cv, int(status.item())
