"""Q/K/V projection parity: the tensor-core GEMM against the fp64 oracle, and the
fused projection + RoPE + cache append against the oracle's RoPE applied to the
kernel's own projection (bit for bit)."""
import numpy as np
import pytest
import torch

import grok_gqa_attention_gb300 as G
import workloads as W
from oracle import bf16, projection as P, rope

pytestmark = pytest.mark.gpu


def acc_bound(K: int) -> float:
    """The tensor cores accumulate a K-term dot in fp32: K/16 additions of a
    16-term chunk into the accumulator, each rounding to half an fp32 ulp of a
    partial sum. With the generated magnitudes partial sums stay below 16, so
    the accumulated error is at most (K/16) * 2^-20 (K = 6144: 3.7e-4)."""
    return (K // 16) * 2.0 ** -20


ACC_BOUND = acc_bound(6144)


def _half_ulp(v):
    return np.spacing(np.abs(v).astype(np.float32)).astype(np.float64) * 2 ** 15


def _projection_check(got_bits, exact, what, max_mismatch_frac=0.01, K=6144):
    """Within half a bf16 ulp of the exact sum plus the fp32 accumulation bound;
    equal to the oracle's rounded bits for all but a small fraction."""
    g = bf16.to_f64(got_bits)
    assert np.all(np.isfinite(g))
    half_ulp = np.maximum(_half_ulp(exact), _half_ulp(g))
    err = np.abs(g - exact)
    assert np.all(err <= half_ulp + acc_bound(K)), f"{what}: worst excess {float((err - half_ulp).max())}"
    frac = float(np.mean(got_bits != bf16.from_f64(exact)))
    assert frac <= max_mismatch_frac, f"{what}: {frac:.4%} of outputs differ from the rounded exact sum"
    return frac


@pytest.fixture(scope="module")
def small():
    return W.projection(B=2, T=200, Tmax=512, start_pos=[100, 37], seed=50)


def test_projection_matches_exact_oracle(small):
    x2d = small.x.reshape(-1, P.MODEL_SIZE)
    w = small.w.cuda()
    y = torch.empty((x2d.shape[0], P.QKV_COLUMNS), dtype=torch.bfloat16, device="cuda")
    G.qkv_project(x2d.cuda(), w, y)
    torch.cuda.synchronize()
    got = W.bits(y.cpu())
    _projection_check(got, P.linear_exact(W.bits(x2d), W.bits(small.w)), "projection M=400")


def test_fused_equals_rope_append_of_own_projection(small):
    B, T = small.x.shape[0], small.x.shape[1]
    Tmax = small.cache_k.shape[1]
    x, w = small.x.cuda(), small.w.cuda()
    y = torch.empty((B * T, P.QKV_COLUMNS), dtype=torch.bfloat16, device="cuda")
    G.qkv_project(x.reshape(B * T, -1), w, y)
    ck, cv = small.cache_k.cuda(), small.cache_v.cuda()
    q_rot = torch.empty((B, T, 48, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = G.alloc_qkv_workspace(B, T)
    G.qkv_rope_append(x, w, small.start_pos.cuda(), q_rot, ck, cv, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yb = W.bits(y.cpu()).reshape(B, T, -1)
    q = yb[..., :6144].reshape(B, T, 48, 128)
    k = yb[..., 6144:7168].reshape(B, T, 8, 128)
    v = yb[..., 7168:].reshape(B, T, 8, 128)
    rq, rk, rv = rope.rope_kv_append(q, k, v, small.start_pos.numpy(), W.bits(small.cache_k), W.bits(small.cache_v))
    assert np.array_equal(W.bits(q_rot.cpu()), rq)
    assert np.array_equal(W.bits(ck.cpu()), rk)   # includes rows outside [start, start+T): untouched
    assert np.array_equal(W.bits(cv.cpu()), rv)


def test_fused_from_position_table_equals_fused(small):
    """The fused projection reading a table of every position (no per-call table kernel)
    writes the same bits as the per-call-table version; a sequence beyond the table is
    reported and left unwritten."""
    B, T = small.x.shape[0], small.x.shape[1]
    Tmax = small.cache_k.shape[1]
    x, w = small.x.cuda(), small.w.cuda()
    start = small.start_pos.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ck1, cv1 = small.cache_k.cuda(), small.cache_v.cuda()
    q1 = torch.empty((B, T, 48, 128), dtype=torch.bfloat16, device="cuda")
    G.qkv_rope_append(x, w, start, q1, ck1, cv1, G.alloc_qkv_workspace(B, T), status)
    ck2, cv2 = small.cache_k.cuda(), small.cache_v.cuda()
    q2 = torch.empty_like(q1)
    ctab, stab = G.rope_cos_sin(0, Tmax)
    G.qkv_rope_append_table(x, w, start, ctab, stab, q2, ck2, cv2, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
    assert torch.equal(ck1.view(torch.int16), ck2.view(torch.int16))
    assert torch.equal(cv1.view(torch.int16), cv2.view(torch.int16))
    # a table covering positions [0, 250): sequence 0 (start 100, T 200) needs up to 299
    ck3, cv3 = small.cache_k.cuda(), small.cache_v.cuda()
    ctab3, stab3 = G.rope_cos_sin(0, 250)
    G.qkv_rope_append_table(x, w, start, ctab3, stab3, torch.empty_like(q1), ck3, cv3, status)
    torch.cuda.synchronize()
    assert int(status.item()) & G.DEV_BAD_START
    assert np.array_equal(W.bits(ck3.cpu())[0], W.bits(small.cache_k)[0])   # sequence 0 untouched
    assert torch.equal(ck3[1].view(torch.int16), ck2[1].view(torch.int16))   # sequence 1 (start 37) written


def test_table_bad_start_in_the_second_half_of_a_row_tile():
    """The epilogue reports a start beyond the position table from the row of
    position 0 of the sequence; with T = 128 sequence 1's first row is the
    second 128-row half of the first 256-row tile."""
    B, T, Tmax = 2, 128, 512
    inp = W.projection(B=B, T=T, Tmax=Tmax, start_pos=[0, 300], seed=54)
    x, w, start = inp.x.cuda(), inp.w.cuda(), inp.start_pos.cuda()
    ctab, stab = G.rope_cos_sin(0, 400)   # sequence 1 needs positions up to 427
    ck, cv = inp.cache_k.cuda(), inp.cache_v.cuda()
    q_rot = torch.zeros((B, T, 48, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.qkv_rope_append_table(x, w, start, ctab, stab, q_rot, ck, cv, status)
    torch.cuda.synchronize()
    assert int(status.item()) == G.DEV_BAD_START
    assert np.array_equal(W.bits(ck.cpu())[1], W.bits(inp.cache_k)[1])
    assert np.array_equal(W.bits(cv.cpu())[1], W.bits(inp.cache_v)[1])
    assert not W.bits(q_rot.cpu())[1].any()
    # sequence 0 as the per-call-table version writes it
    ck1, cv1 = inp.cache_k.cuda(), inp.cache_v.cuda()
    q1 = torch.zeros_like(q_rot)
    st1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.qkv_rope_append(x[:1], w, start[:1], q1[:1], ck1[:1], cv1[:1], G.alloc_qkv_workspace(1, T), st1)
    torch.cuda.synchronize()
    assert int(st1.item()) == 0
    assert torch.equal(q_rot[0].view(torch.int16), q1[0].view(torch.int16))
    assert torch.equal(ck[0].view(torch.int16), ck1[0].view(torch.int16))


def test_fused_full_size_sampled_rows():
    B, T, Tmax = 1, 8192, 8192
    inp = W.projection(B=B, T=T, Tmax=Tmax, start_pos=[0], seed=51)
    x, w = inp.x.cuda(), inp.w.cuda()
    y = torch.empty((B * T, P.QKV_COLUMNS), dtype=torch.bfloat16, device="cuda")
    G.qkv_project(x.reshape(B * T, -1), w, y)
    ck, cv = inp.cache_k.cuda(), inp.cache_v.cuda()
    q_rot = torch.empty((B, T, 48, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.qkv_rope_append(x, w, inp.start_pos.cuda(), q_rot, ck, cv, G.alloc_qkv_workspace(B, T), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(52)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 8191], rng.integers(0, T, 58)]))
    yb = W.bits(y.cpu())[rows]
    # the projection against the exact oracle on the sampled rows
    _projection_check(yb, P.linear_exact(W.bits(inp.x)[0, rows], W.bits(inp.w)), "projection M=8192 (sampled rows)")
    # the fused outputs against the oracle's RoPE of the kernel's projection, row by row
    qb, kb = W.bits(q_rot.cpu())[0], W.bits(ck.cpu())[0]
    vb = W.bits(cv.cpu())[0]
    for n, i in enumerate(rows):
        q = yb[n, :6144].reshape(1, 1, 48, 128)
        k = yb[n, 6144:7168].reshape(1, 1, 8, 128)
        assert np.array_equal(qb[i], rope.rotary_embedding(q, np.array([i]))[0, 0])
        assert np.array_equal(kb[i], rope.rotary_embedding(k, np.array([i]))[0, 0])
        assert np.array_equal(vb[i], yb[n, 7168:].reshape(8, 128))


def test_bad_start_sets_status_and_writes_nothing_for_that_sequence():
    B, T, Tmax = 2, 64, 128
    inp = W.projection(B=B, T=T, Tmax=Tmax, start_pos=[10, Tmax - T + 1], seed=53)
    ck, cv = inp.cache_k.cuda(), inp.cache_v.cuda()
    q_rot = torch.zeros((B, T, 48, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.qkv_rope_append(inp.x.cuda(), inp.w.cuda(), inp.start_pos.cuda(), q_rot, ck, cv,
                      G.alloc_qkv_workspace(B, T), status)
    torch.cuda.synchronize()
    assert int(status.item()) & G.DEV_BAD_START
    assert np.array_equal(W.bits(ck.cpu())[1], W.bits(inp.cache_k)[1])
    assert np.array_equal(W.bits(cv.cpu())[1], W.bits(inp.cache_v)[1])
    assert not W.bits(q_rot.cpu())[1].any()
    assert W.bits(q_rot.cpu())[0].any()             # the valid sequence was written


def test_argument_checks():
    B, T = 1, 8
    x = torch.zeros((B, T, P.MODEL_SIZE), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((P.MODEL_SIZE, P.QKV_COLUMNS), dtype=torch.bfloat16, device="cuda")
    ck = torch.zeros((B, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    q_rot = torch.empty((B, T, 48, 128), dtype=torch.bfloat16, device="cuda")
    start = torch.zeros(B, dtype=torch.int32, device="cuda")
    small_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(G.GrokError):
        G.qkv_rope_append(x, w, start, q_rot, ck, cv, small_ws)
    assert G.load().grok_qkv_project(None, None, 4, None, None, None) == 1
    assert G.qkv_workspace(B, T) == B * T * 64 * 2 * 4


def _rand(gen, shape, scale):
    return (torch.randn(*shape, generator=gen) * scale).to(torch.bfloat16)


# 192-column tiles: N = 576 and 192 are only multiples of 192; N = 6144 at M = 64
# and 600 picks them too (more of the last round of tiles busy)
@pytest.mark.parametrize("M,K,N", [(1, 64, 256), (130, 128, 512), (257, 6144, 256), (64, 768, 6144),
                                   (600, 192, 6144), (300, 192, 576), (1, 64, 192)])
def test_linear_shapes_match_oracle(M, K, N):
    gen = torch.Generator().manual_seed(M * 7 + K + N)
    x = _rand(gen, (M, K), 1.0)
    w = _rand(gen, (K, N), 3.0 / np.sqrt(K))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    G.linear(x.cuda(), w.cuda(), y)
    torch.cuda.synchronize()
    _projection_check(W.bits(y.cpu()), P.linear_exact(W.bits(x), W.bits(w)), f"linear {M}x{K}x{N}", K=K)


@pytest.fixture(scope="module")
def attn_out():
    gen = torch.Generator().manual_seed(60)
    attn = _rand(gen, (2, 200, 48, 128), 3.0)                 # an attention output [B, T, 48, 128]
    w_o = _rand(gen, (6144, 6144), 1.0 / np.sqrt(6144))
    return attn, w_o


def test_output_projection_matches_oracle(attn_out):
    attn, w_o = attn_out
    y = torch.empty((400, 6144), dtype=torch.bfloat16, device="cuda")
    G.linear(attn.reshape(400, 6144).cuda(), w_o.cuda(), y)
    torch.cuda.synchronize()
    exact = P.linear_exact(W.bits(attn).reshape(400, 6144), W.bits(w_o))
    _projection_check(W.bits(y.cpu()), exact, "output projection M=400")


def test_head_sharded_output_projection_partials_sum_to_the_whole(attn_out):
    """Eight ranks, each holding 6 heads (768 features) and their 768 rows of W_o."""
    attn, w_o = attn_out
    ranks, width = 8, 768
    a = attn.reshape(400, 6144)
    total = np.zeros((400, 6144))
    bound = np.zeros((400, 6144))
    for r in range(ranks):
        xr = a[:, r * width:(r + 1) * width].contiguous().cuda()
        wr = w_o[r * width:(r + 1) * width].contiguous().cuda()
        yr = torch.empty((400, 6144), dtype=torch.bfloat16, device="cuda")
        G.linear(xr, wr, yr)
        torch.cuda.synchronize()
        got = W.bits(yr.cpu())
        exact_r = P.output_projection_partial(W.bits(attn), W.bits(w_o), r, ranks).reshape(400, 6144)
        _projection_check(got, exact_r, f"rank {r} partial", K=width)
        g = bf16.to_f64(got)
        total += g
        bound += _half_ulp(g) + acc_bound(width)
    whole = P.linear_exact(W.bits(a), W.bits(w_o))
    assert np.all(np.abs(total - whole) <= bound + 1e-12)


def _int8_weight(gen, K, N):
    w8 = torch.randint(-127, 128, (K, N), generator=gen, dtype=torch.int32).to(torch.int8)
    scales = (torch.rand(N, generator=gen) + 0.5) * (3.0 / np.sqrt(K) / 73.0)   # |w8| has std ~73
    return w8, scales.to(torch.float32)


@pytest.mark.parametrize("K,N", [(96, 48), (6144, 8192)])
def test_dequant_int8_bit_exact(K, N):
    gen = torch.Generator().manual_seed(K + N)
    w8, scales = _int8_weight(gen, K, N)
    w16 = torch.empty((K, N), dtype=torch.bfloat16, device="cuda")
    G.dequant_int8(w8.cuda(), scales.cuda(), w16)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(w16.cpu()), P.dequant_int8(w8.numpy(), scales.numpy()))


@pytest.mark.parametrize("M,K,N", [(130, 768, 512), (32, 512, 576)])
def test_linear_int8_matches_oracle(M, K, N):
    """Dequantize-then-multiply; N = 576 (a multiple of 192, not of 256) takes it at M = 32 too,
    on 192-column tiles."""
    gen = torch.Generator().manual_seed(70 + N)
    x = _rand(gen, (M, K), 1.0)
    w8, scales = _int8_weight(gen, K, N)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(G.linear_int8_workspace(K, N), dtype=torch.uint8, device="cuda")
    G.linear_int8(x.cuda(), w8.cuda(), scales.cuda(), y, ws)
    torch.cuda.synchronize()
    w16 = P.dequant_int8(w8.numpy(), scales.numpy())
    _projection_check(W.bits(y.cpu()), P.linear_exact(W.bits(x), w16), "int8 linear", K=K)
    with pytest.raises(G.GrokError):   # workspace too small
        G.linear_int8(x.cuda(), w8.cuda(), scales.cuda(), y, ws[:16])


def test_outputs_written_with_32_byte_stores_must_be_32_byte_aligned():
    """A 16-byte aligned but not 32-byte aligned output is rejected on the host (nothing is launched)."""
    x = torch.zeros((256, 6144), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((6144, 8192), dtype=torch.bfloat16, device="cuda")
    buf = torch.zeros(256 * 8192 + 16, dtype=torch.bfloat16, device="cuda")
    y_off = buf[8:8 + 256 * 8192].view(256, 8192)          # base + 16 bytes
    assert y_off.data_ptr() % 32 == 16
    with pytest.raises(G.GrokError):
        G.qkv_project(x, w, y_off)
    w8 = torch.zeros((64, 256), dtype=torch.int8, device="cuda")
    sc = torch.ones(256, dtype=torch.float32, device="cuda")
    wbuf = torch.zeros(64 * 256 + 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G.GrokError):
        G.dequant_int8(w8, sc, wbuf[8:8 + 64 * 256].view(64, 256))
    G.dequant_int8(w8, sc, wbuf[16:16 + 64 * 256].view(64, 256))   # 32-byte aligned offset: accepted
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [1, 7, 16, 17, 32])
def test_linear_int8_small_m_matches_oracle(M):
    """Decode-sized M takes the one-pass path (weight dequantized in shared memory)."""
    gen = torch.Generator().manual_seed(90 + M)
    K, N = 1024, 512
    x = _rand(gen, (M, K), 1.0)
    w8, scales = _int8_weight(gen, K, N)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(G.linear_int8_workspace(K, N), dtype=torch.uint8, device="cuda")
    G.linear_int8(x.cuda(), w8.cuda(), scales.cuda(), y, ws)
    torch.cuda.synchronize()
    w16 = P.dequant_int8(w8.numpy(), scales.numpy())
    _projection_check(W.bits(y.cpu()), P.linear_exact(W.bits(x), w16), f"int8 linear M={M}", K=K)
    y2 = torch.empty_like(y)
    G.linear_int8(x.cuda(), w8.cuda(), scales.cuda(), y2, ws)   # deterministic: same bits again
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_linear_int8_small_m_full_size():
    gen = torch.Generator().manual_seed(99)
    M, K, N = 32, 6144, 8192
    x = _rand(gen, (M, K), 1.0)
    w8, scales = _int8_weight(gen, K, N)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(G.linear_int8_workspace(K, N), dtype=torch.uint8, device="cuda")
    G.linear_int8(x.cuda(), w8.cuda(), scales.cuda(), y, ws)
    torch.cuda.synchronize()
    w16 = P.dequant_int8(w8.numpy(), scales.numpy())
    _projection_check(W.bits(y.cpu()), P.linear_exact(W.bits(x), w16), "int8 linear M=32 full size", K=K)
