"""Pins of the oracle's attention: the pages' mask picture, GQA = MHA with repeated
KV heads, a library routine in the uncapped special case, closed forms of the
soft cap and softmax, brute force on tiny inputs, decode = prefill row."""
import math
import struct

import numpy as np
import torch

from oracle import attention as A
from oracle import bf16


def _rand_bf16(rng, shape, scale=3.0):
    return bf16.from_f32((rng.standard_normal(shape) * scale).astype(np.float32))


def test_constants_match_pages(golden):
    vals = {}
    for line in open(golden("constants.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, value = line.split()[:2]
        vals[name] = float(value)
    assert A.ATTN_OUTPUT_MULTIPLIER == vals["attn_output_multiplier"]
    assert abs(vals["attn_output_multiplier"] - 1 / math.sqrt(128)) <= 2 * np.spacing(0.088)
    assert A.MAX_ATTN_VAL == vals["max_attn_val"]
    assert A.MASK_FILL == vals["mask_fill"]
    # KV cache bytes per layer per sequence at 8192 tokens: 2 (k, v) * 8192 * 8 * 128 * 2 B
    assert 2 * 8192 * int(vals["num_kv_heads"]) * int(vals["key_size"]) * 2 == \
        vals["kv_cache_bytes_per_layer_per_sequence_8192"]


def test_causal_mask_matches_printed_6x6(golden):
    rows = [list(map(int, l.split())) for l in open(golden("causal_mask_6x6.txt"))
            if l.strip() and not l.startswith("#")]
    want = np.array(rows, dtype=bool)
    got = A.visible(0, 6, 6, np.arange(6), 6)
    assert np.array_equal(got, want)


def test_mask_brute_force_small():
    """Scalar enumeration of the three rules for every (start, valid, T) with T <= 6."""
    for T in range(1, 7):
        for start in range(0, 5):
            for valid in range(1, T + 1):
                L = start + T
                got = A.visible(start, valid, T, np.arange(T), L)
                for i in range(T):
                    for j in range(L):
                        in_memory = j < start + T
                        causal = j <= start + i
                        is_pad_key = j >= start and (j - start) >= valid
                        assert got[i, j] == (in_memory and causal and not is_pad_key)


def _tiny_case(rng, B=1, T=8, Tmax=8, start=None):
    q = _rand_bf16(rng, (B, T, 48, 128))
    ck = _rand_bf16(rng, (B, Tmax, 8, 128))
    cv = _rand_bf16(rng, (B, Tmax, 8, 128))
    start = np.zeros(B, dtype=np.int64) if start is None else np.asarray(start)
    return q, ck, cv, start


def test_gqa_equals_mha_with_repeated_kv_heads():
    """repeat_kv (ch. 4 §4.5.2): KV head g expanded to query heads 6g..6g+5."""
    rng = np.random.default_rng(10)
    q, ck, cv, start = _tiny_case(rng, B=2, T=8, Tmax=8)
    gqa = A.attention(q, ck, cv, start, None)
    ck48 = np.repeat(ck, 6, axis=2)      # [B, T, 8, 6, d] -> [B, T, 48, d] in order g*6+r
    cv48 = np.repeat(cv, 6, axis=2)
    mha = A.attention(q, ck48, cv48, start, None)
    assert np.array_equal(gqa, mha)
    # and a head mapping h -> h % 8 (the wrong one) would differ
    wrong_k = np.tile(ck, (1, 1, 6, 1))
    wrong_v = np.tile(cv, (1, 1, 6, 1))
    assert not np.array_equal(gqa, A.attention(q, wrong_k, wrong_v, start, None))


def test_uncapped_equals_torch_sdpa():
    """Without the cap, the method is scaled dot-product attention with a causal mask."""
    rng = np.random.default_rng(11)
    B, T = 2, 24
    q, ck, cv, start = _tiny_case(rng, B=B, T=T, Tmax=T)
    valid = np.array([T, 17])
    _, got = A.attention(q, ck, cv, start, valid, return_f64=True, cap=None)
    qt = torch.from_numpy(bf16.to_f64(q)).permute(0, 2, 1, 3)                # [B, 48, T, d]
    kt = torch.from_numpy(bf16.to_f64(ck)).repeat_interleave(6, dim=2).permute(0, 2, 1, 3)
    vt = torch.from_numpy(bf16.to_f64(cv)).repeat_interleave(6, dim=2).permute(0, 2, 1, 3)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    mask = torch.stack([(j <= i) & (j < int(n)) for n in valid])[:, None]   # [B, 1, T, T]
    want = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, scale=1 / math.sqrt(128)).permute(0, 2, 1, 3).numpy()
    assert np.abs(got - want).max() < 1e-10


def test_soft_cap_bounds_and_small_values():
    x = np.linspace(-1e4, 1e4, 100001)
    c = A.soft_cap(x)
    assert np.all(np.abs(c) <= 30.0)
    small = np.linspace(-1, 1, 1001)
    assert np.all(np.abs(A.soft_cap(small) - small) <= np.abs(small) ** 3 / (3 * 900) + 1e-15)


def _one_hot_values(L, d=128):
    """V rows e_j: the output of a query is then its weight vector."""
    v = np.zeros((L, d), dtype=np.float32)
    v[np.arange(L), np.arange(L)] = 1.0
    return bf16.from_f32(v)


def test_two_key_closed_form_with_cap():
    """Weights of two keys are 1/(1+exp(c2-c1)) with c = 30 tanh(s/sqrt(128)/30)."""
    d = 128
    q = np.zeros((1, 2, 48, d), dtype=np.float32)
    k = np.zeros((1, 2, 8, d), dtype=np.float32)
    # query row 1 (sees keys 0 and 1): q = a e_0, keys k0 = b0 e_0, k1 = b1 e_0
    q[0, 1, :, 0] = 16.0
    k[0, 0, :, 0] = 42.5
    k[0, 1, :, 0] = 21.25
    v = _one_hot_values(2)
    cv = np.broadcast_to(v[None, :, None, :], (1, 2, 8, d)).copy()
    out = bf16.to_f64(A.attention(bf16.from_f32(q), bf16.from_f32(k), cv, np.array([0])))
    s = np.array([16.0 * 42.5, 16.0 * 21.25]) / math.sqrt(128)
    c = 30 * np.tanh(s / 30)
    w0 = 1 / (1 + math.exp(c[1] - c[0]))
    assert abs(out[0, 1, 0, 0] - w0) <= 2 ** -9 * w0
    w1 = 1 / (1 + math.exp(c[0] - c[1]))
    assert abs(out[0, 1, 0, 1] - w1) <= 2 ** -8 * w1
    # the cap matters here: the capped weight is ~2e-3, uncapped it would be ~1e-13
    assert 1e-3 < w1 < 1e-2 and math.exp(s[1] - s[0]) < 1e-12
    assert out[0, 0, 0, 0] == 1.0 and out[0, 0, 0, 1] == 0.0      # row 0 sees key 0 only


def test_softmax_rows_sum_to_one_and_masked_weight_zero():
    rng = np.random.default_rng(12)
    T, start, valid = 16, 40, 11
    L = start + T
    q = _rand_bf16(rng, (1, T, 48, 128))
    ck = _rand_bf16(rng, (1, 128, 8, 128))
    cv = np.zeros((1, 128, 8, 128), dtype=np.uint16)
    cv[0, :L] = _one_hot_values(L)[:, None, :]
    cv[0, L:] = bf16.from_f32(np.full((128 - L, 8, 128), np.nan, dtype=np.float32))  # never read
    _, w = A.attention(q, ck, cv, np.array([start]), np.array([valid]), return_f64=True)
    assert np.all(np.isfinite(w))
    assert np.abs(w.sum(axis=-1) - 1).max() < 1e-12
    vis = A.visible(start, valid, T, np.arange(T), L)
    for i in range(T):
        assert np.all(w[0, i, :, :L][:, ~vis[i]] == 0.0)
        assert np.all(w[0, i, :, :L][:, vis[i]] > 0.0)
        assert np.all(w[0, i, :, L:] == 0.0)


def test_brute_force_scalar_loops_tiny():
    """Scalar-Python evaluation on B=1, T<=4, 2 query heads / 1 KV head, d=4."""
    rng = np.random.default_rng(13)
    T, d = 4, 4
    q = _rand_bf16(rng, (1, T, 2, d), 1.0)
    ck = _rand_bf16(rng, (1, T, 1, d), 1.0)
    cv = _rand_bf16(rng, (1, T, 1, d), 1.0)
    _, got = A.attention(q, ck, cv, np.array([0]), np.array([3]), return_f64=True)
    qf, kf, vf = (bf16.to_f64(x) for x in (q, ck, cv))
    for i in range(T):
        for h in range(2):
            logits = []
            for j in range(T):
                if j <= i and j < 3:
                    s = sum(qf[0, i, h, t] * kf[0, j, 0, t] for t in range(d))
                    s = s * 0.08838834764831845
                    logits.append((j, 30.0 * math.tanh(s / 30.0)))
            m = max(c for _, c in logits)
            z = sum(math.exp(c - m) for _, c in logits)
            for t in range(d):
                o = sum(math.exp(c - m) / z * vf[0, j, 0, t] for j, c in logits)
                assert abs(got[0, i, h, t] - o) < 1e-12


def test_decode_equals_prefill_row():
    """A decode step at position t reproduces row t of the prefill (ch. 6 §6.4.2)."""
    rng = np.random.default_rng(14)
    T = 12
    q, ck, cv, start = _tiny_case(rng, B=1, T=T, Tmax=T)
    _, full = A.attention(q, ck, cv, start, None, return_f64=True)
    for t in range(T):
        _, dec = A.decode(q[:, t], ck, cv, np.array([t + 1]), return_f64=True)
        assert np.abs(dec[0] - full[0, t]).max() < 1e-12


def test_rows_api_matches_full():
    rng = np.random.default_rng(15)
    B, T, Tmax = 2, 10, 20
    q, ck, cv, _ = _tiny_case(rng, B=B, T=T, Tmax=Tmax)
    start = np.array([3, 10])
    valid = np.array([10, 6])
    full = A.attention(q, ck, cv, start, valid)
    rows = [(0, 0, 0), (0, 9, 47), (1, 5, 13), (1, 7, 30), (1, 9, 5)]
    bits, _ = A.attention_rows(q, ck, cv, start, valid, T, rows)
    for n, (b, i, h) in enumerate(rows):
        assert np.array_equal(bits[n], full[b, i, h])


def test_chain_mode_sits_near_exact():
    """The pages' own dtype chain (bf16 weights) differs from exact by bf16-level amounts."""
    rng = np.random.default_rng(16)
    q, ck, cv, start = _tiny_case(rng, B=1, T=64, Tmax=64)
    ex = bf16.to_f64(A.attention(q, ck, cv, start, None))
    ch = bf16.to_f64(A.attention(q, ck, cv, start, None, mode="chain"))
    d = np.abs(ex - ch)
    assert d.max() <= 0.0625 + 1e-12
    assert 1e-4 < d.mean() < 5e-3


def test_chain_mode_closed_forms():
    """The pages' dtype chain (ch. 4 §4.5.3: fp32 logits and softmax, weights cast
    to bf16 before the weighted sum) on inputs whose result is known in closed form.

    (a) Three keys with equal logits: each weight is RN32(1/3), which bf16 rounds
    to 0.333984375, so with every value row equal to c the chain returns
    3 * 0.333984375 * c (the exact method returns c).
    (b) Two keys whose raw dot products are 256 and 257: fp32 keeps them apart,
    bf16 would not (257 is a bf16 tie that rounds to 256). The weight of the
    second key is 1 / (1 + exp(c0 - c1)) = 0.5131 with c = 30 tanh(s / sqrt(128) / 30),
    which the chain returns to within one bf16 step (2^-8 on [0.5, 1)); bf16 logits
    would give exactly 0.5.
    """
    d = 16
    q = np.zeros((1, 3, 2, d), np.float32)
    k = np.zeros((1, 3, 1, d), np.float32)
    v = np.zeros((1, 3, 1, d), np.float32)
    q[0, :, :, 0] = 1.0
    k[0, :, 0, 0] = 2.0
    v[0, :, 0, :] = 1.5
    qb, kb, vb = (bf16.from_f32(x) for x in (q, k, v))
    _, o = A.attention(qb, kb, vb, np.array([0]), None, mode="chain", return_f64=True)
    assert np.all(o[0, 2] == 3 * 0.333984375 * 1.5)
    _, o = A.attention(qb, kb, vb, np.array([0]), None, mode="exact", return_f64=True)
    assert np.all(o[0, 2] == 1.5)

    q = np.zeros((1, 2, 2, d), np.float32)
    k = np.zeros((1, 2, 1, d), np.float32)
    v = np.zeros((1, 2, 1, d), np.float32)
    q[0, :, :, 0], q[0, :, :, 1] = 16.0, 1.0
    k[0, 0, 0, 0], k[0, 1, 0, 0], k[0, 1, 0, 1] = 16.0, 16.0, 1.0
    v[0, 1, 0, 0] = 1.0   # feature 0 returns the weight of key 1
    v[0, 0, 0, 1] = 1.0   # feature 1 returns the weight of key 0
    qb, kb, vb = (bf16.from_f32(x) for x in (q, k, v))
    _, o = A.attention(qb, kb, vb, np.array([0]), None, mode="chain", return_f64=True)
    c = 30 * np.tanh(np.array([256.0, 257.0]) / math.sqrt(128) / 30)
    w1 = 1 / (1 + math.exp(c[0] - c[1]))
    assert abs(o[0, 1, 0, 0] - w1) <= 2 ** -8 and abs(o[0, 1, 0, 1] - (1 - w1)) <= 2 ** -9
    assert abs(o[0, 1, 0, 0] - 0.5) > 2 ** -8


def _rn32(x: float) -> float:
    """Round a Python float to the nearest binary32 (ties to even) through struct."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def _rn_bf16(x: float) -> float:
    """Round a binary32 value to bfloat16 (nearest, ties to even) from its bits."""
    u = struct.unpack("<I", struct.pack("<f", x))[0]
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return struct.unpack("<f", struct.pack("<I", (u & 0xFFFF) << 16))[0]


def test_chain_mode_scalar_brute_force():
    """Scalar evaluation of the pages' chain, each step rounded to fp32 on its own
    (ch. 4 §4.5.2-§4.5.4): logits = fp32(q . k); fp32 multiply by fp32(1/sqrt(128));
    fp32 division by 30, fp32 tanh, fp32 multiply by 30; masked logits -1e30;
    fp32 max, fp32 exp of the fp32 difference, fp32 row sum left to right, fp32
    division; weights to bf16; weighted sum of V. No numpy arithmetic is used for
    the chain itself: fp32 rounding goes through struct, tanh and exp are the fp64
    library functions rounded to fp32."""
    rng = np.random.default_rng(18)
    T, d, start, valid = 6, 8, 0, 5
    q = _rand_bf16(rng, (1, T, 2, d), 2.0)
    ck = _rand_bf16(rng, (1, T, 1, d), 2.0)
    cv = _rand_bf16(rng, (1, T, 1, d), 1.0)
    _, got = A.attention(q, ck, cv, np.array([start]), np.array([valid]), mode="chain", return_f64=True)
    qf, kf, vf = (bf16.to_f64(x) for x in (q, ck, cv))
    mult = _rn32(0.08838834764831845)
    for i in range(T):
        for h in range(2):
            logits = []
            for j in range(start + T):
                s = _rn32(sum(qf[0, i, h, t] * kf[0, j, 0, t] for t in range(d)))
                s = _rn32(s * mult)
                s = _rn32(30.0 * _rn32(math.tanh(_rn32(s / 30.0))))
                visible = j <= start + i and j < start + valid
                logits.append(s if visible else _rn32(-1e30))
            m = max(logits)
            e = [_rn32(math.exp(_rn32(x - m))) for x in logits]
            z = 0.0
            for x in e:
                z = _rn32(z + x)
            w = [_rn_bf16(_rn32(x / z)) for x in e]
            for t in range(d):
                o = sum(w[j] * vf[0, j, 0, t] for j in range(start + T))
                assert abs(got[0, i, h, t] - o) < 1e-12, (i, h, t)


def test_full_attention_covers_rows_across_its_row_blocks():
    """attention() evaluates rows in blocks of ROW_BLOCK; at T > ROW_BLOCK every row,
    including those either side of a block edge, equals the one-row evaluation."""
    rng = np.random.default_rng(17)
    T = A.ROW_BLOCK + 44
    q, ck, cv, start = _tiny_case(rng, B=1, T=T, Tmax=T)
    full = A.attention(q, ck, cv, start, None)
    edge = [0, A.ROW_BLOCK - 2, A.ROW_BLOCK - 1, A.ROW_BLOCK, T - 1]
    rows = [(0, i, h) for i in edge for h in (0, 23, 47)]
    bits, _ = A.attention_rows(q, ck, cv, start, np.array([T]), T, rows)
    for n, (b, i, h) in enumerate(rows):
        assert np.array_equal(bits[n], full[b, i, h]), (i, h)


def test_block_api_matches_full():
    """attention_block (whole query tiles, every head) equals the full evaluation,
    on a block that straddles the full evaluation's row blocks, for a chunk on a
    warm cache with key padding."""
    rng = np.random.default_rng(19)
    B, T, Tmax = 2, A.ROW_BLOCK + 40, A.ROW_BLOCK + 100
    q, ck, cv, _ = _tiny_case(rng, B=B, T=T, Tmax=Tmax)
    start = np.array([0, 60])
    valid = np.array([T, T - 50])
    full = A.attention(q, ck, cv, start, valid)
    for b, i0, i1 in ((0, 0, 8), (1, A.ROW_BLOCK - 5, A.ROW_BLOCK + 7), (1, T - 3, T)):
        got = A.attention_block(q, ck, cv, start, valid, T, b, i0, i1)
        assert np.array_equal(got, full[b, i0:i1]), (b, i0, i1)
