"""Pins of the oracle's Q/K/V projection: exact rational brute force, identity and
one-hot weights (column layout), exact scaling, a library matmul, and the fused
step's position-0 special case."""
from fractions import Fraction

import numpy as np
import torch

from oracle import bf16, projection as P, rope
from tests.exact_util import nearest_bf16, nearest_f32


ONE = np.uint16(0x3F80)  # bf16 1.0


def _rand_bf16(rng, shape, scale=1.0):
    return bf16.from_f32((rng.standard_normal(shape) * scale).astype(np.float32))


def test_linear_equals_exact_rational_brute_force():
    rng = np.random.default_rng(20)
    x = _rand_bf16(rng, (2, 3, 5))
    w = _rand_bf16(rng, (5, 4))
    got = bf16.to_f64(P.linear(x, w))
    xf, wf = bf16.to_f64(x), bf16.to_f64(w)
    for a in range(2):
        for t in range(3):
            for n in range(4):
                exact = sum(Fraction(float(xf[a, t, i])) * Fraction(float(wf[i, n])) for i in range(5))
                assert got[a, t, n] == nearest_bf16(exact)


def test_identity_weights_return_x():
    rng = np.random.default_rng(21)
    x = _rand_bf16(rng, (1, 3, 256), 3.0)
    w = np.zeros((256, 256), dtype=np.uint16)
    w[np.arange(256), np.arange(256)] = ONE
    assert np.array_equal(P.linear(x, w), x)


def test_one_hot_columns_land_in_the_right_head_and_feature():
    rng = np.random.default_rng(22)
    K = 64  # the projection is generic in the input width; the head split is in the 8192 columns
    x = _rand_bf16(rng, (1, 2, K))
    cases = [(0, "q", 0, 0), (6143, "q", 47, 127), (130, "q", 1, 2), (6144, "k", 0, 0), (6144 + 3 * 128 + 5, "k", 3, 5),
             (7168, "v", 0, 0), (8191, "v", 7, 127)]
    for col, which, head, d in cases:
        w = np.zeros((K, P.QKV_COLUMNS), dtype=np.uint16)
        w[7, col] = ONE
        out = dict(zip("qkv", P.qkv_projection(x, w)))
        t = out[which]
        assert np.array_equal(t[:, :, head, d], x[:, :, 7])
        mask = np.ones(t.shape, dtype=bool)
        mask[:, :, head, d] = False
        assert not t[mask].any()
        assert all(not out[o].any() for o in "qkv" if o != which)


def test_scaling_by_a_power_of_two_is_exact():
    rng = np.random.default_rng(23)
    x = _rand_bf16(rng, (1, 4, 64))
    w = _rand_bf16(rng, (64, 32))
    x2 = bf16.from_f64(bf16.to_f64(x) * 4.0)
    assert np.array_equal(bf16.to_f64(P.linear(x2, w)), bf16.to_f64(P.linear(x, w)) * 4.0)


def test_linear_matches_torch_matmul_in_fp64():
    rng = np.random.default_rng(24)
    x = _rand_bf16(rng, (3, 7, 96))
    w = _rand_bf16(rng, (96, 40))
    ref = torch.from_numpy(bf16.to_f64(x)) @ torch.from_numpy(bf16.to_f64(w))
    assert np.array_equal(P.linear(x, w), bf16.from_f64(ref.numpy()))


def test_fused_step_at_position_zero_keeps_the_projection():
    rng = np.random.default_rng(25)
    K = 64
    x = _rand_bf16(rng, (1, 1, K))
    w = _rand_bf16(rng, (K, P.QKV_COLUMNS), 3.0 / np.sqrt(K))
    ck = _rand_bf16(rng, (1, 4, 8, 128))
    cv = _rand_bf16(rng, (1, 4, 8, 128))
    q, k, v = P.qkv_projection(x, w)
    q_rot, nk, nv = P.qkv_rope_append(x, w, np.array([0]), ck, cv)
    assert np.array_equal(q_rot, q)            # cos 0 = 1, sin 0 = 0
    assert np.array_equal(nk[0, 0], k[0, 0]) and np.array_equal(nv[0, 0], v[0, 0])
    assert np.array_equal(nk[0, 1:], ck[0, 1:])
    # at another position the rotation is the RoPE oracle's
    q_rot3, nk3, _ = P.qkv_rope_append(x, w, np.array([3]), ck, cv)
    assert np.array_equal(q_rot3, rope.rotary_embedding(q, np.array([3])))


def test_output_projection_reads_heads_in_order():
    """Input column h*128 + d of W_o multiplies head h, feature d of the attention output."""
    rng = np.random.default_rng(26)
    attn = _rand_bf16(rng, (1, 2, P.N_Q_HEADS, P.HEAD_DIM))
    for h, d in [(0, 0), (5, 77), (47, 127)]:
        w = np.zeros((P.N_Q_HEADS * P.HEAD_DIM, 256), dtype=np.uint16)
        w[h * 128 + d, 3] = ONE
        y = P.output_projection(attn, w)
        assert np.array_equal(y[:, :, 3], attn[:, :, h, d])
        assert not np.delete(y, 3, axis=-1).any()


def test_output_projection_shards_sum_to_the_whole():
    rng = np.random.default_rng(27)
    attn = _rand_bf16(rng, (1, 3, P.N_Q_HEADS, P.HEAD_DIM))
    w = _rand_bf16(rng, (P.N_Q_HEADS * P.HEAD_DIM, 256), 3.0 / np.sqrt(6144))
    whole = P.linear_exact(attn.reshape(1, 3, -1), w)
    for ranks in (2, 8):
        parts = sum(P.output_projection_partial(attn, w, r, ranks) for r in range(ranks))
        assert np.abs(parts - whole).max() < 1e-12


def test_dequant_int8_matches_exact_products_rounded_twice():
    """int8 (8 bits) x fp32 (24 bits) fits fp64 exactly, so float(w) * float(s) is the exact
    product; np.float32 of it is the fp32 rounding and the brute-force search the bf16 one."""
    rng = np.random.default_rng(28)
    w8 = rng.integers(-128, 128, size=(6, 5)).astype(np.int8)
    scales = (rng.random(5) * 1e-3 + 1e-4).astype(np.float32)
    got = bf16.to_f64(P.dequant_int8(w8, scales))
    for i in range(6):
        for n in range(5):
            exact = float(w8[i, n]) * float(scales[n])          # exact in fp64
            r32 = float(np.float32(exact))
            assert got[i, n] == nearest_bf16(Fraction(r32))


def test_dequant_int8_unit_and_power_of_two_scales_are_exact():
    w8 = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(16, 16)
    for s in (1.0, 0.25, 2.0 ** -10):
        got = bf16.to_f64(P.dequant_int8(w8, np.full(16, s, dtype=np.float32)))
        assert np.array_equal(got, w8.astype(np.float64) * s)


def test_linear_int8_is_linear_on_the_dequantized_weight():
    rng = np.random.default_rng(29)
    x = _rand_bf16(rng, (1, 3, 64))
    w8 = rng.integers(-127, 128, size=(64, 256)).astype(np.int8)
    scales = (rng.random(256) * 0.01).astype(np.float32)
    assert np.array_equal(P.linear_int8(x, w8, scales), P.linear(x, P.dequant_int8(w8, scales)))
    # a per-channel scale only scales its own output column (power-of-two ratio: exact)
    s2 = scales.copy()
    s2[7] *= 4.0
    a, b = bf16.to_f64(P.linear_int8(x, w8, scales)), bf16.to_f64(P.linear_int8(x, w8, s2))
    assert np.array_equal(b[..., 7], 4.0 * a[..., 7])
    assert np.array_equal(np.delete(a, 7, axis=-1), np.delete(b, 7, axis=-1))


def test_dequant_int8_two_roundings_at_decisive_elements():
    """Where rounding w * s straight to bf16 would give another value than rounding it to
    fp32 first (ch. 4 §4.1: ``astype(scales.dtype) * scales``, then the cast to bf16), the
    oracle takes the two roundings. Such elements are built directly: for a bf16 midpoint
    tau and an int8 w that is not a power of two, an fp32 scale next to tau / w makes the
    exact product lie just off tau while its fp32 rounding is tau itself."""
    rng = np.random.default_rng(30)
    ties = ((rng.integers(0x3880, 0x3F80, size=256).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    odd = [v for v in range(-127, 128) if v and abs(v) & (abs(v) - 1)]
    ws, ss = [], []
    for tau, w in zip(ties, rng.choice(odd, size=len(ties))):
        s0 = np.float32(float(tau) / int(w))
        for k in range(-3, 4):
            sc = s0
            for _ in range(abs(k)):
                sc = np.nextafter(sc, np.float32(np.inf if k > 0 else -np.inf))
            exact = Fraction(int(w)) * Fraction(float(sc))
            if nearest_f32(exact) == Fraction(float(tau)) and nearest_bf16(Fraction(float(tau))) != nearest_bf16(exact):
                ws.append(int(w))
                ss.append(sc)
                break
        if len(ws) == 24:
            break
    assert len(ws) == 24
    got = bf16.to_f64(P.dequant_int8(np.array(ws, dtype=np.int8)[None, :], np.array(ss, dtype=np.float32)))[0]
    for k, (w, sc) in enumerate(zip(ws, ss)):
        exact = Fraction(w) * Fraction(float(sc))
        assert got[k] == nearest_bf16(nearest_f32(exact))
        assert got[k] != nearest_bf16(exact)                     # the case is decisive
