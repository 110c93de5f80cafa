"""Pins of the oracle's RoPE and cache append (closed forms, invariants, the pages' examples)."""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import bf16, rope
from tests.exact_util import nearest_bf16, nearest_f32


def _rand_bf16(rng, shape, scale=3.0):
    return bf16.from_f32((rng.standard_normal(shape) * scale).astype(np.float32))


def test_inv_freq_closed_form():
    f = rope.inv_freq(128)
    assert f.dtype == np.float32 and f.shape == (64,)
    assert f[0] == np.float32(1.0)                  # omega_0 = 1 (ch. 4 §4.3.2)
    want = np.array([10000.0 ** (-j / 64.0) for j in range(64)])
    assert np.all(np.abs(f.astype(np.float64) - want) <= 2 * np.spacing(f).astype(np.float64))
    assert np.all(np.diff(f) < 0)
    # lowest frequency: 10000**(-126/128) ~ 1.155e-4 (the page rounds it to "1.17e-4")
    assert abs(float(f[63]) - 1.1548e-4) < 1e-7


def test_rotate_half_neox_pairing():
    x = np.array([0.0, 1.0, 2.0, 3.0], dtype=np.float32)
    assert np.array_equal(rope.rotate_half(x), np.array([-2.0, -3.0, 0.0, 1.0], dtype=np.float32))


def test_head_dim_4_worked_example_pairs_i_with_i_plus_half():
    """ch. 4 §4.3.1.1: with head_dim 4 the rotation pairs (x0, x2) and (x1, x3)."""
    rng = np.random.default_rng(3)
    x = _rand_bf16(rng, (1, 5, 1, 4))
    offset = np.array([7])
    y = bf16.to_f64(rope.rotary_embedding(x, offset))
    xf = bf16.to_f64(x)
    w = [1.0, 10000.0 ** (-0.5)]                    # omega_i = base**(-2i/d), d = 4
    for ti in range(5):
        t = 7 + ti
        for i in range(2):
            c, s = math.cos(t * w[i]), math.sin(t * w[i])
            a, b = xf[0, ti, 0, i], xf[0, ti, 0, i + 2]
            want = (a * c - b * s, a * s + b * c)    # 2x2 rotation of (x_i, x_{i+d/2})
            got = (y[0, ti, 0, i], y[0, ti, 0, i + 2])
            for g_, w_ in zip(got, want):
                assert abs(g_ - w_) <= 2 ** -7 * max(abs(w_), 1e-3) + 1e-6


def test_position_zero_is_identity_bit_exact():
    rng = np.random.default_rng(4)
    x = _rand_bf16(rng, (2, 1, 8, 128))
    assert np.array_equal(rope.rotary_embedding(x, np.array([0, 0])), x)


def test_rotation_preserves_norm():
    rng = np.random.default_rng(5)
    x = _rand_bf16(rng, (1, 64, 8, 128))
    off = np.array([1000])
    y = bf16.to_f64(rope.rotary_embedding(x, off))
    n0 = np.linalg.norm(bf16.to_f64(x), axis=-1)
    n1 = np.linalg.norm(y, axis=-1)
    assert np.all(np.abs(n1 / n0 - 1) < 2 ** -8)


def test_dot_product_depends_only_on_relative_position():
    """<R(m) q, R(n) k> = <R(m - n) q, k> (ch. 4, RoPE motivation)."""
    rng = np.random.default_rng(6)
    q = _rand_bf16(rng, (1, 1, 1, 128))
    k = _rand_bf16(rng, (1, 1, 1, 128))
    for m, n in [(5, 3), (100, 37), (4000, 3990), (8191, 0)]:
        qm = bf16.to_f64(rope.rotary_embedding(q, np.array([m])))[0, 0, 0]
        kn = bf16.to_f64(rope.rotary_embedding(k, np.array([n])))[0, 0, 0]
        qd = bf16.to_f64(rope.rotary_embedding(q, np.array([m - n])))[0, 0, 0]
        k0 = bf16.to_f64(k)[0, 0, 0]
        lhs, rhs = qm @ kn, qd @ k0
        scale = np.linalg.norm(qm) * np.linalg.norm(kn)
        assert abs(lhs - rhs) < 2 ** -6 * scale


def test_offset_equals_per_token_positions():
    """t = arange(T) + offset: a chunk rotated at once equals its tokens rotated one by one."""
    rng = np.random.default_rng(7)
    x = _rand_bf16(rng, (2, 6, 3, 128))
    off = np.array([0, 6144])
    y = rope.rotary_embedding(x, off)
    for b in range(2):
        for i in range(6):
            yi = rope.rotary_embedding(x[b:b + 1, i:i + 1], np.array([off[b] + i]))
            assert np.array_equal(y[b, i], yi[0, 0])


def test_cos_sin_table_rounding_is_decided_for_every_supported_position():
    """All positions < 65536: each fp64 cos/sin is far from an fp32 midpoint (guard never fires)."""
    t = np.arange(rope.MAX_POSITION, dtype=np.float32)[None, :]
    ph = rope.phase(t, rope.inv_freq(128))
    c, s = rope.cos_sin(ph)                        # raises on a near-tie
    assert c.dtype == np.float32 and s.dtype == np.float32
    assert np.all(c[0, 0] == 1.0) and np.all(s[0, 0] == 0.0)


def test_near_tie_guard_fires():
    mid = np.float64(np.float32(1.5)) + np.spacing(np.float32(1.5)) / 2
    with pytest.raises(ArithmeticError):
        rope.check_no_near_ties(np.array([mid]))


def test_positions_out_of_range_rejected():
    with pytest.raises(ValueError):
        rope.positions(np.array([65530]), 16)


def test_update_into_writes_only_the_slice():
    rng = np.random.default_rng(8)
    mem = _rand_bf16(rng, (3, 16, 8, 128))
    upd = _rand_bf16(rng, (3, 4, 8, 128))
    start = np.array([0, 5, 12])
    out = rope.update_into(mem, start, upd)
    for b in range(3):
        s = start[b]
        assert np.array_equal(out[b, s:s + 4], upd[b])
        assert np.array_equal(out[b, :s], mem[b, :s])
        assert np.array_equal(out[b, s + 4:], mem[b, s + 4:])
    with pytest.raises(ValueError):
        rope.update_into(mem, np.array([0, 0, 13]), upd)


def test_rope_kv_append_rotates_k_not_v():
    rng = np.random.default_rng(9)
    q = _rand_bf16(rng, (1, 4, 48, 128))
    k = _rand_bf16(rng, (1, 4, 8, 128))
    v = _rand_bf16(rng, (1, 4, 8, 128))
    ck = _rand_bf16(rng, (1, 32, 8, 128))
    cv = _rand_bf16(rng, (1, 32, 8, 128))
    start = np.array([10])
    q_rot, nk, nv = rope.rope_kv_append(q, k, v, start, ck, cv)
    assert np.array_equal(nv[0, 10:14], v[0])                       # V is a bit copy
    assert np.array_equal(nk[0, 10:14], rope.rotary_embedding(k, start)[0])
    assert np.array_equal(q_rot, rope.rotary_embedding(q, start))
    assert not np.array_equal(nk[0, 10:14], k[0])


def _rotated_brute_force(x_f, t: int, i: int, freqs) -> float:
    """One output feature by exact rationals: the pages' fp32 chain, each step rounded on its own."""
    dim = len(x_f)
    ph = nearest_f32(Fraction(t) * Fraction(float(freqs[i % (dim // 2)])))    # fp32 t * fp32 inv_freq
    c = nearest_f32(Fraction(math.cos(float(ph))))
    s = nearest_f32(Fraction(math.sin(float(ph))))
    partner = -x_f[i + dim // 2] if i < dim // 2 else x_f[i - dim // 2]      # rotate_half
    a = nearest_f32(Fraction(float(x_f[i])) * c)
    b = nearest_f32(Fraction(float(partner)) * s)
    return nearest_bf16(nearest_f32(a + b))


def test_rotation_follows_the_fp32_rounding_chain_exactly():
    """ch. 4 §4.3.1 in the pages' dtypes: fp32 positions and inv_freq, their fp32 product as
    the phase, fp32 cos and sin, bf16 x promoted to fp32, x*cos and rotate_half(x)*sin and
    their sum each rounded to fp32, then the cast to bf16. Checked by exact-rational brute
    force near the largest position, on random elements and on the elements where rounding
    the products and the sum only once would change the bf16 result."""
    rng = np.random.default_rng(17)
    T, H, off = 2048, 8, rope.MAX_POSITION - 2048
    x = _rand_bf16(rng, (1, T, H, 128))
    y = bf16.to_f64(rope.rotary_embedding(x, np.array([off])))
    freqs = rope.inv_freq(128)          # pinned on its own by the closed form above
    xf = bf16.to_f32(x)[0]
    # selection only: elements where one rounding of x*c + rh*s differs from three
    t = np.arange(T, dtype=np.float32) + np.float32(off)
    ph = (t[:, None] * freqs[None, :]).astype(np.float32)
    ph = np.concatenate((ph, ph), axis=-1)[:, None, :].astype(np.float64)
    c, s = np.cos(ph).astype(np.float32), np.sin(ph).astype(np.float32)
    rh = np.concatenate((-xf[..., 64:], xf[..., :64]), axis=-1)
    once = bf16.from_f64(xf.astype(np.float64) * c + rh.astype(np.float64) * s)
    thrice = bf16.from_f32((xf * c).astype(np.float32) + (rh * s).astype(np.float32))
    decisive = [tuple(e) for e in np.argwhere(once != thrice)[:16]]
    assert len(decisive) >= 8
    picks = decisive + [tuple(int(v) for v in rng.integers((T, H, 128))) for _ in range(96)]
    for ti, h, i in picks:
        assert y[0, ti, h, i] == _rotated_brute_force(xf[ti, h], off + ti, i, freqs), (ti, h, i)
