"""The fp16-mode prefill softmax evaluates half of its tanh as a polynomial on the FMA pipe.

The constants live in the CUDA source; this test reads them from there and
checks the same fp32 steps (z = y*y, yz = y*z, Horner in z with fused
multiply-adds, t = fma(yz, q, y)) against tanh in fp64 over the range the
kernel allows it, |y| <= 1.5 (a warp whose chunk holds a larger |y| in one of
the polynomial's columns takes tanh.approx instead). The bar is the measured
absolute error of tanh.approx.f32 on sm_103 (7.8e-6): the polynomial must not
be less accurate than the instruction it replaces.
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "grok_gqa_attention_gb300", "csrc", "prefill.cu")
TANH_APPROX_ABS_ERR = 7.8e-6


def _source():
    return open(SRC).read()


def _function_body():
    src = _source()
    start = src.index("uint64_t tanh_poly_f2(")
    return src[start:src.index("\n}\n", start)]


def _range():
    m = re.search(r"constexpr float kTanhPolyRange = ([0-9.]+)f;", _source())
    return np.float32(float(m.group(1)))


def _coefficients():
    """Q's coefficients from highest to lowest degree, as fp32."""
    consts = re.findall(r"f2_pack\((-?0x[0-9a-fA-F.]+p[-+]?\d+)f,\s*(-?0x[0-9a-fA-F.]+p[-+]?\d+)f\)", _function_body())
    assert consts and all(a == b for a, b in consts)
    return [np.float32(float.fromhex(a)) for a, _ in consts]


def _fma32(a, b, c):
    # an fp32 fused multiply-add: the fp64 product of two fp32 values is exact
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(np.float32)


def _device_tanh(y):
    y = y.astype(np.float32)
    z = (y * y).astype(np.float32)
    yz = (y * z).astype(np.float32)
    c = _coefficients()
    q = _fma32(c[0], z, c[1])
    for ck in c[2:]:
        q = _fma32(q, z, ck)
    return _fma32(yz, q, y)


def test_coefficients_follow_the_taylor_series_of_tanh():
    c = _coefficients()
    assert len(c) == 6
    # tanh(y) = y - y^3/3 + 2y^5/15 - 17y^7/315 + ...: the low-order terms of a
    # good fit on [0, 1.5] stay near them (higher ones absorb the truncation).
    low = np.array(c[::-1][:3], dtype=np.float64)
    assert np.allclose(low, [-1 / 3, 2 / 15, -17 / 315], rtol=0.1)


def test_absolute_error_over_the_allowed_range():
    a = _range()
    assert a == np.float32(1.5)
    y = np.linspace(-a, a, 2_000_001).astype(np.float32)
    # the kernel checks the raw logit against kTanhPolyRange / kY, so y = fl(s * kY)
    # may exceed the range by a rounding or two
    edge = np.float32(a) * (1 + np.arange(0, 8) * 2.0 ** -24)
    y = np.concatenate([y, edge.astype(np.float32), -edge.astype(np.float32), np.float32([0.0, 2 ** -20, 1e-3])])
    err = np.abs(_device_tanh(y).astype(np.float64) - np.tanh(y.astype(np.float64)))
    assert err.max() < 3.2e-6 < TANH_APPROX_ABS_ERR


def test_odd_and_bounded():
    y = np.linspace(0, 1.5, 100_001).astype(np.float32)
    t = _device_tanh(y)
    assert np.array_equal(_device_tanh(-y), -t)
    assert np.all(np.abs(t) < 1.0) and np.all(np.diff(t.astype(np.float64)) >= 0)


def test_useless_beyond_the_range():
    """Why the kernel checks the range: a little beyond it the fit departs from tanh."""
    y = np.float32([2.5, 3.0])
    assert np.all(np.abs(_device_tanh(y) - np.tanh(y.astype(np.float64))) > 1e-4)
