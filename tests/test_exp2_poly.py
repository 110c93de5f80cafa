"""The prefill softmax evaluates part of its exp2 as a polynomial on the FMA pipe.

The constants live in the CUDA source; this test reads them from there and
checks the same fp32 steps (round to nearest integer by adding 1.5 * 2^23,
Horner with fused multiply-adds, exponent-field add) against 2^x in fp64 over
every input the kernel can give it: x = 30 log2(e) (tanh(y) - 1), i.e. [-86.6, 0].
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "grok_gqa_attention_gb300", "csrc", "common.cuh")
K_T = 30.0 * 1.4426950408889634


def _function_body():
    src = open(SRC).read()
    start = src.index("void exp2_poly_f2(")
    return src[start:src.index("\n}\n", start)]


def _coefficients():
    """Horner coefficients from highest to lowest degree, as fp32."""
    consts = re.findall(r"f2_pack\((0x[0-9a-fA-F.]+p[-+]?\d+)f,\s*(0x[0-9a-fA-F.]+p[-+]?\d+)f\)", _function_body())
    assert consts and all(a == b for a, b in consts)
    return [np.float32(float.fromhex(a)) for a, _ in consts]


def _fma32(a, b, c):
    # an fp32 fused multiply-add: the fp64 product of two fp32 values is exact
    return (a.astype(np.float64) * b.astype(np.float64) + np.float64(c)).astype(np.float32)


def _device_exp2(x):
    big = np.float32(12582912.0)
    assert "f2_pack(12582912.0f, 12582912.0f)" in _function_body()
    t = (x + big).astype(np.float32)
    f = (x - (t - big).astype(np.float32)).astype(np.float32)
    c = _coefficients()
    q = np.full_like(f, c[0])
    for ck in c[1:]:
        q = _fma32(q, f, ck)
    return (q.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))).view(np.float32)


def test_coefficients_are_a_degree_4_fit_of_exp2():
    c = _coefficients()
    assert len(c) == 5
    # close to the Taylor coefficients (ln 2)^k / k! of 2^f
    taylor = [np.log(2.0) ** k / np.prod(range(1, k + 1)) for k in range(4, -1, -1)]
    assert np.allclose(np.array(c, dtype=np.float64), taylor, rtol=2e-2)


def test_relative_error_over_the_kernel_input_range():
    x = np.linspace(-2 * K_T, 0.0, 1_000_001).astype(np.float32)
    x = np.concatenate([x, np.float32([-0.5, 0.5 - 2 ** -24, -1.5, -86.5, -2 * K_T, 0.0])])
    x = x[x <= 0]
    got = _device_exp2(x).astype(np.float64)
    rel = np.abs(got / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 3e-6
    assert np.all(np.isfinite(got)) and np.all(got > 0)


def test_integer_arguments_are_near_exact_powers_of_two():
    x = -np.arange(0, 87, dtype=np.float32)
    got = _device_exp2(x).astype(np.float64)
    assert np.all(np.abs(got / np.exp2(x.astype(np.float64)) - 1.0) < 1e-6)
