"""Shared helpers of the parity tests: the tolerance check and GPU runners.

Tolerance (stated for attention outputs): compare the kernel's bf16 output with
the exact fp64 oracle rounded to bf16. Pass if the mean absolute difference is
at most 1e-3 and the maximum at most 1e-2, except that an element may exceed
1e-2 when it is a one-ulp disagreement of the two bf16 values (a single bf16
ulp is 2^-6..2^-4 at the output magnitudes here, so the literal maximum bar
cannot hold for any correctly rounded kernel). KV-cache and rotated-Q contents
must match bit for bit.
"""
from __future__ import annotations

import json
import os

import numpy as np

from oracle import bf16

MEAN_TOL = 1e-3
MAX_TOL = 1e-2


def compare(got_bits: np.ndarray, ref_bits: np.ndarray) -> dict:
    g = bf16.to_f64(got_bits)
    r = bf16.to_f64(ref_bits)
    d = np.abs(g - r)
    big = d > MAX_TOL
    ulps = np.abs(got_bits.astype(np.int64) - ref_bits.astype(np.int64))
    return {
        "finite": bool(np.all(np.isfinite(g))),
        "max_abs": float(d.max()) if d.size else 0.0,
        "mean_abs": float(d.mean()) if d.size else 0.0,
        "n_above_max_tol": int(big.sum()),
        "frac_above_max_tol": float(big.mean()) if d.size else 0.0,
        "max_ulps_above_tol": int(ulps[big].max()) if big.any() else 0,
        "frac_exact": float((ulps == 0).mean()) if d.size else 1.0,
    }


def assert_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> dict:
    st = compare(got_bits, ref_bits)
    log = os.environ.get("GROK_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, "n": int(got_bits.size), **st}) + "\n")
    assert st["finite"], f"{what}: non-finite outputs"
    assert st["mean_abs"] <= MEAN_TOL, f"{what}: mean abs {st['mean_abs']:.3e} > {MEAN_TOL} ({st})"
    assert st["max_ulps_above_tol"] <= 1, f"{what}: elements above {MAX_TOL} beyond one bf16 ulp ({st})"
    return st
