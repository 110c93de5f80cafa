"""Pins of the oracle's bf16 rounding against torch's conversion and brute force."""
import numpy as np
import torch

from oracle import bf16


def _torch_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_from_f32_matches_torch_rounding():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 3,
        rng.standard_normal(1000).astype(np.float32) * 1e-39,   # fp32 subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 1.0, 1.00390625, 1.01171875,
                  3.3895314e38, -3.3895314e38], dtype=np.float32),
    ])
    # every tie pattern: low 16 bits = 0x8000 with both parities of the kept bit
    ties = (np.arange(0, 1 << 16, 7, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    x = np.concatenate([x, ties])
    assert np.array_equal(bf16.from_f32(x), _torch_bits(x))


def test_widen_is_exact_round_trip():
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = bf16.to_f32(allbits)
    finite = np.isfinite(f)
    assert np.array_equal(bf16.from_f32(f[finite]), allbits[finite])
    assert np.array_equal(bf16.to_f64(allbits[finite]), f[finite].astype(np.float64))


def test_from_f64_single_rounding_cases():
    cases = {
        1.0 + 2.0 ** -8: 1.0,                       # tie, kept bit even: down
        1.0 + 3 * 2.0 ** -8: 1.0 + 2.0 ** -6,       # tie, kept bit odd: up to even
        1.0 + 2.0 ** -8 + 2.0 ** -40: 1.0 + 2.0 ** -7,  # just above a tie: up (fp32 would tie down)
        -(1.0 + 2.0 ** -8 + 2.0 ** -40): -(1.0 + 2.0 ** -7),
        2.0 ** -130 + 2.0 ** -134: 2.0 ** -130,     # bf16 subnormal range, tie to even
        0.0: 0.0,
    }
    x = np.array(list(cases.keys()))
    want = np.array(list(cases.values()))
    assert np.array_equal(bf16.to_f64(bf16.from_f64(x)), want)


def test_from_f64_brute_force_nearest():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))
    got = bf16.to_f64(bf16.from_f64(x))
    # brute force: the two bf16 neighbours by enumeration of the truncated pattern
    lo_bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    cands = []
    for delta in (-1, 0, 1):
        cb = (lo_bits.astype(np.int64) + delta).astype(np.uint16)
        cands.append(bf16.to_f64(cb))
    cands = np.stack(cands)                       # [3, n]
    err = np.abs(cands - x[None])
    best = err.min(axis=0)
    assert np.array_equal(np.abs(got - x), best)  # got is one of the nearest neighbours
    # and among equally near neighbours the even pattern is taken
    gb = bf16.from_f64(x)
    ties = (err == best[None]).sum(axis=0) > 1
    assert np.all(gb[ties] % 2 == 0)
