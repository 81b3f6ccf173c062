"""Error bound of the library's FMA-pipe 2^y (CPU emulation of its fp32 steps).

The scoring kernel evaluates a share of its exponentials as 2^y = 2^f * 2^n with
n = round(y), |f| <= 1/2 and a degree-4 polynomial for 2^f.  This test reads the
coefficients from the CUDA source and checks, with float32 arithmetic, that the
relative error stays below 5e-6 over the range the kernel uses (y <= 0), and that
inputs below the clamp give a tiny non-negative value rather than garbage.
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "decode_kv_cache_03_gb300", "csrc", "kara_sm100.cuh")


def coeffs():
    text = open(SRC).read()
    c = {int(k): np.float32(float(v)) for k, v in re.findall(r"kExp2C(\d) = ([0-9.eE+-]+)f", text)}
    assert sorted(c) == [0, 1, 2, 3, 4]
    return [c[i] for i in range(5)]


def fma32(a, b, c):
    # exact product of two float32 values in float64, one rounding of the sum to float32
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def poly_exp2(y):
    c = coeffs()
    y = np.maximum(y.astype(np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)
    t = (y + magic).astype(np.float32)
    f = (y - (t - magic).astype(np.float32)).astype(np.float32)
    p = np.full_like(f, c[4])
    for k in (3, 2, 1, 0):
        p = fma32(p, f, np.full_like(f, c[k]))
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.view(np.float32)


def test_relative_error_bound():
    y = np.concatenate([np.linspace(-125.0, 0.0, 2_000_001, dtype=np.float32),
                        -np.random.default_rng(0).exponential(3.0, 200_000).astype(np.float32)])
    y = y[y >= -125.0]
    got = poly_exp2(y).astype(np.float64)
    ref = np.exp2(y.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 5e-6, rel.max()


def test_exact_at_integers_within_bound_and_positive_below_clamp():
    y = np.arange(-126, 1, dtype=np.float32)
    got = poly_exp2(y).astype(np.float64)
    assert np.all(np.abs(got - np.exp2(y.astype(np.float64))) / np.exp2(y.astype(np.float64)) < 5e-6)
    low = poly_exp2(np.float32([-126.4, -127.0, -500.0, -np.inf]))
    assert np.all(low >= 0) and np.all(low < 2.0 ** -125)
