"""Error bound of the FMA-pipe 2^x used for part of the forward softmax
(exp2_poly2 in csrc/tc_common.cuh): the header's coefficients, run through
the same fp32 steps on the CPU (clamp at -126, rounding by the 1.5 * 2^23
constant, Horner scheme with fused multiply-adds, exponent-field add), stay
within 3e-6 relative of 2^x on [-126, 0] and never produce a negative, NaN
or oversized value below that range.  The GPU path itself is covered by the
parity tests (O and LSE against the oracle)."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(__file__), "..", "content_adaptive_block_02_b300", "csrc",
                   "tc_common.cuh")


def _coeffs():
    txt = open(HDR).read()
    c = [float(re.search(r"kExp2C%d = ([0-9.e+-]+)f" % k, txt).group(1)) for k in range(5)]
    return [np.float32(v) for v in c]


def _fma32(a, b, c):
    # a*b of two fp32 values is exact in fp64; one rounding of the sum to fp32
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _exp2_poly(x):
    c = _coeffs()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic).astype(np.float32)).astype(np.float32)
    p = _fma32(np.full_like(f, c[4]), f, np.full_like(f, c[3]))
    for k in (2, 1, 0):
        p = _fma32(p, f, np.full_like(f, c[k]))
    bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_relative_error_on_the_softmax_range():
    x = np.concatenate([np.linspace(-126.0, 0.0, 2_000_001),
                        -np.random.default_rng(0).exponential(3.0, 200_000)]).astype(np.float32)
    x = x[x >= -126.0]
    y = _exp2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.all(np.isfinite(y))
    assert np.max(np.abs(y - ref) / ref) < 3e-6


def test_exact_at_zero_within_bound_and_monotone_grid():
    y0 = float(_exp2_poly(np.zeros(1, np.float32))[0])
    assert abs(y0 - 1.0) < 3e-6
    x = np.linspace(-20.0, 0.0, 100_001).astype(np.float32)
    y = _exp2_poly(x)
    assert np.all(np.diff(y.astype(np.float64)) >= -3e-6 * y[1:])


def test_below_the_range_is_tiny_and_nonnegative():
    x = np.array([-126.5, -127.0, -200.0, -1e6, -3.0e38], np.float32)
    y = _exp2_poly(x).astype(np.float64)
    assert np.all(y >= 0.0) and np.all(y <= 2.0 ** -125)
