"""CPU check of the polynomial exp2 used for part of the forward's exponentials.

The steps of `exp2_poly_pair` (csrc/tc_ptx.cuh) are replayed in numpy float32:
clamp at -126, round-to-nearest via the 1.5 * 2^23 shifter, f = x - n,
a degree-3 polynomial for 2^f, and 2^n added to the exponent bits.  The
coefficients are read from the CUDA source so the test follows the kernel.
The result must stay within 1e-4 relative of 2^x (P is then rounded to bf16,
whose own step is 2^-9) on a dense grid over the range the softmax produces.
"""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def coefficients():
    src = open(os.path.join(ROOT, "domain_ring_attention_gb300", "csrc", "tc_ptx.cuh")).read()
    body = src[src.index("void exp2_poly_pair"):]
    body = body[:body.index("\n}\n")]
    vals = [float(v) for v in re.findall(r"f2_pack\((-?[0-9.]+)f, \1f\)", body)]
    # shifter, -shifter, -1, then c3, c2, c1, c0
    assert vals[:3] == [12582912.0, -12582912.0, -1.0], vals
    return np.float32(vals[3]), np.float32(vals[4]), np.float32(vals[5]), np.float32(vals[6])


def poly_exp2(x):
    c3, c2, c1, c0 = coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t + np.float32(-12582912.0)).astype(np.float32)
    f = (n * np.float32(-1.0) + x).astype(np.float32)
    p = (f * c3 + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = (t.view(np.uint32).astype(np.uint64) * (1 << 23) + p.view(np.uint32).astype(np.uint64)) % (1 << 32)
    return bits.astype(np.uint32).view(np.float32)


def test_poly_exp2_relative_error():
    x = np.linspace(-125.0, 8.0, 2_000_003, dtype=np.float64).astype(np.float32)
    got = poly_exp2(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got / ref - 1.0)
    assert rel.max() < 1e-4, rel.max()


def test_poly_exp2_special_values():
    x = np.array([0.0, 1.0, -1.0, 8.0, -0.5, 0.5, -126.0, -200.0, -np.inf], dtype=np.float32)
    got = poly_exp2(x)
    assert np.all(np.isfinite(got)) and np.all(got > 0)
    np.testing.assert_allclose(got[:6], np.exp2(x[:6].astype(np.float64)), rtol=1e-4)
    assert got[-1] < 1e-37 and got[-2] < 1e-37      # clamped: ~2^-126 instead of 0
