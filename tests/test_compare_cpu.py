"""The GPU tests' comparison rule (tests/gpu_common.py, assert_close), checked on the CPU.

Gradients are held to the bound relative to their RMS; a gradient that vanishes exactly (one visible key per
query: dS = 0, so dQ = dK = 0) has no RMS to speak of, and is measured on the scale of the case's dV instead.
"""
import numpy as np
import pytest

from gpu_common import assert_close


def test_relative_bound_on_an_ordinary_gradient():
    ref = np.random.default_rng(1).standard_normal((4, 64))
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert_close(ref + 5e-4 * rms, ref, "bf16", "dq", rel_rms=True, scale=1.0)
    with pytest.raises(AssertionError):
        assert_close(ref + 5e-2 * rms, ref, "bf16", "dq", rel_rms=True, scale=1.0)


def test_vanishing_gradient_is_measured_on_the_given_scale():
    ref = np.zeros((4, 64))
    assert_close(np.zeros((4, 64)), ref, "bf16", "dq", rel_rms=True, scale=1.0)
    assert_close(np.full((4, 64), 1e-6), ref, "f32", "dq", rel_rms=True, scale=1.0)
    noise = np.full((4, 64), 1e-17)                       # float64 rounding noise as the reference
    assert_close(np.zeros((4, 64)), noise, "f32", "dq", rel_rms=True, scale=1.0)
    with pytest.raises(AssertionError):
        assert_close(np.full((4, 64), 0.5), ref, "bf16", "dq", rel_rms=True, scale=1.0)


def test_scale_does_not_loosen_an_ordinary_gradient():
    # a small but non-vanishing gradient keeps its own RMS as the measure
    ref = 1e-3 * np.random.default_rng(2).standard_normal((4, 64))
    with pytest.raises(AssertionError):
        assert_close(ref * 1.1, ref, "bf16", "dq", rel_rms=True, scale=1.0)
