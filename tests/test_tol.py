"""The attention tolerance helper itself (CPU): each bound fails on its own."""
import numpy as np
import pytest

from tests import _tol


def test_exact_passes():
    ref = np.linspace(-3, 3, 101)
    r = _tol.check(ref.copy(), ref, "bf16")
    assert r["max_abs"] == 0 and r["max_rel_big"] == 0


def test_relative_bound_fails_alone():
    # |ref| = 0.15: abs error 1.9e-3 is within 2e-3, but 1.27 % relative
    ref = np.array([0.15, -0.5, 0.01])
    out = ref + np.array([1.9e-3, 0.0, 0.0])
    with pytest.raises(AssertionError, match="max rel error"):
        _tol.check(out, ref, "fp16")


def test_absolute_bound_fails_alone():
    # |ref| = 0.05 is below the relative floor: 2.5e-3 absolute must fail
    ref = np.array([0.05, 1.0])
    out = ref + np.array([2.5e-3, 0.0])
    with pytest.raises(AssertionError, match="max abs error"):
        _tol.check(out, ref, "bf16")


def test_bf16_rounding_is_held_to_the_relative_bound_only():
    # bf16 at |ref| = 1: half an ulp is 3.9e-3, above the absolute bound; the
    # relative bound (1 %) still applies there
    ref = np.array([1.0, 0.3])
    _tol.check(ref + np.array([3.9e-3, 0.0]), ref, "bf16")
    with pytest.raises(AssertionError, match="max rel error"):
        _tol.check(ref + np.array([1.1e-2, 0.0]), ref, "bf16")
    # in fp16 the same element is held to 2e-3
    with pytest.raises(AssertionError, match="max abs error"):
        _tol.check(ref + np.array([3.9e-3, 0.0]), ref, "fp16")


def test_non_finite_output_fails():
    ref = np.array([0.2, 0.3])
    with pytest.raises(AssertionError, match="non-finite"):
        _tol.check(np.array([np.nan, 0.3]), ref, "fp16")
