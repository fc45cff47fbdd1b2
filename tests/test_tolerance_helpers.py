"""The parity tolerances' helper (CPU): the relative-RMSE floor of the
gradient comparisons may only apply where the reference gradient is zero."""
import numpy as np
import pytest

from gpu_util import GRAD_REL_RMSE, rel_rmse


def test_floor_applies_to_a_zero_reference():
    # dQ / dK with a single key are zero in the oracle; the GPU leaves float32
    # rounding residue, measured against the floor
    assert rel_rmse(np.full(16, 1e-7), np.zeros(16)) == pytest.approx(1e-3)


def test_floor_refuses_a_small_nonzero_reference():
    # a real gradient of RMS 5e-5 must not be compared against the floor
    ref = np.full(16, 5e-5)
    with pytest.raises(AssertionError):
        rel_rmse(ref * 1.5, ref)


def test_ordinary_reference_is_relative():
    ref = np.linspace(-1.0, 1.0, 64)
    assert rel_rmse(ref * (1 + GRAD_REL_RMSE / 2), ref) == pytest.approx(GRAD_REL_RMSE / 2)
