"""The tolerance check of the GPU parity tests, on synthetic arrays (no GPU):
the kappa-scaled bound relaxes only ill-conditioned rows and reports what it
relaxed."""
import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16_MAX, compare


def _rows(n=8, dv=16, seed=0):
    rng = np.random.default_rng(seed)
    want = rng.standard_normal((n, dv))
    return want, want.copy()


def test_plain_bound_holds_and_fails():
    want, got = _rows()
    got[3, 5] += 0.5 * TOL_BF16_MAX
    compare(torch.from_numpy(got), want, "bf16")
    got[3, 5] += TOL_BF16_MAX
    with pytest.raises(AssertionError):
        compare(torch.from_numpy(got), want, "bf16")


def test_kappa_relaxes_an_ill_conditioned_row_and_reports_it():
    want, got = _rows(n=64, dv=64)
    got[3, 5] += 3 * TOL_BF16_MAX  # above the plain bound, below 5x it
    kappa = np.ones(64)
    kappa[3] = 5.0
    st = compare(torch.from_numpy(got), want, "bf16", kappa=kappa)
    assert st["rows_over_plain_bound"] == 1
    assert st["min_kappa_over_plain_bound"] == 5.0
    assert st["max_abs"] == pytest.approx(3 * TOL_BF16_MAX, rel=1e-6)
    assert st["well_conditioned_rows_over"] == 0


def test_kappa_never_relaxes_a_well_conditioned_row():
    want, got = _rows(n=64, dv=64)
    got[7, 1] += 1.2 * TOL_BF16_MAX
    kappa = np.ones(64)
    kappa[7] = 1.4  # a scaled bound would admit 1.4 x 2e-2, the plain one does not
    with pytest.raises(AssertionError, match="well_conditioned_rows_over"):
        compare(torch.from_numpy(got), want, "bf16", kappa=kappa)


def test_kappa_bound_still_caps_ill_conditioned_rows():
    want, got = _rows(n=64, dv=64)
    got[9, 0] += 6 * TOL_BF16_MAX
    kappa = np.ones(64)
    kappa[9] = 5.0
    with pytest.raises(AssertionError):
        compare(torch.from_numpy(got), want, "bf16", kappa=kappa)
