"""The agreement rules themselves (tests/parity.py), on hand-made arrays (CPU)."""
import numpy as np
import pytest

from tests import parity as P


def _pair(err_at_small):
    ref = np.array([[0.25, 300.0, -2.0]])
    out = ref.copy()
    out[0, 0] += err_at_small
    lse = np.array([10.0])
    return out, lse, ref, lse.copy()


def test_unit_scale_bound():
    out, lse, ref, rl = _pair(0.009)          # within 1e-2 of a small element
    P.check_out_lse(out, lse, ref, rl)
    out, lse, ref, rl = _pair(0.011)          # beyond it
    with pytest.raises(AssertionError):
        P.check_out_lse(out, lse, ref, rl)
    big = np.full((1, 1000), 300.0)           # relative above 1 (one element off)
    for rel, ok in ((9e-3, True), (1.1e-2, False)):
        o = big.copy()
        o[0, 7] *= 1 + rel
        if ok:
            P.check_out_lse(o, np.array([1.0]), big, np.array([1.0]))
        else:
            with pytest.raises(AssertionError):
                P.check_out_lse(o, np.array([1.0]), big, np.array([1.0]))


def test_packed_pool_bound_scales_with_the_largest_v():
    # an element of 0.25 built from rows of |V| up to 100: the logit-error
    # bound 2 * 2e-4 * 100 = 0.04 admits an error of 0.03, not one of 0.05
    out, lse, ref, rl = _pair(0.03)
    vmax = np.array([[100.0, 100.0, 100.0]])
    _, _, unit = P.check_out_lse(out, lse, ref, rl, vmax=vmax)
    assert unit == pytest.approx(P.OUT_MAX_ABS * 0.03 / 0.04)
    out, lse, ref, rl = _pair(0.05)
    with pytest.raises(AssertionError):
        P.check_out_lse(out, lse, ref, rl, vmax=vmax)
    # with small V the unit-scale bound still rules
    out, lse, ref, rl = _pair(0.011)
    with pytest.raises(AssertionError):
        P.check_out_lse(out, lse, ref, rl, vmax=np.array([[1.0, 1.0, 1.0]]))


def test_lse_is_absolute_and_neg_inf_must_match():
    out = np.zeros((1, 2))
    ref_lse = np.array([20.0, -np.inf])
    P.check_out_lse(out, ref_lse + np.array([9e-5, 0.0]), out, ref_lse)
    with pytest.raises(AssertionError):
        P.check_out_lse(out, ref_lse + np.array([1.1e-4, 0.0]), out, ref_lse)
    with pytest.raises(AssertionError):
        P.check_out_lse(out, np.array([20.0, 0.0]), out, ref_lse)
    P.check_out_lse(out, ref_lse + np.array([1.5e-4, 0.0]), out, ref_lse, lse_tol=P.LSE_TOL_DS_MLA)
