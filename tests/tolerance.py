"""Parity tolerance for bf16 outputs.

The stated bound is max-abs error <= 2e-2 and mean-abs error <= 2e-3 on bf16
outputs and gradients, lse within 1e-3.  A bf16 number carries 8 significant
bits, so rounding a value in [2^e, 2^(e+1)) to bf16 alone can move it by half
a unit in the last place, 2^(e-8): 0.0156 for values in [4, 8) and more than
2e-2 from 8 upwards.  The max-abs bound is therefore applied to the error in
excess of that unavoidable output rounding (of the reference value, or of the
larger of two compared bf16 results); the mean-abs bound is applied to the raw
error.

Every check records its raw max-abs error beside the error beyond output
rounding (RESULTS); the test session prints them as a summary.
"""
import os

import numpy as np

TOL_MAX, TOL_MEAN, TOL_LSE = 2e-2, 2e-3, 1e-3

# (name, raw max-abs, max-abs beyond output rounding, mean-abs, tol_max, tol_mean)
RESULTS = []


NOTES = []


def note(msg):
    """A line for the session summary (e.g. how long the fp64 oracle took)."""
    NOTES.append(msg)


def _record(name, raw, excess, mean, tol_max, tol_mean):
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    RESULTS.append((f"{test}::{name}" if test else name, raw, excess, mean, tol_max, tol_mean))


def bf16_half_ulp(x):
    """Half a bf16 unit in the last place at the magnitude of x (elementwise)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, np.finfo(np.float64).tiny)))
    return np.where(a > 0, np.exp2(e - 8.0), 0.0)


def check_bf16(name, got, want, tol_max=TOL_MAX, tol_mean=TOL_MEAN, ulps=1):
    """Assert the bf16 output `got` matches `want`; `ulps` half-ulps of output
    rounding are excused from the max-abs bound (2 when both sides are bf16)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - want)
    excess = np.maximum(err - ulps * bf16_half_ulp(np.maximum(np.abs(want), np.abs(got))), 0.0)
    if err.size:
        _record(name, float(err.max()), float(excess.max()), float(err.mean()), tol_max, tol_mean)
    assert excess.max() <= tol_max and err.mean() <= tol_mean, (
        f"{name}: max-abs {err.max():.3e}, beyond bf16 output rounding {excess.max():.3e} (tol {tol_max}), "
        f"mean-abs {err.mean():.3e} (tol {tol_mean})")


def check_fp32(name, got, want, tol=TOL_LSE):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - want)
    if err.size:
        _record(name, float(err.max()), float(err.max()), float(err.mean()), tol, tol)
    assert err.max() <= tol, f"{name}: max-abs {err.max():.3e} (tol {tol})"
