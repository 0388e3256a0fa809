"""The GELU epilogues of the FFN GEMM evaluate the normal CDF from erfc(z) =
t exp(-z^2 + c(t)), t = 1 / (1 + z/2), with the ten Chebyshev-fitted
coefficients of Numerical Recipes in C (2nd ed., section 6.2, erfcc), whose
fractional error the book states as below 1.2e-7 everywhere.  The GPU parity
tests see that function only through bf16 outputs; this reads the
coefficients out of the kernel source and checks, on the CPU, that they
meet the stated bound (a mistyped digit would not), and that the fp32
evaluation order of the kernel keeps Phi within its rounding bound of an
independent erfc over the whole range, tail included.
"""
import os
import re

import numpy as np
import pytest

SRC = os.path.join(os.path.dirname(__file__), "..", "sequence_blockwise_self_gb300", "csrc", "ffn.cu")


def _coefficients():
    src = open(SRC).read()
    body = src[src.index("float normal_cdf(float a, float z2)"):]
    body = body[:body.index("\n}\n")]
    first = float(re.search(r"float c = (-?[0-9.]+)f;", body).group(1))
    rest = [float(v) for v in re.findall(r"c = fmaf\(c, t, (-?[0-9.]+)f\);", body)]
    return [first] + rest          # highest degree first, as Horner's rule runs


def _erfc_fit(z, coef, dtype):
    z = np.asarray(z, dtype=dtype)
    t = (dtype(1) / (dtype(1) + dtype(0.5) * z)).astype(dtype)
    c = np.full_like(z, dtype(coef[0]))
    for k in coef[1:]:
        c = (c * t + dtype(k)).astype(dtype)
    return t, c


def test_the_kernel_has_the_ten_coefficients():
    coef = _coefficients()
    assert len(coef) == 10
    assert coef[-1] == pytest.approx(-1.26551223) and coef[0] == pytest.approx(0.17087277)


def test_the_fit_meets_its_stated_fractional_error():
    special = pytest.importorskip("scipy.special")
    z = np.linspace(0.0, 26.0, 400001)
    t, c = _erfc_fit(z, _coefficients(), np.float64)
    fit = t * np.exp(-z * z + c)
    ref = special.erfc(z)
    ok = ref > 1e-300
    assert np.max(np.abs(fit[ok] / ref[ok] - 1.0)) < 1.2e-7


def test_fp32_evaluation_keeps_phi_accurate_in_the_tail():
    """The kernel's order of operations in fp32 (exp in fp64 here: the
    device exponential adds its own few-ulp error, covered by the GPU test's
    3e-5 slack): Phi(a) within 6e-7 + 1.2e-7 z^2 relative for a in [-12, 12]
    -- the fit (1.2e-7) and a handful of fp32 roundings of O(1) values
    (t, the Horner steps, the products; 6e-8 each), plus the roundings of
    z^2 = a^2 / 2 and of c - z^2, each up to half an ulp of z^2 inside the
    exponential."""
    special = pytest.importorskip("scipy.special")
    f = np.float32
    a = np.linspace(-12.0, 12.0, 240001).astype(f)
    z2 = (f(0.5) * a * a).astype(f)
    z = (np.abs(a) * f(0.70710678118654752)).astype(f)
    t, c = _erfc_fit(z, _coefficients(), f)
    half_erfc = (f(0.5) * t * np.exp((c - z2).astype(np.float64)).astype(f)).astype(f)
    phi = np.where(a < 0, half_erfc, (f(1) - half_erfc).astype(f))
    ref = 0.5 * special.erfc(-a.astype(np.float64) / np.sqrt(2.0))
    bound = 6e-7 + 1.2e-7 * z2.astype(np.float64)
    assert np.all(np.abs(phi / ref - 1.0) <= bound)
