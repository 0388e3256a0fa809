"""The bf16 half-ulp used by the parity tolerance matches torch's bf16
rounding: every value moves by at most the computed half-ulp, and the bound
is reached (it is not loose by a factor of two)."""
import numpy as np
import torch

from tolerance import bf16_half_ulp


def test_half_ulp_bounds_bf16_rounding():
    x = np.random.default_rng(0).standard_normal(200000) * np.exp2(np.random.default_rng(1).integers(-6, 6, 200000))
    x = x.astype(np.float32).astype(np.float64)  # the kernels round fp32 accumulators to bf16
    r = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    hu = bf16_half_ulp(x)
    assert np.all(np.abs(r - x) <= hu * (1 + 1e-12))
    assert np.max(np.abs(r - x) / hu) > 0.99
    assert bf16_half_ulp(5.0) == 2.0 ** -6 and bf16_half_ulp(1.0) == 2.0 ** -8 and bf16_half_ulp(0.0) == 0.0
