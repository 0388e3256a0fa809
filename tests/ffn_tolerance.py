"""Parity bound for the blockwise feed-forward block (bf16 on the GPU against
the fp64 oracle).

The GPU computes y = x + gelu(x W1^T + b1) W2^T + b2 with bf16 operands,
fp32 accumulation and the hidden activation rounded to bf16 between the
layers (it is the second GEMM's operand); the oracle computes the same
block in fp64 from the same bf16 values.  Per element of y:
  * output rounding: half a bf16 ulp of y (at most 2^-8 |y|);
  * the hidden rounding carried through W2: each h_f moves by at most half
    a bf16 ulp (2^-8 |h_f|), roughly uniformly, so the error of y_d has
    standard deviation at most 2^-8 / sqrt(3) * sqrt(sum_f (h_f W2_fd)^2);
    six of those are allowed;
  * fp32 accumulation and the GELU evaluation (Phi to 1.2e-7 relative):
    1e-4 absolute (several orders below the terms above at these sizes).
On top, the errors must be typical, not bunched near their bounds: the
mean-abs error stays within a quarter of the mean bound (a faithful
computation lands near one sixth of it: one standard deviation plus a
quarter ulp of output rounding on average).
"""
import math

import numpy as np

import oracle
from tolerance import bf16_half_ulp


def f64(t):
    return t.detach().float().cpu().double().numpy()


def ffn_reference(x, w1, b1, w2, b2):
    """Oracle y for the rows of x (torch tensors, any device; w1 [F, D] and
    w2 [D, F] output-major) and the per-element bound on |y_gpu - y|."""
    W1, W2 = f64(w1).T.copy(), f64(w2).T.copy()   # oracle layout: W1 [D][F], W2 [F][D]
    y, h = oracle.ffn(f64(x), W1, f64(b1), W2, f64(b2), hidden=True)
    sigma = 2.0 ** -8 / math.sqrt(3.0) * np.sqrt((h * h) @ (W2 * W2))
    return y, bf16_half_ulp(y) + 6.0 * sigma + 1e-4


def check_ffn(got, want, bound):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - want)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"error {err[worst]:.3e} above its bound {bound[worst]:.3e} at {worst}; "
                                  f"max-abs {err.max():.3e}")
    assert err.mean() <= 0.25 * bound.mean(), f"mean-abs {err.mean():.3e}, mean bound {bound.mean():.3e}"
