"""Backward of the blockwise feed-forward block on the GB300 through the C
ABI, against the fp64 oracle.

The GPU recomputes a = x W1^T + b1 in fp32 per block and rounds gelu'(a),
da = (dy W2) * gelu'(a) and h = gelu(a) to bf16 once each (they are GEMM
operands); the weight-gradient sums run in fp32.  Bound per element, from
those roundings (each at most half a bf16 ulp, 2^-8 relative, roughly
uniform and independent across the terms of a sum, so a sum of n such
terms errs with standard deviation 2^-8 / sqrt(3) * sqrt(k) * sqrt(sum of
the squared terms), k = roundings per term):
  dx  = dy + da W1       : k = 2 (gelu', da) over f, plus dx's own output
                           rounding (half a bf16 ulp)
  dW2 = sum_m dy h       : k = 1 (h) over rows
  dW1 = sum_m x da       : k = 2 over rows
  db1 = sum_m da         : k = 2 over rows
  db2 = sum_m dy         : exact inputs, fp32 sums
Six standard deviations plus 1e-4 (relative to each output's scale) for the
fp32 arithmetic are allowed; the mean error must stay within a quarter of
the mean bound.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from ffn_tolerance import f64
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs
from tolerance import bf16_half_ulp

pytestmark = pytest.mark.gpu
U = 2.0 ** -8 / math.sqrt(3.0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


def check(name, got, want, bound):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), name
    err = np.abs(got - want)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"{name}: error {err[worst]:.3e} above its bound {bound[worst]:.3e} at {worst}; "
                                  f"max-abs {err.max():.3e}")
    assert err.mean() <= 0.25 * bound.mean(), f"{name}: mean-abs {err.mean():.3e}, mean bound {bound.mean():.3e}"


# (M, D, F, block_rows): ragged last blocks (44 and 232 rows: K padded to 64)
CASES = [
    (300, 256, 512, 128),
    (512, 512, 1024, 256),
    (1000, 256, 768, 384),
    (2048, 1024, 4096, 1024),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M{}D{}F{}R{}".format(*c))
def test_ffn_backward_matches_the_oracle(case):
    M, D, F, R = case
    x, w1, b1, w2, b2 = inputs.make_ffn_inputs(M, D, F, seed=80 + M)
    g = torch.Generator().manual_seed(81 + M)
    dy = torch.randn((M, D), generator=g).to(torch.bfloat16)
    dx, dw1, db1, dw2, db2 = ra.ring_attn_ffn_bwd(*(t.cuda() for t in (x, w1, b1, w2, dy)), block_rows=R)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0

    W1, W2 = f64(w1).T.copy(), f64(w2).T.copy()          # oracle layout: W1 [D][F], W2 [F][D]
    X, DY = f64(x), f64(dy)
    rdx, rdw1, rdb1, rdw2, rdb2, h, da = oracle.ffn_bwd(X, W1, f64(b1), W2, DY, hidden=True)
    w1o = f64(w1)                                         # [F][D]
    check("dx", f64(dx), rdx, bf16_half_ulp(rdx) + 6 * U * math.sqrt(2) * np.sqrt((da * da) @ (w1o * w1o)) + 1e-4)
    # weight gradients in the library's layouts: dw1 [F][D] = W1 grad^T, dw2 [D][F]
    check("dw2", f64(dw2), rdw2.T, 6 * U * np.sqrt((DY * DY).T @ (h * h)) + 1e-4 * np.abs(rdw2).max())
    check("dw1", f64(dw1), rdw1.T, 6 * U * math.sqrt(2) * np.sqrt((da * da).T @ (X * X)) + 1e-4 * np.abs(rdw1).max())
    check("db1", f64(db1), rdb1, 6 * U * math.sqrt(2) * np.sqrt((da * da).sum(axis=0)) + 1e-4 * np.abs(rdb1).max())
    check("db2", f64(db2), rdb2, 1e-4 * max(1.0, np.abs(rdb2).max()) + np.zeros_like(rdb2))


def test_ffn_backward_zero_second_layer():
    """W2 = 0: dx = dy exactly (da = 0, one rounding of dy + 0), no gradient
    reaches W1 or b1."""
    M, D, F = 260, 256, 512
    x, w1, b1, w2, _ = inputs.make_ffn_inputs(M, D, F, seed=90)
    dy = torch.randn((M, D), generator=torch.Generator().manual_seed(91)).to(torch.bfloat16)
    dx, dw1, db1, dw2, db2 = ra.ring_attn_ffn_bwd(x.cuda(), w1.cuda(), b1.cuda(), torch.zeros_like(w2).cuda(),
                                                  dy.cuda(), block_rows=128)
    assert torch.equal(dx.cpu(), dy)
    assert not dw1.any() and not db1.any()


def test_ffn_backward_at_the_benchmark_width_sampled_rows():
    """The benchmark's FFN width (D = 3584, F = 14336, blocks of 8192 rows)
    over two blocks: dx on sampled rows (block and tile edges included)
    against the oracle, which a row's dx depends on alone, with the bound of
    the small cases; db2 against the fp64 column sums of dy over every row;
    the weight gradients finite."""
    wl = inputs.FFN_WORKLOADS["ffn_gqa_128k"]
    R, D, F = wl.block_rows, wl.D, wl.F
    M = 2 * R
    x, w1, b1, w2, _ = inputs.make_ffn_inputs(M, D, F, seed=95)
    dy = torch.randn((M, D), generator=torch.Generator().manual_seed(96)).to(torch.bfloat16)
    dx, dw1, db1, dw2, db2 = ra.ring_attn_ffn_bwd(*(t.cuda() for t in (x, w1, b1, w2, dy)), block_rows=R)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    for name, t in (("dw1", dw1), ("db1", db1), ("dw2", dw2)):
        assert torch.isfinite(t).all(), name

    rows = np.asarray(inputs.ffn_sample_rows(M, R, 40, seed=95))
    idx = torch.as_tensor(rows)
    W1, W2 = f64(w1).T.copy(), f64(w2).T.copy()
    rdx, _, _, _, _, _, da = oracle.ffn_bwd(f64(x[idx]), W1, f64(b1), W2, f64(dy[idx]), hidden=True)
    w1o = f64(w1)
    check("dx", f64(dx.cpu()[idx]), rdx,
          bf16_half_ulp(rdx) + 6 * U * math.sqrt(2) * np.sqrt((da * da) @ (w1o * w1o)) + 1e-4)
    rdb2 = f64(dy).sum(axis=0)
    check("db2", f64(db2), rdb2, 1e-4 * max(1.0, np.abs(rdb2).max()) + np.zeros_like(rdb2))
