"""Blockwise feed-forward (BPT) on the GB300 through the C ABI, against the
fp64 oracle, within the per-element bound of ffn_tolerance.py (output
rounding plus the bf16 rounding of the hidden activation carried through
the second layer).
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from ffn_tolerance import check_ffn as check
from ffn_tolerance import f64
from ffn_tolerance import ffn_reference
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs
from tolerance import bf16_half_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


def reference(x, w1, b1, w2, b2, rows=None):
    return ffn_reference(x if rows is None else x[torch.as_tensor(rows)], w1, b1, w2, b2)


# (M, D, F, block_rows): ragged row counts, several blocks, several column
# tiles of both GEMMs, block_rows larger than M
CASES = [
    (128, 256, 1024, 128),
    (300, 256, 1024, 128),
    (1000, 512, 2048, 384),
    (77, 768, 512, 256),
    (640, 256, 2816, 640),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M{}D{}F{}R{}".format(*c))
def test_ffn_matches_the_oracle(case):
    M, D, F, R = case
    x, w1, b1, w2, b2 = inputs.make_ffn_inputs(M, D, F, seed=40 + M + D)
    y = ra.ring_attn_ffn_fwd(*(t.cuda() for t in (x, w1, b1, w2, b2)), block_rows=R)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    want, bound = reference(x, w1, b1, w2, b2)
    check(f64(y), want, bound)


def test_ffn_block_size_does_not_change_the_result():
    """Rows are independent and each output tile sums K in the same order
    whatever the block, so every block size gives the same bits."""
    M, D, F = 1000, 512, 1536
    dev = [t.cuda() for t in inputs.make_ffn_inputs(M, D, F, seed=7)]
    ys = [ra.ring_attn_ffn_fwd(*dev, block_rows=R) for R in (128, 256, 384, 1024, 4096)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


@pytest.mark.parametrize("R", [128, 256, 384])
def test_ffn_in_place(R):
    """y = x: a block's output rows replace its input rows only after the
    block has read them, and no launch touches rows of another block (with
    256-row tile pairs, blocks of 128 or 384 rows end inside a tile)."""
    M, D, F = 700, 256, 1024
    x, w1, b1, w2, b2 = inputs.make_ffn_inputs(M, D, F, seed=8)
    dev = [t.cuda() for t in (x, w1, b1, w2, b2)]
    y = ra.ring_attn_ffn_fwd(*dev, block_rows=R)
    xin = dev[0].clone()
    out = ra.ring_attn_ffn_fwd(xin, *dev[1:], block_rows=R, y=xin)
    assert out.data_ptr() == xin.data_ptr()
    assert torch.equal(xin, y)


def test_ffn_zero_second_layer_is_residual_plus_bias():
    """W2 = 0: y = bf16(x + b2) exactly (one rounding of an exact sum)."""
    M, D, F = 260, 256, 512
    x, w1, b1, w2, b2 = inputs.make_ffn_inputs(M, D, F, seed=9)
    y = ra.ring_attn_ffn_fwd(x.cuda(), w1.cuda(), b1.cuda(), torch.zeros_like(w2).cuda(), b2.cuda(), block_rows=128)
    want = (x.double() + b2.double()).float().to(torch.bfloat16)
    assert torch.equal(y.cpu(), want)


def test_ffn_full_size_sampled_rows():
    """The benchmark's workload (M = 131072 rows, D = 3584, F = 14336, blocks
    of 8192 rows) in the launch configuration the benchmark times; rows at
    block and tile edges plus random rows against the oracle."""
    w = inputs.FFN_WORKLOADS["ffn_gqa_128k"]
    x, w1, b1, w2, b2 = inputs.make_ffn_inputs(w.M, w.D, w.F, inputs.FFN_SEEDS[w.name])
    y = ra.ring_attn_ffn_fwd(*(t.cuda() for t in (x, w1, b1, w2, b2)), block_rows=w.block_rows)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    rows = inputs.ffn_sample_rows(w.M, w.block_rows, 96, seed=1)
    want, bound = reference(x, w1, b1, w2, b2, rows=rows)
    check(f64(y[torch.as_tensor(rows).cuda()]), want, bound)


def test_ffn_hidden_activation_keeps_relative_accuracy_in_the_gelu_tail():
    """gelu(a) = a Phi(a) per element, over a in [-9.5, 9.5], against the
    fp64 oracle within half a bf16 ulp plus 3e-5 relative (the fp32 rounding
    of a and of the exponentials): the tail a << 0, where Phi(a) falls to
    1e-19, must keep its relative accuracy (1 + erf(a / sqrt 2) cancels to 0
    in fp32 below a = -5.4).  Each row of x has one nonzero entry, so every
    first-layer sum is one exact bf16 product and a = fp32(product + b1);
    b1 sweeps the range.  On return the workspace holds the last block's h."""
    M, D, F = 256, 256, 1024
    g = torch.Generator().manual_seed(11)
    x = torch.zeros((M, D))
    x[torch.arange(M), torch.arange(M) % D] = (torch.rand(M, generator=g) - 0.5).to(torch.bfloat16).float()
    x = x.to(torch.bfloat16)
    w1 = (torch.rand((F, D), generator=g) - 0.5).to(torch.bfloat16)
    b1 = torch.linspace(-9.0, 9.0, F, dtype=torch.float32)
    w2 = torch.zeros((D, F), dtype=torch.bfloat16)
    b2 = torch.zeros(D, dtype=torch.float32)
    ws = torch.zeros(ra.ffn_workspace_size(D, F, M), dtype=torch.uint8, device="cuda")
    ra.ring_attn_ffn_fwd(*(t.cuda() for t in (x, w1, b1, w2, b2)), block_rows=M, workspace=ws)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    h = f64(ws[:M * F * 2].view(torch.bfloat16).view(M, F))
    _, want = oracle.ffn(f64(x), f64(w1).T.copy(), f64(b1), f64(w2).T.copy(), f64(b2), hidden=True)
    assert np.any((want < 0) & (want > -1e-17)) and want.max() > 9.0   # the range is covered, tail included
    bound = bf16_half_ulp(np.maximum(np.abs(want), np.abs(h))) + 3e-5 * np.abs(want)
    err = np.abs(h - want)
    worst = np.unravel_index(np.argmax(err / np.maximum(bound, 1e-300)), err.shape)
    assert np.all(err <= bound), f"h at {worst}: {h[worst]:.6e} against {want[worst]:.6e}"
