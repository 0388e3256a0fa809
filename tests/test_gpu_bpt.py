"""The blockwise transformer forward (BPT: per query block, attention over
every key/value block, then the FFN and the residual) on the GB300 through
the C ABI.

The attention part (token-major output and lse) is checked against the
fp64 oracle's attention with the attention bounds of tolerance.py, and is
bit-identical to ring_attn_fwd's output (same kernel and work items).  The
FFN part is checked against the oracle's FFN applied to the GPU's own
attention output (the FFN's input as the GPU holds it), within the bound
of ffn_tolerance.py, and is bit-identical to ring_attn_ffn_fwd on that
input (same GEMMs over the same row blocks).
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from ffn_tolerance import check_ffn, f64, ffn_reference
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs
from tolerance import check_bf16, check_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


# (B, Hq, Hkv, L, d, N, causal, F, block_rows, ffn rows checked (0: all))
CASES = [
    (1, 2, 1, 1024, 128, 4, True, 1024, 256, 0),
    (2, 4, 2, 1000, 64, 4, True, 512, 512, 0),     # ragged L, two batches: stores stop at each batch's L
    (1, 4, 4, 768, 64, 2, False, 768, 256, 0),
    (1, 28, 4, 2048, 128, 4, True, 14336, 512, 64),  # the GQA heads (D = 3584, F = 4 D)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}L{}d{}N{}{}F{}R{}".format(
    *c[:6], "c" if c[6] else "e", c[7], c[8]))
def test_bpt_forward(case):
    B, Hq, Hkv, L, d, N, causal, F, R, n_rows = case
    D = Hq * d
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=60 + L + Hq, with_grad=False)
    _, w1, b1, w2, b2 = inputs.make_ffn_inputs(1, D, F, seed=61 + F)
    dev = [t.cuda() for t in (q, k, v, w1, b1, w2, b2)]
    a_tok, lse, y = ra.ring_attn_bpt_fwd(*dev[:3], *dev[3:], N, causal, block_rows=R)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0

    # attention: against the oracle, and bit-equal to the fused forward
    o_ref, lse_ref = oracle.fwd(f64(q), f64(k), f64(v), causal)
    check_bf16("a_tok", f64(a_tok), o_ref.transpose(0, 2, 1, 3).reshape(B, L, D))
    check_fp32("lse", f64(lse), lse_ref)
    o, lse2 = ra.ring_attn_fwd(*dev[:3], N, causal)
    assert torch.equal(a_tok, o.transpose(1, 2).reshape(B, L, D))
    assert torch.equal(lse, lse2)

    # feed-forward: on the GPU's attention output, against the oracle and
    # bit-equal to the blockwise FFN call on the same rows
    x = a_tok.reshape(B * L, D)
    y_ffn = torch.empty_like(x)
    for b in range(B):
        ra.ring_attn_ffn_fwd(x[b * L:(b + 1) * L], *dev[3:], block_rows=R, y=y_ffn[b * L:(b + 1) * L])
    assert torch.equal(y.reshape(B * L, D), y_ffn)
    rows = (torch.arange(B * L) if not n_rows else
            torch.as_tensor(inputs.ffn_sample_rows(B * L, R, n_rows, seed=2)))
    want, bound = ffn_reference(x[rows.cuda()], *dev[3:])
    check_ffn(f64(y.reshape(B * L, D)[rows.cuda()]), want, bound)


# (B, Hq, Hkv, L, d, N, causal, F, block_rows)
BWD_CASES = [
    (1, 2, 1, 1024, 128, 4, True, 1024, 256),
    (2, 4, 2, 1000, 64, 4, True, 512, 512),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "B{}Hq{}Hkv{}L{}d{}N{}{}F{}R{}".format(
    *c[:6], "c" if c[6] else "e", c[7], c[8]))
def test_bpt_backward(case):
    """The chain rule through y = a + FFN(a), a = attention(q, k, v): the
    attention gradients against the oracle's attention backward driven by
    the oracle's gradient at a (dy plus the FFN's input gradient, on the
    GPU's a); the FFN's weight gradients equal ring_attn_ffn_bwd on a."""
    B, Hq, Hkv, L, d, N, causal, F, R = case
    D = Hq * d
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=65 + L + Hq, with_grad=False)
    _, w1, b1, w2, b2 = inputs.make_ffn_inputs(1, D, F, seed=66 + F)
    dy = torch.randn((B, L, D), generator=torch.Generator().manual_seed(67)).to(torch.bfloat16)
    dev = [t.cuda() for t in (q, k, v, w1, b1, w2, b2)]
    a_tok, lse, _ = ra.ring_attn_bpt_fwd(*dev[:3], *dev[3:], N, causal, block_rows=R)
    dq, dk, dv, dw1, db1, dw2, db2 = ra.ring_attn_bpt_bwd(*dev[:3], a_tok, lse, dev[3], dev[4], dev[5],
                                                          dy.cuda(), N, causal, block_rows=R)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0

    # gradient at the attention output, by the oracle, from the GPU's a
    x = f64(a_tok).reshape(B * L, D)
    da = oracle.ffn_bwd(x, f64(w1).T.copy(), f64(b1), f64(w2).T.copy(), f64(dy).reshape(B * L, D))[0]
    dO = da.reshape(B, L, Hq, d).transpose(0, 2, 1, 3)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(f64(q), f64(k), f64(v), dO, causal)
    check_bf16("dq", f64(dq), dq_ref)
    check_bf16("dk", f64(dk), dk_ref)
    check_bf16("dv", f64(dv), dv_ref)

    # the FFN part is the blockwise FFN backward on the token rows
    fdx, fdw1, fdb1, fdw2, fdb2 = ra.ring_attn_ffn_bwd(a_tok.reshape(B * L, D), dev[3], dev[4], dev[5],
                                                       dy.cuda().reshape(B * L, D), block_rows=R)
    assert torch.equal(dw1, fdw1) and torch.equal(dw2, fdw2)
    torch.testing.assert_close(db1, fdb1, rtol=1e-5, atol=1e-4)   # column sums by fp32 atomics
    torch.testing.assert_close(db2, fdb2, rtol=1e-5, atol=1e-4)
