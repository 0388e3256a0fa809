"""USP (Ulysses groups of U ranks and a ring across R groups) on one GPU,
through the C ABI, against the fp64 oracle and the fused kernels.

The N = U R sequence shards are built here from the definition ("Large-
scale distributed AI model training series: sequence parallelism", section
8.2; the rank layout of include/ring_attn.h): rank n = r U + u holds the
tokens of its ring group's part of the sequence, contiguous shards for the
encoder (or R = 1), and for the causal ring the fold: group r owns
sub-chunks r and 2R-1-r, rank u piece u of each.  Attention is exact, so
the result is the plain definition: o, dq, dk, dv within 2e-2 max-abs
beyond bf16 rounding and 2e-3 mean-abs, lse within 1e-3; the forward is
bit-equal to ring_attn_fwd with R ring chunks on the natural layout (the
same kernel and plan per (batch, head)).
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs
from tolerance import check_bf16, check_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


def f64(t):
    return t.detach().float().cpu().double().numpy()


def usp_positions(L, U, R, causal):
    """[N, C] sequence position of token i of rank n = r U + u."""
    N = U * R
    C = L // N
    pos = np.zeros((N, C), dtype=np.int64)
    for n in range(N):
        r, u = divmod(n, U)
        for i in range(C):
            if not causal or R == 1:
                pos[n, i] = n * C + i
            else:
                c = L // (2 * R)
                piece = c // U
                pos[n, i] = r * c + u * piece + i if i < piece else (2 * R - 1 - r) * c + u * piece + (i - piece)
    return pos


def to_shards(x, pos):
    """[B, H, L, ...] -> [N, B, H, C, ...]."""
    p = torch.as_tensor(pos, device=x.device)
    return x[:, :, p].movedim(2, 0).contiguous()


def from_shards(x, pos, L):
    """[N, B, H, C, ...] -> [B, H, L, ...]."""
    N, B, H, C = x.shape[:4]
    out = torch.empty((B, H, L, *x.shape[4:]), dtype=x.dtype, device=x.device)
    out[:, :, torch.as_tensor(pos, device=x.device)] = x.movedim(0, 2)
    return out


def test_positions_cover_the_sequence():
    for L, U, R, causal in ((1024, 2, 2, True), (96, 3, 2, True), (60, 2, 3, False), (64, 4, 1, True)):
        pos = usp_positions(L, U, R, causal)
        assert sorted(pos.ravel().tolist()) == list(range(L))


# (B, Hq, Hkv, L, d, U, R, causal)
CASES = [
    (1, 4, 2, 1024, 128, 2, 2, True),
    (2, 4, 4, 512, 64, 2, 2, False),
    (1, 8, 4, 2048, 128, 4, 2, True),
    (1, 2, 2, 1024, 64, 1, 4, True),    # a pure ring through the USP layout
    (1, 28, 4, 4096, 128, 4, 4, True),  # the GQA heads: Ulysses degree 4, ring of 4
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}L{}d{}U{}R{}{}".format(*c[:7], "c" if c[7] else "e"))
def test_usp_forward_and_backward_match_the_oracle(case):
    B, Hq, Hkv, L, d, U, R, causal = case
    pos = usp_positions(L, U, R, causal)
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=71 + sum(case[:7]))
    qs, ks, vs, dOs = (to_shards(x.cuda(), pos) for x in (q, k, v, dO))
    o, lse = ra.ring_attn_usp_fwd(qs, ks, vs, U, causal)
    dq, dk, dv = ra.ring_attn_usp_bwd(qs, ks, vs, o, lse, dOs, U, causal)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    o_n, lse_n = from_shards(o, pos, L), from_shards(lse, pos, L)
    dq_n, dk_n, dv_n = (from_shards(x, pos, L) for x in (dq, dk, dv))

    o_ref, lse_ref = oracle.fwd(f64(q), f64(k), f64(v), causal)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(f64(q), f64(k), f64(v), f64(dO), causal)
    check_bf16("o", f64(o_n), o_ref)
    check_fp32("lse", f64(lse_n), lse_ref)
    check_bf16("dq", f64(dq_n), dq_ref)
    check_bf16("dk", f64(dk_n), dk_ref)
    check_bf16("dv", f64(dv_n), dv_ref)

    o_f, lse_f = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), R, causal)
    assert torch.equal(o_n, o_f) and torch.equal(lse_n, lse_f)


# (B, Hq, Hkv, L, d, U, R, causal): the benchmark's GQA heads at 32k, and
# 64 x 64 heads of 256 tokens over 16 Ulysses ranks -- 65,536 (rank, batch,
# head) slices, more than one grid dimension holds, so the all-to-all's
# launch takes its third dimension
SCALE_CASES = [(1, 28, 4, 32768, 128, 4, 4, True), (64, 64, 16, 256, 64, 16, 1, False)]


@pytest.mark.parametrize("case", SCALE_CASES,
                         ids=lambda c: "B{}Hq{}Hkv{}L{}d{}U{}R{}{}".format(*c[:7], "c" if c[7] else "e"))
def test_usp_at_scale_equals_the_fused_kernels(case):
    """At sizes the oracle cannot take whole: the USP forward is bit-equal to
    the fused forward with R ring chunks (the same kernel and plan per
    (batch, head) once the all-to-all has permuted the shards), and the
    backward equals the fused backward up to the order of its fp32
    reduce-adds (dq; and dk, dv with grouped queries): within one bf16
    step of the value, plus 1e-4 for the reordered fp32 sums of values near
    zero (the oracle's bound is 2e-2)."""
    B, Hq, Hkv, L, d, U, R, causal = case
    pos = usp_positions(L, U, R, causal)
    q, k, v, dO = (x.cuda() for x in inputs.make_inputs(B, Hq, Hkv, L, d, seed=170 + sum(case[:7])))
    qs, ks, vs, dOs = (to_shards(x, pos) for x in (q, k, v, dO))
    o, lse = ra.ring_attn_usp_fwd(qs, ks, vs, U, causal)
    dq, dk, dv = ra.ring_attn_usp_bwd(qs, ks, vs, o, lse, dOs, U, causal)
    o_f, lse_f = ra.ring_attn_fwd(q, k, v, R, causal)
    dq_f, dk_f, dv_f = ra.ring_attn_bwd(q, k, v, o_f, lse_f, dO, R, causal)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    assert torch.equal(from_shards(o, pos, L), o_f) and torch.equal(from_shards(lse, pos, L), lse_f)
    for name, got, ref in (("dq", dq, dq_f), ("dk", dk, dk_f), ("dv", dv, dv_f)):
        g, r = from_shards(got, pos, L).float(), ref.float()
        step = r.abs() * 2.0 ** -7 + 1e-4  # one bf16 step of the value, and fp32 order noise
        assert bool(((g - r).abs() <= step).all()), f"{name}: max diff {float((g - r).abs().max()):.3e}"
