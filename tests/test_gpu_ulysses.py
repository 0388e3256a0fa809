"""Ulysses sequence parallelism on one GPU, through the C ABI, against the
fp64 oracle and the fused kernels.

Every tensor goes in and out as sequence shards stacked rank-major,
[N][B][H][L/N][d]; the library moves them to head shards and back (the two
all-to-alls of the pages' DeepSpeed-Ulysses section) around the fused
attention.  Attention is exact, so the result is the plain definition:
o, dq, dk, dv within 2e-2 max-abs beyond bf16 rounding and 2e-3 mean-abs,
lse within 1e-3 (tolerance.py).
"""
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs
from tolerance import TOL_LSE, check_bf16, check_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


def f64(t):
    return t.detach().float().cpu().double().numpy()


def to_shards(x, N):
    """[B, H, L, ...] in sequence order -> [N, B, H, L/N, ...] rank-major."""
    B, H, L = x.shape[:3]
    return x.reshape(B, H, N, L // N, *x.shape[3:]).movedim(2, 0).contiguous()


def from_shards(x):
    N, B, H, C = x.shape[:4]
    return x.movedim(0, 2).reshape(B, H, N * C, *x.shape[4:])


# (B, Hq, Hkv, L, d, N, causal)
CASES = [
    (1, 4, 2, 512, 128, 2, True),
    (2, 4, 4, 256, 64, 4, False),
    (1, 8, 4, 1024, 128, 4, True),
    (1, 28, 4, 2048, 128, 4, True),   # the GQA heads of the benchmark, Ulysses degree 4
    (1, 2, 2, 384, 64, 2, True),      # tokens per shard not a multiple of the tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}L{}d{}N{}{}".format(*c[:6], "c" if c[6] else "e"))
def test_ulysses_forward_and_backward_match_the_oracle(case):
    B, Hq, Hkv, L, d, N, causal = case
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=31 + sum(case[:6]))
    qs, ks, vs, dOs = (to_shards(x.cuda(), N) for x in (q, k, v, dO))
    o, lse = ra.ring_attn_ulysses_fwd(qs, ks, vs, causal)
    dq, dk, dv = ra.ring_attn_ulysses_bwd(qs, ks, vs, o, lse, dOs, causal)
    torch.cuda.synchronize()
    st, site = ra.device_status()
    assert st == 0, f"device status {st} at site {site:#x}"
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), causal)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(q.double(), k.double(), v.double(), dO.double(), causal)
    check_bf16("o", f64(from_shards(o)), o_ref)
    check_fp32("lse", f64(from_shards(lse)), lse_ref, TOL_LSE)
    check_bf16("dq", f64(from_shards(dq)), dq_ref)
    check_bf16("dk", f64(from_shards(dk)), dk_ref)
    check_bf16("dv", f64(from_shards(dv)), dv_ref)


def test_ulysses_equals_the_fused_kernel():
    """Same attention, other layout: the head-shard problem is the fused
    kernel with batch N*B; the result agrees with the fused kernel on the
    whole tensors."""
    B, Hq, Hkv, L, d, N = 2, 8, 4, 1024, 128, 4
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=99)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_f, lse_f = ra.ring_attn_fwd(qd, kd, vd, 1, True)
    o, lse = ra.ring_attn_ulysses_fwd(to_shards(qd, N), to_shards(kd, N), to_shards(vd, N), True)
    torch.cuda.synchronize()
    # one chunk on both sides: the same kernel, plan and summation order per (b, h)
    assert torch.equal(from_shards(o), o_f)
    assert torch.equal(from_shards(lse), lse_f)
