"""The online softmax's rescale of the running output, on the GPU.

With N(0,1) inputs a row's maximum rarely grows by more than the kernel's
threshold (8 in log2 units) after the first key tile, so the step that
rescales the accumulated O (and l) to a new maximum would go unexercised.
Here the key rows of tile t are scaled by 1 + 2t and the queries by 2: in
ring order with one chunk the tiles are visited by position, and each
row's maximum grows by well over the threshold from tile to tile (checked
on the CPU from fp64 scores before the GPU runs).  The fused forward at
d = 64 and 128, causal and not, with grouped queries and a ragged length,
and the accumulating ring step (whose first tile rescales the running
result read from memory) must still equal the fp64 oracle within the
parity bounds (o: bf16 outputs, lse: 1e-3).  The section this follows:
"Large-scale distributed AI model training series: sequence parallelism",
6.2 Ring Attention (the blockwise online-softmax correction).
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs
from tolerance import TOL_LSE, check_bf16, check_fp32

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
THRESHOLD = 8.0  # log2 units


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


def f64(t):
    return t.detach().float().cpu().double().numpy()


def growing_inputs(B, Hq, Hkv, L, d, seed):
    """q scaled by 2, key rows of 128-row tile t by 1 + 2t (bf16)."""
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=seed, with_grad=False)
    tile = torch.arange(L) // 128
    k = (k.float() * (1.0 + 2.0 * tile.float())[None, None, :, None]).to(torch.bfloat16)
    q = (q.float() * 2.0).to(torch.bfloat16)
    return q, k, v


def rescaling_rows(q, k, causal, head=0):
    """Fraction of head `head`'s rows whose maximum (log2 units) grows by more
    than the threshold at some key tile after the first, in position order."""
    d = q.shape[-1]
    G = q.shape[1] // k.shape[1]
    s = (q[0, head].double() @ k[0, head // G].double().T).numpy() / np.sqrt(d) * LOG2E
    L = s.shape[0]
    if causal:
        s = np.where(np.tril(np.ones((L, L), dtype=bool)), s, -np.inf)
    n_t = (L + 127) // 128
    tile_max = np.stack([s[:, 128 * t:128 * (t + 1)].max(axis=1) for t in range(n_t)], axis=1)
    run = np.maximum.accumulate(tile_max, axis=1)
    grows = (tile_max[:, 1:] > run[:, :-1] + THRESHOLD) & np.isfinite(run[:, :-1])
    return grows.any(axis=1).mean()


# (B, Hq, Hkv, L, d, causal)
CASES = [(1, 2, 1, 1024, 64, False), (1, 2, 1, 1024, 64, True), (1, 2, 1, 1024, 128, False),
         (1, 4, 2, 1024, 128, True), (2, 2, 1, 1000, 64, False), (1, 2, 2, 1000, 128, False)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}L{}d{}".format(*c[:5]) + ("c" if c[5] else "e"))
def test_fused_forward_rescales_a_growing_maximum(case):
    B, Hq, Hkv, L, d, causal = case
    q, k, v = growing_inputs(B, Hq, Hkv, L, d, seed=500 + L + d)
    frac = rescaling_rows(q, k, causal)
    assert frac > 0.5, f"only {frac:.2f} of the rows cross the rescale threshold"
    o, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), 1, causal)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), causal)
    check_bf16("o", f64(o), o_ref)
    check_fp32("lse", f64(lse), lse_ref, TOL_LSE)


@pytest.mark.parametrize("d", [64, 128])
def test_accumulating_step_rescales_the_running_result(d):
    """Two chunks, non-causal: rank 0 accumulates its own chunk, then rank
    1's, whose keys are far larger, so the step starts by rescaling the
    running result it read (rank 1 visits them the other way round)."""
    B, Hq, Hkv, L, N = 1, 2, 1, 1024, 2
    q, k, v = growing_inputs(B, Hq, Hkv, L, d, seed=600 + d)
    C = L // N
    # rank 0's rows: chunk 1's first key tile against the maximum over chunk 0
    s = (q[0, 0].double() @ k[0, 0].double().T).numpy() / np.sqrt(d) * LOG2E
    frac = (s[:C, C:C + 128].max(axis=1) > s[:C, :C].max(axis=1) + THRESHOLD).mean()
    assert frac > 0.3, f"only {frac:.2f} of rank 0's rows rescale the running result"
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), False)
    for r in range(N):
        rows = torch.arange(r * C, (r + 1) * C)
        o_run = torch.zeros((B, Hq, C, d), dtype=torch.float32, device="cuda")
        lse_run = torch.full((B, Hq, C), float("-inf"), dtype=torch.float32, device="cuda")
        for src in oracle.ring_sources(r, N):
            srows = torch.arange(src * C, (src + 1) * C).cuda()
            ra.ring_attn_fwd_step_accumulate(qd[:, :, rows.cuda()].contiguous(), kd[:, :, srows].contiguous(),
                                             vd[:, :, srows].contiguous(), o_run, lse_run, N, False, r, src,
                                             schedule="fold")
        torch.cuda.synchronize()
        assert ra.device_status()[0] == 0
        idx = rows.numpy()
        check_bf16(f"o_run r{r}", f64(o_run), o_ref[:, :, idx])
        check_fp32(f"lse_run r{r}", f64(lse_run), lse_ref[:, :, idx], TOL_LSE)
