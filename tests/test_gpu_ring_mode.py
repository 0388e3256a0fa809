"""Ring mode on the GPU, through the C ABI, against the fp64 oracle.

One ring step (ring_attn_fwd_step) is compared with the oracle's ring_step
for every (rank, source) pair of small rings, for each chunk map (the fold,
stripes, contiguous causal chunks); the whole ring in each schedule,
including DistFlashAttention's balanced one; the merge kernel with the
oracle's merge; the whole ring run step by step on one GPU
(ring_attn_ring_fwd) with the oracle's plain forward and with the fused
forward.  Tolerances as for the fused path (tolerance.py): o within 2e-2
max-abs beyond bf16 output rounding and 2e-3 mean-abs, lse within 1e-3;
the merge alone, fp32 in and out, within 1e-5.  The accumulating step
(ring_attn_fwd_step_accumulate) against the oracle and against a step
followed by a merge.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


def f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_status_ok():
    st, site = ra.device_status()
    assert st == 0, f"device status {st} at site {site:#x}"


def chunk_positions(L, N, causal, r, schedule="fold"):
    return torch.tensor([p for p in range(L) if oracle.owner_rank(L, N, causal, p, schedule=schedule) == r],
                        dtype=torch.long)


def case_id(c):
    return "B{}Hq{}Hkv{}L{}d{}N{}".format(*c[:6]) + ("c" if c[6] else "e") + "-" + c[7]


# (B, Hq, Hkv, L, d, N, causal, schedule): chunks of whole 128-row tiles
STEP_CASES = [
    (1, 4, 2, 1024, 128, 4, True, "fold"),    # sub-chunks of one tile: every block spans both
    (2, 2, 1, 1024, 64, 4, False, "fold"),
    (1, 2, 2, 1536, 128, 3, True, "fold"),    # sub-chunks of two tiles
    (1, 2, 1, 768, 64, 3, False, "fold"),
    (1, 3, 1, 3072, 128, 4, True, "fold"),    # sub-chunks of three tiles: a block straddles them
    (1, 4, 2, 1024, 128, 4, True, "striped"),  # stripes: every step the same tile triangle
    (1, 2, 1, 1536, 64, 3, True, "striped"),
    (1, 3, 1, 1280, 128, 5, True, "striped"),  # L % 2N != 0: stripes only
    (1, 2, 2, 1024, 64, 8, False, "striped"),
    (1, 4, 2, 1024, 128, 4, True, "contiguous"),  # contiguous causal chunks: blocks below, on, above the diagonal
    (1, 2, 1, 1280, 64, 5, True, "dfa"),          # the same blocks, DistFlashAttention's chunk map
]


@pytest.mark.parametrize("case", STEP_CASES, ids=case_id)
def test_every_step_of_a_small_ring_matches_the_oracle(case):
    B, Hq, Hkv, L, d, N, causal, schedule = case
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=sum(case[:6]))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for r in range(N):
        rows = chunk_positions(L, N, causal, r, schedule)
        q_chunk = qd[:, :, rows.cuda()].contiguous()
        for src in range(N):
            srows = chunk_positions(L, N, causal, src, schedule)
            k_chunk = kd[:, :, srows.cuda()].contiguous()
            v_chunk = vd[:, :, srows.cuda()].contiguous()
            o_s, lse_s = ra.ring_attn_fwd_step(q_chunk, k_chunk, v_chunk, N, causal, r, src, schedule=schedule)
            torch.cuda.synchronize()
            assert_status_ok()
            o_ref, lse_ref = oracle.ring_step(q.double(), k.double(), v.double(), causal, N, r, src,
                                              schedule=schedule)
            o_ref, lse_ref = o_ref[:, :, rows.numpy()], lse_ref[:, :, rows.numpy()]
            got_o, got_l = f64(o_s), f64(lse_s)
            empty = np.isneginf(lse_ref)
            assert np.array_equal(np.isneginf(got_l), empty), f"rank {r} src {src}: rows with no visible key differ"
            assert np.all(got_o[empty] == 0.0)
            if (~empty).any():
                check_bf16(f"o_s r{r} s{src}", got_o[~empty], o_ref[~empty])
                check_fp32(f"lse_s r{r} s{src}", got_l[~empty], lse_ref[~empty], TOL_LSE)


@pytest.mark.parametrize("case", STEP_CASES, ids=case_id)
def test_step_accumulate_matches_the_oracle_and_step_then_merge(case):
    """Every rank runs its blocks in ring order accumulating into a running
    result that starts empty (lse = -inf); the result equals the plain
    definition on the rank's rows, and the partial-result path (step, then
    merge).  The two GPU paths round P to bf16 relative to different maxima
    (the running one, the block's own), so they agree within the parity
    bound, not to fp32 rounding."""
    B, Hq, Hkv, L, d, N, causal, schedule = case
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=3 + sum(case[:6]))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), causal)
    C = L // N
    for r in range(N):
        rows = chunk_positions(L, N, causal, r, schedule)
        q_chunk = qd[:, :, rows.cuda()].contiguous()
        o_run = torch.zeros((B, Hq, C, d), dtype=torch.float32, device="cuda")
        lse_run = torch.full((B, Hq, C), float("-inf"), dtype=torch.float32, device="cuda")
        o_m, lse_m = o_run.clone(), lse_run.clone()
        for src in oracle.ring_sources(r, N):
            srows = chunk_positions(L, N, causal, src, schedule).cuda()
            k_chunk, v_chunk = kd[:, :, srows].contiguous(), vd[:, :, srows].contiguous()
            ra.ring_attn_fwd_step_accumulate(q_chunk, k_chunk, v_chunk, o_run, lse_run, N, causal, r, src,
                                             schedule=schedule)
            o_s, lse_s = ra.ring_attn_fwd_step(q_chunk, k_chunk, v_chunk, N, causal, r, src, schedule=schedule)
            ra.ring_attn_merge(o_m, lse_m, o_s, lse_s)
        torch.cuda.synchronize()
        assert_status_ok()
        idx = rows.numpy()
        check_bf16(f"o_run r{r}", f64(o_run), o_ref[:, :, idx])
        check_fp32(f"lse_run r{r}", f64(lse_run), lse_ref[:, :, idx], TOL_LSE)
        check_bf16(f"o_run vs step+merge r{r}", f64(o_run), f64(o_m), ulps=0)
        check_fp32(f"lse_run vs step+merge r{r}", f64(lse_run), f64(lse_m), 1e-4)


def test_step_accumulate_keeps_rows_that_see_nothing():
    """Causal, the fold: rank 0's first sub-chunk sees none of rank 1's keys,
    so accumulating that block leaves those rows' running result as it was
    (o bit for bit; lse up to the rounding of its trip through log2 units),
    while the second sub-chunk's rows change."""
    B, Hq, Hkv, L, d, N = 1, 2, 1, 1024, 128, 4
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=71)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rows0 = chunk_positions(L, N, True, 0).cuda()
    rows1 = chunk_positions(L, N, True, 1).cuda()
    q_chunk = qd[:, :, rows0].contiguous()
    C, c = L // N, L // (2 * N)
    gen = torch.Generator(device="cpu").manual_seed(5)
    o_run = torch.randn((B, Hq, C, d), generator=gen).cuda()
    lse_run = torch.randn((B, Hq, C), generator=gen).cuda()
    o0, l0 = o_run.clone(), lse_run.clone()
    ra.ring_attn_fwd_step_accumulate(q_chunk, kd[:, :, rows1].contiguous(), vd[:, :, rows1].contiguous(), o_run,
                                     lse_run, N, True, 0, 1)
    torch.cuda.synchronize()
    assert_status_ok()
    assert torch.equal(o_run[:, :, :c], o0[:, :, :c])
    assert (lse_run[:, :, :c] - l0[:, :, :c]).abs().max().item() <= 2e-6 * max(1.0, l0.abs().max().item())
    assert not torch.equal(lse_run[:, :, c:], l0[:, :, c:])


@pytest.mark.parametrize("d", [64, 128])
def test_merge_matches_the_oracle(d):
    rng = np.random.default_rng(d)
    rows = 3000
    o_a, o_b = rng.standard_normal((rows, d)), rng.standard_normal((rows, d))
    l_a, l_b = rng.standard_normal(rows) * 4, rng.standard_normal(rows) * 4
    l_a[::7] = -np.inf      # side a empty
    l_b[::5] = -np.inf      # side b empty (both, every 35th row)
    l_b[1::11] = l_a[1::11] + 60.0   # one side dominates
    ta = torch.tensor(o_a, dtype=torch.float32)
    tb = torch.tensor(o_b, dtype=torch.float32)
    tla = torch.tensor(l_a, dtype=torch.float32)
    tlb = torch.tensor(l_b, dtype=torch.float32)
    o, lse = ta.cuda(), tla.cuda()
    o_out = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    ra.ring_attn_merge(o, lse, tb.cuda(), tlb.cuda(), o_out=o_out)
    torch.cuda.synchronize()
    want_o, want_l = oracle.merge(ta.double().numpy(), tla.double().numpy(), tb.double().numpy(),
                                  tlb.double().numpy())
    got_o, got_l = f64(o), f64(lse)
    np.testing.assert_array_equal(np.isneginf(got_l), np.isneginf(want_l))
    fin = np.isfinite(want_l)
    assert np.abs(got_l[fin] - want_l[fin]).max() <= 1e-5
    assert np.abs(got_o - want_o).max() <= 1e-5
    assert torch.equal(o_out.cpu(), o.cpu().to(torch.bfloat16))


# (B, Hq, Hkv, L, d, N, causal, schedule)
RING_CASES = [
    (1, 4, 2, 1024, 128, 4, True, "fold"),
    (2, 2, 1, 1024, 64, 4, False, "fold"),
    (1, 3, 1, 3072, 128, 4, True, "fold"),
    (1, 4, 4, 4096, 64, 8, False, "fold"),
    (1, 2, 2, 1024, 128, 1, True, "fold"),   # one rank: a single step, nothing to merge
    (1, 4, 2, 1024, 128, 4, True, "striped"),
    (1, 2, 1, 1280, 128, 5, True, "striped"),
    (1, 4, 2, 1024, 128, 4, True, "contiguous"),  # the unbalanced ring
    (1, 4, 2, 1024, 128, 4, True, "dfa"),   # 3 launches, the last with workers 0, 1 idle
    (1, 3, 1, 1280, 128, 5, True, "dfa"),   # odd N: 3 launches, all workers busy
    (2, 2, 2, 2048, 64, 8, True, "dfa"),    # the pages' example: 8 workers, 5 launches
    (1, 2, 1, 256, 128, 2, True, "dfa"),    # 2 launches, the second half idle
    (1, 2, 2, 1024, 64, 1, True, "dfa"),    # one worker
]


def _fused_chunks(L, N):
    return N if L % (2 * N) == 0 else 1  # the fused kernels' fold needs L % 2N


@pytest.mark.parametrize("case", RING_CASES, ids=case_id)
def test_whole_ring_on_one_gpu_matches_the_oracle_and_the_fused_kernel(case):
    B, Hq, Hkv, L, d, N, causal, schedule = case
    q, k, v, _ = inputs.make_inputs(B, Hq, Hkv, L, d, seed=7 + sum(case[:6]))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = ra.ring_attn_ring_fwd(qd, kd, vd, N, causal, schedule=schedule)
    o_f, lse_f = ra.ring_attn_fwd(qd, kd, vd, _fused_chunks(L, N), causal)
    torch.cuda.synchronize()
    assert_status_ok()
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), causal)
    check_bf16("o (ring mode)", f64(o), o_ref)
    check_fp32("lse (ring mode)", f64(lse), lse_ref, TOL_LSE)
    check_bf16("o (ring mode vs fused)", f64(o), f64(o_f), ulps=2)
    check_fp32("lse (ring mode vs fused)", f64(lse), f64(lse_f), TOL_LSE)


@pytest.mark.parametrize("schedule", ["fold", "striped", "dfa"])
def test_ring_mode_at_32k_on_sampled_rows(schedule):
    w = inputs.WORKLOADS["gqa_32k"]
    q, k, v, _ = inputs.workload_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = ra.ring_attn_ring_fwd(qd, kd, vd, w.n_chunks, w.causal, schedule=schedule)
    torch.cuda.synchronize()
    assert_status_ok()
    rows = inputs.sample_rows(w.L, w.n_chunks, w.causal, 64, seed=5)
    o_ref, lse_ref, _ = oracle.fwd_rows(q.double(), k.double(), v.double(), w.causal, rows)
    check_bf16("o (ring mode, 32k)", f64(o[:, :, rows]), o_ref)
    check_fp32("lse (ring mode, 32k)", f64(lse[:, :, rows]), lse_ref, TOL_LSE)


@pytest.mark.parametrize("case", RING_CASES, ids=case_id)
def test_ring_backward_matches_the_oracle_and_the_fused_kernel(case):
    B, Hq, Hkv, L, d, N, causal, schedule = case
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=13 + sum(case[:6]))
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = ra.ring_attn_fwd(qd, kd, vd, 1, causal)
    dq, dk, dv = ra.ring_attn_ring_bwd(qd, kd, vd, o, lse, dOd, N, causal, schedule=schedule)
    dq_f, dk_f, dv_f = ra.ring_attn_bwd(qd, kd, vd, o, lse, dOd, 1, causal)
    torch.cuda.synchronize()
    assert_status_ok()
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(q.double(), k.double(), v.double(), dO.double(), causal)
    for name, got, want, fused in (("dq", dq, dq_ref, dq_f), ("dk", dk, dk_ref, dk_f), ("dv", dv, dv_ref, dv_f)):
        check_bf16(f"{name} (ring mode)", f64(got), want)
        check_bf16(f"{name} (ring mode vs fused)", f64(got), f64(fused), ulps=2)


@pytest.mark.parametrize("schedule", ["fold", "striped", "dfa"])
def test_ring_backward_at_32k_matches_the_fused_kernel(schedule):
    w = inputs.WORKLOADS["gqa_32k"]
    q, k, v, dO = (x.cuda() for x in inputs.workload_inputs(w))
    o, lse = ra.ring_attn_fwd(q, k, v, w.n_chunks, w.causal)
    got = ra.ring_attn_ring_bwd(q, k, v, o, lse, dO, w.n_chunks, w.causal, schedule=schedule)
    want = ra.ring_attn_bwd(q, k, v, o, lse, dO, w.n_chunks, w.causal)
    torch.cuda.synchronize()
    assert_status_ok()
    for name, g, f in zip(("dq", "dk", "dv"), got, want):
        check_bf16(f"{name} (ring mode vs fused, 32k)", f64(g), f64(f), ulps=2)
