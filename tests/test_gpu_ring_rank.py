"""The per-rank calls of a multi-GPU ring on the GPU, through the C ABI:
ring_attn_fwd_step_accumulate for the forward and ring_attn_bwd_rank_*
(with ring_attn_grad_to_bf16) for the backward.  One process plays every
rank of the ring in the order ring_dist runs them -- at step s rank r
holds the key/value chunk of rank (r - s) mod N and, in the backward, that
chunk's travelling fp32 dK/dV accumulators -- with no communication (this
pool gives one GPU per run; the exchange itself is tested over gloo ranks
on the CPU).  Every rank's o, lse, dq, dk, dv against the fp64 oracle on its
rows, with the parity bounds of tolerance.py.
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


def positions(L, N, causal, r, schedule):
    return torch.tensor([p for p in range(L) if oracle.owner_rank(L, N, causal, p, schedule=schedule) == r],
                        dtype=torch.long)


# (B, Hq, Hkv, L, d, N, causal, schedule): chunks of whole 128-row tiles
CASES = [
    (1, 4, 2, 1024, 128, 4, True, "fold"),
    (2, 2, 2, 768, 64, 3, False, "fold"),
    (1, 3, 1, 1536, 128, 3, True, "striped"),
    (1, 2, 1, 1024, 64, 4, True, "contiguous"),
    (1, 2, 2, 512, 128, 1, True, "fold"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}L{}d{}N{}".format(*c[:6]) +
                         ("c" if c[6] else "e") + "-" + c[7])
def test_every_rank_of_an_emulated_ring(case):
    B, Hq, Hkv, L, d, N, causal, schedule = case
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=90 + sum(case[:6]))
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    C = L // N
    pos = [positions(L, N, causal, r, schedule).cuda() for r in range(N)]
    ch = lambda x, r: x[:, :, pos[r]].contiguous()  # noqa: E731

    # forward: each rank accumulates its blocks in ring order
    o_run = [torch.zeros((B, Hq, C, d), dtype=torch.float32, device="cuda") for _ in range(N)]
    lse_run = [torch.full((B, Hq, C), float("-inf"), dtype=torch.float32, device="cuda") for _ in range(N)]
    for s in range(N):
        for r in range(N):
            src = (r - s) % N
            ra.ring_attn_fwd_step_accumulate(ch(qd, r), ch(kd, src), ch(vd, src), o_run[r], lse_run[r], N, causal, r,
                                             src, schedule=schedule)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), causal)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(q.double(), k.double(), v.double(), dO.double(), causal)
    for r in range(N):
        idx = pos[r].cpu().numpy()
        check_bf16(f"o rank {r}", f64(o_run[r]), o_ref[:, :, idx])
        check_fp32(f"lse rank {r}", f64(lse_run[r]), lse_ref[:, :, idx], TOL_LSE)

    # backward: dQ local; dK/dV accumulators travel with their chunk
    o = [x.to(torch.bfloat16) for x in o_run]
    ranks = [ra.RankBackward(o[r], ch(dOd, r), lse_run[r], Hkv, N, causal, schedule=schedule) for r in range(N)]
    dk_acc = [torch.zeros((B, Hkv, C, d), dtype=torch.float32, device="cuda") for _ in range(N)]
    dv_acc = [torch.zeros_like(a) for a in dk_acc]
    for s in range(N):
        for r in range(N):
            src = (r - s) % N
            ranks[r].step(ch(qd, r), ch(kd, src), ch(vd, src), dk_acc[src], dv_acc[src], r, src)
    dq = [ranks[r].end() for r in range(N)]
    dk = [ra.grad_to_bf16(dk_acc[r], 1.0 / d ** 0.5) for r in range(N)]
    dv = [ra.grad_to_bf16(dv_acc[r], 1.0) for r in range(N)]
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    for r in range(N):
        idx = pos[r].cpu().numpy()
        check_bf16(f"dq rank {r}", f64(dq[r]), dq_ref[:, :, idx])
        check_bf16(f"dk rank {r}", f64(dk[r]), dk_ref[:, :, idx])
        check_bf16(f"dv rank {r}", f64(dv[r]), dv_ref[:, :, idx])


# (B, Hq, Hkv, L, d, N): DistFlashAttention across N emulated ranks (causal,
# contiguous chunks of whole tiles); N = 3 and 5 pair every launch, 4 leaves
# the middle one unpaired
DFA_CASES = [(1, 4, 2, 1536, 128, 3), (1, 2, 1, 1024, 64, 4), (1, 2, 2, 1280, 128, 5)]


@pytest.mark.parametrize("case", DFA_CASES, ids=lambda c: "B{}Hq{}Hkv{}L{}d{}N{}".format(*c))
def test_distflash_protocol_of_an_emulated_ring(case):
    """Each rank's launches of DistFlashAttention's schedule in the order of
    ring_dist: its own block, or the block of a later rank's queries against
    its own keys (a partial result merged by ring_attn_merge at the owner;
    a fp32 dQ partial added by ring_attn_add_f32 into the owner's
    accumulator, dK/dV kept by the helper and added at the end)."""
    from sequence_blockwise_self_gb300.ring_dist import _dfa_roles
    B, Hq, Hkv, L, d, N = case
    schedule = "dfa"
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=130 + sum(case))
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    C = L // N
    pos = [positions(L, N, True, r, schedule).cuda() for r in range(N)]
    ch = lambda x, r: x[:, :, pos[r]].contiguous()  # noqa: E731

    o_run = [torch.zeros((B, Hq, C, d), dtype=torch.float32, device="cuda") for _ in range(N)]
    lse_run = [torch.full((B, Hq, C), float("-inf"), dtype=torch.float32, device="cuda") for _ in range(N)]
    for t in range(N // 2 + 1):
        for r in range(N):
            own, helper_of, _ = _dfa_roles(N, r, t)
            if own:
                ra.ring_attn_fwd_step_accumulate(ch(qd, r), ch(kd, r - t), ch(vd, r - t), o_run[r], lse_run[r], N,
                                                 True, r, r - t, schedule="contiguous")
            if helper_of is not None:
                o_p = torch.zeros_like(o_run[0])
                lse_p = torch.full_like(lse_run[0], float("-inf"))
                ra.ring_attn_fwd_step_accumulate(ch(qd, helper_of), ch(kd, r), ch(vd, r), o_p, lse_p, N, True,
                                                 helper_of, r, schedule="contiguous")
                ra.ring_attn_merge(o_run[helper_of], lse_run[helper_of], o_p, lse_p)
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), True)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(q.double(), k.double(), v.double(), dO.double(), True)
    for r in range(N):
        idx = pos[r].cpu().numpy()
        check_bf16(f"o rank {r}", f64(o_run[r]), o_ref[:, :, idx])
        check_fp32(f"lse rank {r}", f64(lse_run[r]), lse_ref[:, :, idx], TOL_LSE)

    o = [x.to(torch.bfloat16) for x in o_run]
    ranks = [ra.RankBackward(o[r], ch(dOd, r), lse_run[r], Hkv, N, True, schedule="contiguous") for r in range(N)]
    acc = [(torch.zeros((B, Hkv, C, d), dtype=torch.float32, device="cuda"),
            torch.zeros((B, Hkv, C, d), dtype=torch.float32, device="cuda")) for _ in range(N)]
    home = [(torch.zeros_like(a[0]), torch.zeros_like(a[1])) for a in acc]
    for t in range(N // 2 + 1):
        for r in range(N):
            own, helper_of, _ = _dfa_roles(N, r, t)
            if own:
                ranks[r].step(ch(qd, r), ch(kd, r - t), ch(vd, r - t), acc[r - t][0], acc[r - t][1], r, r - t)
            if helper_of is not None:
                a = helper_of
                helper = ra.RankBackward(o[a], ch(dOd, a), lse_run[a], Hkv, N, True, schedule="contiguous")
                helper.step(ch(qd, a), ch(kd, r), ch(vd, r), home[r][0], home[r][1], a, r)
                ranks[a].add_dq(helper.dq_accumulator())
    dq = [ranks[r].end() for r in range(N)]
    for r in range(N):
        ra.add_f32(acc[r][0], home[r][0])
        ra.add_f32(acc[r][1], home[r][1])
    dk = [ra.grad_to_bf16(acc[r][0], 1.0 / d ** 0.5) for r in range(N)]
    dv = [ra.grad_to_bf16(acc[r][1], 1.0) for r in range(N)]
    torch.cuda.synchronize()
    assert ra.device_status()[0] == 0
    for r in range(N):
        idx = pos[r].cpu().numpy()
        check_bf16(f"dq rank {r}", f64(dq[r]), dq_ref[:, :, idx])
        check_bf16(f"dk rank {r}", f64(dk[r]), dk_ref[:, :, idx])
        check_bf16(f"dv rank {r}", f64(dv[r]), dv_ref[:, :, idx])


def test_ring_driver_with_the_library_ops_on_one_rank():
    """ring_dist's driver with its default ops (the library's kernels) on a
    one-rank process group: DistFlashAttention's schedule at N = 1 needs no
    exchange, so the driver's CUDA path -- running result, block, end;
    rank backward, partial adds, conversion -- runs end to end on the GPU
    and must equal the fp64 oracle."""
    import os
    import socket

    import torch.distributed as dist

    from sequence_blockwise_self_gb300 import ring_dist

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        B, Hq, Hkv, L, d = 1, 4, 2, 512, 128
        q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=141)
        qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
        o, lse = ring_dist.ring_attention_fwd(qd, kd, vd, True, schedule="dfa")
        dq, dk, dv = ring_dist.ring_attention_bwd(qd, kd, vd, o, lse, dOd, True, schedule="dfa")
        torch.cuda.synchronize()
        assert ra.device_status()[0] == 0
    finally:
        dist.destroy_process_group()
    o_ref, lse_ref = oracle.fwd(q.double(), k.double(), v.double(), True)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(q.double(), k.double(), v.double(), dO.double(), True)
    check_bf16("o", f64(o), o_ref)
    check_fp32("lse", f64(lse), lse_ref, TOL_LSE)
    check_bf16("dq", f64(dq), dq_ref)
    check_bf16("dk", f64(dk), dk_ref)
    check_bf16("dv", f64(dv), dv_ref)
