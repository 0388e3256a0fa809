"""The multi-GPU ring driver (ring_dist) on CPU ranks: gloo, world sizes 2
to 4, one process per rank.  Each rank runs ring_attention_fwd and
ring_attention_bwd on its own chunk with the per-block arithmetic of the
fp64 oracle (test infrastructure): a received key/value chunk is placed at
its owner's positions of an otherwise zero sequence and the oracle's ring
step / block backward takes it from there, so a chunk that arrives at the
wrong rank or step, or a dK/dV accumulator that travels wrongly, changes
the result.  Every rank's o, lse, dq, dk, dv must equal the plain
definition on its rows ("Large-scale distributed AI model training series:
sequence parallelism", sections 2.3 and 6.2).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _positions(L, n, causal, rank, schedule):
    return np.array([p for p in range(L) if oracle.owner_rank(L, n, causal, p, schedule=schedule) == rank])


class OracleRingOps:
    """ring_dist's per-rank blocks in fp64 on the CPU, from the oracle."""

    acc_dtype = torch.float64

    def __init__(self, L, Hkv, causal, schedule, n):
        self.L, self.Hkv, self.causal, self.schedule, self.n = L, Hkv, causal, schedule, n

    def _embed(self, x, rank):
        B, H, C, d = x.shape
        full = np.zeros((B, H, self.L, d))
        full[:, :, _positions(self.L, self.n, self.causal, rank, self.schedule)] = x.numpy()
        return full

    def _rows(self, full, rank):
        return torch.from_numpy(np.ascontiguousarray(full[:, :, _positions(self.L, self.n, self.causal, rank,
                                                                            self.schedule)]))

    def fwd_begin(self, q):
        B, Hq, C, d = q.shape
        return torch.zeros((B, Hq, C, d), dtype=torch.float64), torch.full((B, Hq, C), float("-inf"),
                                                                           dtype=torch.float64)

    def fwd_block(self, q, k, v, o_run, lse_run, n, causal, rank, src, schedule):
        o_s, lse_s = oracle.ring_step(self._embed(q, rank), self._embed(k, src), self._embed(v, src), causal, n,
                                      rank, src, schedule=schedule)
        pos = _positions(self.L, n, causal, rank, schedule)
        o, lse = oracle.merge(o_run.numpy(), lse_run.numpy(), o_s[:, :, pos], lse_s[:, :, pos])
        o_run.copy_(torch.from_numpy(o))
        lse_run.copy_(torch.from_numpy(lse))

    def fwd_end(self, o_run, lse_run):
        return o_run, lse_run

    def bwd_begin(self, o, dO, lse, Hkv, n, causal, schedule):
        return {"o": o, "dO": dO, "lse": lse, "D": (dO * o).sum(-1), "dq": torch.zeros_like(o)}

    def bwd_block(self, state, q, k, v, dk_acc, dv_acc, rank, src):
        B, Hq, C, _ = q.shape
        lse = np.zeros((B, Hq, self.L))
        D = np.zeros((B, Hq, self.L))
        pos = _positions(self.L, self.n, self.causal, rank, self.schedule)
        lse[:, :, pos] = state["lse"].numpy()
        D[:, :, pos] = state["D"].numpy()
        dq, dk, dv = oracle.ring_step_bwd(self._embed(q, rank), self._embed(k, src), self._embed(v, src),
                                          self._embed(state["dO"], rank), lse, D, self.causal, self.n, rank, src,
                                          schedule=self.schedule)
        state["dq"] += self._rows(dq, rank)
        dk_acc += self._rows(dk, src)
        dv_acc += self._rows(dv, src)

    def bwd_end(self, state, dk_acc, dv_acc, d):
        return state["dq"], dk_acc, dv_acc


def _worker(rank, world, port, shape, schedule, out):
    from sequence_blockwise_self_gb300 import ring_dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, Hq, Hkv, L, d, causal = shape
        gen = torch.Generator().manual_seed(123)
        q, k, v, dO = (torch.randn((B, H, L, d), generator=gen, dtype=torch.float64) for H in (Hq, Hkv, Hkv, Hq))
        pos = torch.from_numpy(_positions(L, world, causal, rank, schedule))
        mine = [x[:, :, pos].contiguous() for x in (q, k, v, dO)]
        ops = OracleRingOps(L, Hkv, causal, schedule, world)
        o, lse = ring_dist.ring_attention_fwd(*mine[:3], causal, schedule=schedule, ops=ops)
        dq, dk, dv = ring_dist.ring_attention_bwd(*mine[:3], o, lse, mine[3], causal, schedule=schedule, ops=ops)
        out[rank] = tuple(t.numpy() for t in (o, lse, dq, dk, dv))
    finally:
        dist.destroy_process_group()


# (B, Hq, Hkv, L, d, causal), world size, schedule
CASES = [((1, 2, 1, 24, 4, True), 2, "fold"), ((1, 2, 2, 24, 4, False), 3, "fold"),
         ((2, 4, 2, 32, 4, True), 4, "fold"), ((1, 2, 1, 24, 4, True), 3, "striped"),
         ((1, 3, 1, 24, 4, True), 4, "contiguous")]


@pytest.mark.parametrize("shape,world,schedule", CASES,
                         ids=[f"L{c[0][3]}-N{c[1]}-{c[2]}{'-causal' if c[0][5] else ''}" for c in CASES])
def test_ring_driver_over_gloo_ranks_equals_the_plain_definition(shape, world, schedule):
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, shape, schedule, out), nprocs=world, start_method="spawn",
                       join=True)
    B, Hq, Hkv, L, d, causal = shape
    gen = torch.Generator().manual_seed(123)
    q, k, v, dO = (torch.randn((B, H, L, d), generator=gen, dtype=torch.float64) for H in (Hq, Hkv, Hkv, Hq))
    o_ref, lse_ref = oracle.fwd(q, k, v, causal)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(q, k, v, dO, causal)
    for rank in range(world):
        pos = _positions(L, world, causal, rank, schedule)
        o, lse, dq, dk, dv = out[rank]
        for name, got, want in (("o", o, o_ref), ("lse", lse, lse_ref), ("dq", dq, dq_ref), ("dk", dk, dk_ref),
                                ("dv", dv, dv_ref)):
            np.testing.assert_allclose(got, want[:, :, pos], rtol=0, atol=1e-10, err_msg=f"{name} rank {rank}")


def test_ring_driver_rejects_the_distflash_schedule():
    from sequence_blockwise_self_gb300 import ring_dist
    with pytest.raises(ValueError):
        ring_dist.ring_attention_fwd(None, None, None, True, schedule="dfa")
