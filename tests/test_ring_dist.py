"""The multi-GPU ring driver (ring_dist) on CPU ranks: gloo, world sizes 2
to 6, one process per rank, for the ring's chunk maps and for
DistFlashAttention's protocol (helpers receive query chunks, return
partial results and dQ).  Each rank runs ring_attention_fwd and
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

    # DistFlashAttention's helper blocks
    def fwd_merge(self, o_run, lse_run, o_s, lse_s):
        o, lse = oracle.merge(o_run.numpy(), lse_run.numpy(), o_s.numpy(), lse_s.numpy())
        o_run.copy_(torch.from_numpy(o))
        lse_run.copy_(torch.from_numpy(lse))

    def bwd_dq_partial(self, state):
        return state["dq"]

    def bwd_add_dq(self, state, partial):
        state["dq"] += partial

    def add(self, dst, src):
        dst += src


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


# (B, Hq, Hkv, L, d, causal), world size, schedule.  DistFlashAttention at
# world sizes 2 (no helper), 3 and 5 (odd: every launch pairs), 4 and 6
# (even: the middle launch pairs nobody).
CASES = [((1, 2, 1, 24, 4, True), 2, "fold"), ((1, 2, 2, 24, 4, False), 3, "fold"),
         ((2, 4, 2, 32, 4, True), 4, "fold"), ((1, 2, 1, 24, 4, True), 3, "striped"),
         ((1, 3, 1, 24, 4, True), 4, "contiguous"), ((1, 2, 1, 16, 4, True), 2, "dfa"),
         ((1, 2, 1, 24, 4, True), 3, "dfa"), ((2, 2, 2, 32, 4, True), 4, "dfa"),
         ((1, 3, 1, 30, 4, True), 5, "dfa"), ((1, 2, 1, 36, 4, True), 6, "dfa")]


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


def test_ring_driver_rejects_unknown_schedules_and_non_causal_distflash():
    from sequence_blockwise_self_gb300 import ring_dist
    with pytest.raises(ValueError):
        ring_dist.ring_attention_fwd(None, None, None, True, schedule="zigzag")
    with pytest.raises(ValueError):
        ring_dist.ring_attention_bwd(None, None, None, None, None, None, True, schedule="zigzag")


def test_distflash_roles_cover_every_causal_block_once():
    """DistFlashAttention's launches in the driver (SP series section 7.2):
    every block (a, b <= a) runs exactly once -- on rank a at launch a - b
    when a - b <= n/2, else on helper b at launch n - (a - b) -- and no rank
    runs two blocks in one launch."""
    from sequence_blockwise_self_gb300.ring_dist import _dfa_roles
    for n in range(1, 13):
        seen = {}
        for t in range(n // 2 + 1):
            for r in range(n):
                own, helper_of, helped_by = _dfa_roles(n, r, t)
                blocks = ([(r, r - t)] if own else []) + ([(helper_of, r)] if helper_of is not None else [])
                assert len(blocks) <= 1, (n, t, r)
                for blk in blocks:
                    assert blk not in seen, (n, blk)
                    seen[blk] = t
                if helped_by is not None:  # the helper agrees on the pairing
                    assert _dfa_roles(n, helped_by, t)[1] == r
        assert set(seen) == {(a, b) for a in range(n) for b in range(a + 1)}, n
