"""Ring attention across GPUs: one process per GPU, each holding one chunk.

The ring of "Large-scale distributed AI model training series: sequence
parallelism" (section 2.3 Ring Self-Attention, section 6.2 Ring Attention):
rank r keeps its query chunk while the key/value chunks travel round the
ring -- at step s it holds the keys and values of rank (r - s) mod N and
sends them on to rank r + 1 while it computes with them.

* Forward: every block is accumulated into the rank's running result (the
  online softmax continues across blocks, ring_attn_fwd_step_accumulate),
  so no partial result is exchanged; the key/value transfer of step s + 1
  overlaps the block of step s.
* Backward (activations recomputed from lse): K and V travel again, and
  with them the fp32 dK, dV accumulators of their chunk: each rank adds its
  block's contributions into the accumulators it holds and passes them on;
  after the last step they are one rank short of home and take one more
  hop.  dQ stays local.

* DistFlashAttention ("dfa", section 7.2; contiguous causal chunks): only
  N/2 + 1 launches.  At launch t rank w >= t runs its own block (its
  queries, the keys of chunk w - t, which travel as in the ring); a rank
  w < t that the plain ring would leave idle instead runs the block of
  rank a = N - t + w against its own keys -- the owner sends it q (and, in
  the backward, o, dO and lse), and it returns the partial result (o, lse)
  or the fp32 dQ partial, which the owner merges or adds.  That block's
  dK/dV stay with the helper, which owns those keys.  After the last
  launch the travelling dK/dV accumulators go home in one hop.

Tensors are the rank's chunk in chunk order ([B, H, C, d]) under the
schedule's chunk map ("fold", "striped", "contiguous" or "dfa"; positions
per include/ring_attn.h).  The exchange uses torch.distributed point-to-point
operations (NCCL between GPUs, gloo on CPU), the blocks run through `ops`
-- by default the library's kernels on this rank's GPU.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import capi

RING_SCHEDULES = ("fold", "striped", "contiguous", "dfa")


class CudaRingOps:
    """The per-rank blocks on this process's GPU (the library's kernels)."""

    acc_dtype = torch.float32  # the travelling dK, dV accumulators

    def fwd_begin(self, q):
        B, Hq, C, d = q.shape
        o_run = torch.zeros((B, Hq, C, d), dtype=torch.float32, device=q.device)
        lse_run = torch.full((B, Hq, C), float("-inf"), dtype=torch.float32, device=q.device)
        return o_run, lse_run

    def fwd_block(self, q, k, v, o_run, lse_run, n_chunks, causal, rank, src, schedule):
        capi.ring_attn_fwd_step_accumulate(q, k, v, o_run, lse_run, n_chunks, causal, rank, src, schedule=schedule)

    def fwd_end(self, o_run, lse_run):
        return o_run.to(torch.bfloat16), lse_run

    def bwd_begin(self, o, dO, lse, Hkv, n_chunks, causal, schedule):
        return capi.RankBackward(o, dO, lse, Hkv, n_chunks, causal, schedule=schedule)

    def bwd_block(self, state, q, k, v, dk_acc, dv_acc, rank, src):
        state.step(q, k, v, dk_acc, dv_acc, rank, src)

    def bwd_end(self, state, dk_acc, dv_acc, d):
        scale = 1.0 / d ** 0.5
        return state.end(), capi.grad_to_bf16(dk_acc, scale), capi.grad_to_bf16(dv_acc, 1.0)

    # DistFlashAttention's helper blocks
    def fwd_merge(self, o_run, lse_run, o_s, lse_s):
        capi.ring_attn_merge(o_run, lse_run, o_s, lse_s)

    def bwd_dq_partial(self, state):
        return state.dq_accumulator()

    def bwd_add_dq(self, state, partial):
        state.add_dq(partial)

    def add(self, dst, src):
        capi.add_f32(dst, src)


def _send_recv(send, recv, dst, src, group):
    """Post sends of `send` to dst and receives into `recv` from src; returns
    the requests (one grouped launch on NCCL, so the ring cannot deadlock)."""
    ops = [dist.P2POp(dist.isend, t, dst, group) for t in send]
    ops += [dist.P2POp(dist.irecv, t, src, group) for t in recv]
    return dist.batch_isend_irecv(ops)


def _wait(reqs):
    for r in reqs:
        r.wait()


def _ring(group):
    n = dist.get_world_size(group)
    r = dist.get_rank(group)
    return n, r, dist.get_global_rank(group, (r + 1) % n) if group else (r + 1) % n, \
        dist.get_global_rank(group, (r - 1) % n) if group else (r - 1) % n


def _peer(group, rank):
    return dist.get_global_rank(group, rank) if group else rank


def _dfa_roles(n, r, t):
    """Launch t of DistFlashAttention's schedule for rank r: whether it runs
    its own block (r, r - t), the owner whose block (a, r) it runs for it
    (None if none) and the helper that runs its block (r, r + t - n) (None
    if none).  Launch t = n - t (even n) pairs nobody."""
    paired = t < n - t
    helper_of = n - t + r if (r < t and paired) else None
    helped_by = r + t - n if (r >= n - t and paired) else None
    return r >= t, helper_of, helped_by


def _p2p(ops_list):
    return dist.batch_isend_irecv(ops_list) if ops_list else []


def ring_attention_fwd(q, k, v, causal: bool, group=None, schedule: str = "fold", ops=None):
    """This rank's share of softmax(q k^T / sqrt(d)) v over the ring: q
    [B, Hq, C, d], k, v [B, Hkv, C, d] are the rank's chunk; returns its rows'
    o (bf16 with the default ops) and lse (fp32)."""
    if schedule not in RING_SCHEDULES:
        raise ValueError(f"schedule must be one of {RING_SCHEDULES}")
    ops = ops or CudaRingOps()
    if schedule == "dfa":
        return _dfa_fwd(q, k, v, causal, group, ops)
    n, r, nxt, prv = _ring(group)
    o_run, lse_run = ops.fwd_begin(q)
    cur = (k, v)
    for s in range(n):
        reqs = []
        if s + 1 < n:  # the next chunk travels while this block runs
            nxt_buf = (torch.empty_like(k), torch.empty_like(v))
            reqs = _send_recv(cur, nxt_buf, nxt, prv, group)
        ops.fwd_block(q, cur[0], cur[1], o_run, lse_run, n, causal, r, (r - s) % n, schedule)
        if reqs:
            _wait(reqs)
            cur = nxt_buf
    return ops.fwd_end(o_run, lse_run)


def ring_attention_bwd(q, k, v, o, lse, dO, causal: bool, group=None, schedule: str = "fold", ops=None):
    """Gradients of sum(dO * o) for this rank's chunk: returns (dq, dk, dv)
    of the rank's rows.  o, lse from ring_attention_fwd."""
    if schedule not in RING_SCHEDULES:
        raise ValueError(f"schedule must be one of {RING_SCHEDULES}")
    ops = ops or CudaRingOps()
    if schedule == "dfa":
        return _dfa_bwd(q, k, v, o, lse, dO, causal, group, ops)
    n, r, nxt, prv = _ring(group)
    Hkv, d = k.shape[1], k.shape[3]
    state = ops.bwd_begin(o, dO, lse, Hkv, n, causal, schedule)
    kv = (k, v)
    acc = (torch.zeros(k.shape, dtype=ops.acc_dtype, device=k.device),
           torch.zeros(v.shape, dtype=ops.acc_dtype, device=v.device))
    for s in range(n):
        src = (r - s) % n
        reqs = []
        if s + 1 < n:  # the next key/value chunk travels while this block runs
            kv_next = (torch.empty_like(k), torch.empty_like(v))
            reqs = _send_recv(kv, kv_next, nxt, prv, group)
        ops.bwd_block(state, q, kv[0], kv[1], acc[0], acc[1], r, src)
        # the accumulators carry this block's contributions: they follow
        # their chunk to the next rank (after the last block: one hop home)
        acc_next = (torch.empty_like(acc[0]), torch.empty_like(acc[1]))
        reqs += _send_recv(acc, acc_next, nxt, prv, group)
        _wait(reqs)
        acc = acc_next
        if s + 1 < n:
            kv = kv_next
    return ops.bwd_end(state, acc[0], acc[1], d)


def _dfa_fwd(q, k, v, causal, group, ops):
    if not causal:
        raise ValueError("DistFlashAttention's schedule is for causal attention")
    n, r, nxt, prv = _ring(group)
    o_run, lse_run = ops.fwd_begin(q)
    cur = (k, v)  # at launch t: the keys and values of chunk r - t
    for t in range(n // 2 + 1):
        own, helper_of, helped_by = _dfa_roles(n, r, t)
        kv_reqs = []
        if t + 1 <= n // 2:  # the next launch's chunk travels meanwhile
            nxt_buf = (torch.empty_like(k), torch.empty_like(v))
            kv_reqs = _send_recv(cur, nxt_buf, nxt, prv, group)
        q_in = torch.empty_like(q) if helper_of is not None else None
        q_reqs = _p2p(([dist.P2POp(dist.irecv, q_in, _peer(group, helper_of), group)] if helper_of is not None
                       else []) +
                      ([dist.P2POp(dist.isend, q, _peer(group, helped_by), group)] if helped_by is not None
                       else []))
        if own:
            ops.fwd_block(q, cur[0], cur[1], o_run, lse_run, n, causal, r, r - t, "contiguous")
        _wait(q_reqs)
        back = []
        if helper_of is not None:  # owner helper_of's block against this rank's keys
            o_p, lse_p = ops.fwd_begin(q_in)
            ops.fwd_block(q_in, k, v, o_p, lse_p, n, causal, helper_of, r, "contiguous")
            back = [dist.P2POp(dist.isend, o_p, _peer(group, helper_of), group),
                    dist.P2POp(dist.isend, lse_p, _peer(group, helper_of), group)]
        if helped_by is not None:
            o_in, lse_in = torch.empty_like(o_run), torch.empty_like(lse_run)
            back += [dist.P2POp(dist.irecv, o_in, _peer(group, helped_by), group),
                     dist.P2POp(dist.irecv, lse_in, _peer(group, helped_by), group)]
        _wait(_p2p(back))
        if helped_by is not None:
            ops.fwd_merge(o_run, lse_run, o_in, lse_in)
        if kv_reqs:
            _wait(kv_reqs)
            cur = nxt_buf
    return ops.fwd_end(o_run, lse_run)


def _dfa_bwd(q, k, v, o, lse, dO, causal, group, ops):
    if not causal:
        raise ValueError("DistFlashAttention's schedule is for causal attention")
    n, r, nxt, prv = _ring(group)
    Hkv, d = k.shape[1], k.shape[3]
    state = ops.bwd_begin(o, dO, lse, Hkv, n, causal, "contiguous")
    kv = (k, v)
    acc = (torch.zeros(k.shape, dtype=ops.acc_dtype, device=k.device),
           torch.zeros(v.shape, dtype=ops.acc_dtype, device=v.device))  # travel with chunk r - t
    home = (torch.zeros_like(acc[0]), torch.zeros_like(acc[1]))  # this chunk's share of the helped blocks
    last = n // 2
    for t in range(last + 1):
        own, helper_of, helped_by = _dfa_roles(n, r, t)
        kv_reqs = []
        if t < last:
            kv_next = (torch.empty_like(k), torch.empty_like(v))
            kv_reqs = _send_recv(kv, kv_next, nxt, prv, group)
        ins, outs = [], []
        if helper_of is not None:
            got = (torch.empty_like(q), torch.empty_like(o), torch.empty_like(dO), torch.empty_like(lse))
            ins = [dist.P2POp(dist.irecv, x, _peer(group, helper_of), group) for x in got]
        if helped_by is not None:
            outs = [dist.P2POp(dist.isend, x, _peer(group, helped_by), group) for x in (q, o, dO, lse)]
        x_reqs = _p2p(ins + outs)
        if own:
            ops.bwd_block(state, q, kv[0], kv[1], acc[0], acc[1], r, r - t)
        _wait(x_reqs)
        back = []
        if helper_of is not None:  # owner helper_of's block against this rank's keys
            qa, oa, dOa, lsea = got
            hstate = ops.bwd_begin(oa, dOa, lsea, Hkv, n, causal, "contiguous")
            ops.bwd_block(hstate, qa, k, v, home[0], home[1], helper_of, r)
            back = [dist.P2POp(dist.isend, ops.bwd_dq_partial(hstate), _peer(group, helper_of), group)]
        if helped_by is not None:
            dq_in = torch.empty_like(ops.bwd_dq_partial(state))
            back += [dist.P2POp(dist.irecv, dq_in, _peer(group, helped_by), group)]
        _wait(_p2p(back))
        if helped_by is not None:
            ops.bwd_add_dq(state, dq_in)
        # the accumulators follow their chunk; after the last launch, home
        dst, src = ((nxt, prv) if t < last else (_peer(group, (r - t) % n), _peer(group, (r + t) % n)))
        if dst == _peer(group, r):
            acc_next = acc
        else:
            acc_next = (torch.empty_like(acc[0]), torch.empty_like(acc[1]))
            _wait(_send_recv(acc, acc_next, dst, src, group))
        acc = acc_next
        if kv_reqs:
            _wait(kv_reqs)
            kv = kv_next
    ops.add(acc[0], home[0])
    ops.add(acc[1], home[1])
    return ops.bwd_end(state, acc[0], acc[1], d)
