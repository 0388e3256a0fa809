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

Tensors are the rank's chunk in chunk order ([B, H, C, d]) under the
schedule's chunk map ("fold", "striped" or "contiguous"; positions per
include/ring_attn.h).  The exchange uses torch.distributed point-to-point
operations (NCCL between GPUs, gloo on CPU), the blocks run through `ops`
-- by default the library's kernels on this rank's GPU.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import capi

RING_SCHEDULES = ("fold", "striped", "contiguous")


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


def ring_attention_fwd(q, k, v, causal: bool, group=None, schedule: str = "fold", ops=None):
    """This rank's share of softmax(q k^T / sqrt(d)) v over the ring: q
    [B, Hq, C, d], k, v [B, Hkv, C, d] are the rank's chunk; returns its rows'
    o (bf16 with the default ops) and lse (fp32)."""
    if schedule not in RING_SCHEDULES:
        raise ValueError(f"schedule must be one of {RING_SCHEDULES}")
    ops = ops or CudaRingOps()
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
