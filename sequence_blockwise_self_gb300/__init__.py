"""GB300-native (sm_103a) blockwise Ring Self-Attention.

Public API (torch tensors in, torch tensors out; the arithmetic runs in the
library's CUDA kernels):
    ring_attn_fwd(q, k, v, n_chunks, causal) -> (o, lse)
    ring_attn_bwd(q, k, v, o, lse, dO, n_chunks, causal) -> (dq, dk, dv)
Ring mode (the ring run step by step, as each rank of a multi-GPU ring
would): ring_attn_fwd_step, ring_attn_merge, ring_attn_ring_fwd,
ring_attn_ring_bwd.
Ulysses on one GPU (sequence shards -> head shards -> back):
ring_attn_ulysses_fwd, ring_attn_ulysses_bwd; USP (Ulysses groups and a ring
across them): ring_attn_usp_fwd, ring_attn_usp_bwd.
Blockwise feed-forward (BPT): ring_attn_ffn_fwd, ring_attn_ffn_bwd; the blockwise transformer
forward (attention, then FFN, per query block) and its backward:
ring_attn_bpt_fwd, ring_attn_bpt_bwd.
Host-only queries: owner_rank, fwd_plan, bwd_plan, step_plan.
"""
from .capi import (  # noqa: F401
    RingAttnError,
    bwd_plan,
    bwd_workspace_size,
    device_status,
    fwd_plan,
    load,
    owner_rank,
    profile_enable,
    profile_read,
    release,
    selftest_bounded_wait,
    step_plan,
    schedule_launches,
    schedule_pairs,
    SCHEDULES,
    ring_attn_bwd,
    ring_attn_bwd_noalloc,
    ring_attn_fwd,
    ring_attn_ffn_fwd,
    ring_attn_ffn_bwd,
    ffn_workspace_size,
    ffn_bwd_workspace_size,
    ring_attn_bpt_fwd,
    ring_attn_bpt_bwd,
    bpt_workspace_size,
    bpt_bwd_workspace_size,
    ring_attn_fwd_step,
    ring_attn_fwd_step_accumulate,
    RankBackward,
    grad_to_bf16,
    add_f32,
    ring_attn_merge,
    ring_attn_ring_fwd,
    ring_fwd_workspace_size,
    ring_attn_ring_bwd,
    ring_bwd_workspace_size,
    ring_attn_ulysses_bwd,
    ring_attn_ulysses_fwd,
    ring_attn_usp_bwd,
    ring_attn_usp_fwd,
    ulysses_workspace_size,
    usp_workspace_size,
    strerror,
)
