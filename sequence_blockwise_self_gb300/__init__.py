"""GB300-native (sm_103a) blockwise Ring Self-Attention.

Public API (torch tensors in, torch tensors out; the arithmetic runs in the
library's CUDA kernels):
    ring_attn_fwd(q, k, v, n_chunks, causal) -> (o, lse)
    ring_attn_bwd(q, k, v, o, lse, dO, n_chunks, causal) -> (dq, dk, dv)
Host-only queries: owner_rank, fwd_plan, bwd_plan.
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
    ring_attn_bwd,
    ring_attn_bwd_noalloc,
    ring_attn_fwd,
    strerror,
)
