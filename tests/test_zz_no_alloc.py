"""ring_attn_bwd_noalloc: the backward pass for callers that cannot call
cudaMalloc -- code whose device memory is owned by another allocator, or
that cannot accept the device synchronisation cudaMalloc/cudaFree may cause.
It works in the library's static device array instead of a workspace, so its
gradients must equal those of ring_attn_bwd, call after call (the array
keeps the previous call's contents, which must not leak into the next).

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import sequence_blockwise_self_gb300 as ra
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import capi
from sequence_blockwise_self_gb300 import inputs

pytestmark = pytest.mark.gpu

from tolerance import check_bf16  # the parity tolerance of the other GPU tests


def _close(name, got, want):
    # both sides are bf16 results: two half-ulps of output rounding excused
    check_bf16(name, got.float().cpu().double().numpy(), want.float().cpu().double().numpy(), ulps=2)


def test_noalloc_backward_matches_workspace_backward_on_two_calls_in_a_row():
    lib_build.build()
    lib = ra.load()
    # (B, Hq, Hkv, L, d, n_chunks, causal): the second call has another shape,
    # head size and mask, so stale statistics or plan from the first would show.
    shapes = [(1, 4, 2, 1024, 128, 4, True), (2, 2, 2, 640, 64, 5, False)]
    cases = []
    for i, (B, Hq, Hkv, L, d, N, causal) in enumerate(shapes):
        q, k, v, dO = (t.cuda() for t in inputs.make_inputs(B, Hq, Hkv, L, d, seed=500 + i))
        o, lse = ra.ring_attn_fwd(q, k, v, N, causal)
        ref = ra.ring_attn_bwd(q, k, v, o, lse, dO, N, causal)
        out = (torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan")))
        cases.append(((q, k, v, o, lse, dO, N, causal), ref, out))
    torch.cuda.synchronize()
    # the two calls of the allocation-free entry point, back to back
    for args, _, (dq, dk, dv) in cases:
        ra.ring_attn_bwd_noalloc(*args, dq, dk, dv)
    torch.cuda.synchronize()
    st, site = ra.device_status()
    assert st == 0, f"device status {st} at {site:#x}"
    for (_, (dq_r, dk_r, dv_r), (dq, dk, dv)) in cases:
        _close("dq", dq, dq_r)
        _close("dk", dk, dk_r)
        _close("dv", dv, dv_r)

    # a problem whose workspace does not fit the static array is refused
    # before anything is touched or launched
    fake = [ctypes.c_void_p(1 << 20)] * 9
    B, Hq, L, d = 1, 32, 8192, 128
    assert ra.bwd_workspace_size(B, Hq, Hq, L, d, 8, True) > capi_limit()
    rc = lib.ring_attn_bwd_noalloc(*fake, B, Hq, Hq, L, d, 8, 1, ctypes.c_void_p(0))
    assert rc == capi.ERR_WORKSPACE


def capi_limit():
    return 64 * 1024 * 1024


def test_noalloc_backward_at_the_size_limit():
    """The largest MHA problem at d = 128 the static array serves: 129,024
    rows, whose fp32 dQ accumulator and statistics leave 16 KB of the array
    for the launch plan; the gradients equal ring_attn_bwd's, so the upper
    end of the array (and the plan placed after the workspace) is right."""
    lib_build.build()
    ra.load()
    B, Hq, Hkv, L, d, N, causal = 1, 16, 16, 8064, 128, 3, False
    ws = ra.bwd_workspace_size(B, Hq, Hkv, L, d, N, causal)
    assert capi_limit() - 16384 <= ws <= capi_limit() - 1024
    q, k, v, dO = (t.cuda() for t in inputs.make_inputs(B, Hq, Hkv, L, d, seed=530))
    o, lse = ra.ring_attn_fwd(q, k, v, N, causal)
    dq_r, dk_r, dv_r = ra.ring_attn_bwd(q, k, v, o, lse, dO, N, causal)
    dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
    ra.ring_attn_bwd_noalloc(q, k, v, o, lse, dO, N, causal, dq, dk, dv)
    torch.cuda.synchronize()
    st, site = ra.device_status()
    assert st == 0, f"device status {st} at {site:#x}"
    _close("dq", dq, dq_r)
    _close("dk", dk, dk_r)
    _close("dv", dv, dv_r)


def test_noalloc_backward_captured_in_a_cuda_graph_and_replayed():
    """A call captured into a CUDA graph (after one plain call of the same
    shape) replays the whole backward: its gradients equal ring_attn_bwd's,
    and after the inputs change in place a second replay follows them."""
    lib_build.build()
    ra.load()
    B, Hq, Hkv, L, d, N, causal = 1, 4, 2, 1024, 128, 4, True
    q, k, v, dO = (t.cuda() for t in inputs.make_inputs(B, Hq, Hkv, L, d, seed=520))
    o, lse = ra.ring_attn_fwd(q, k, v, N, causal)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ra.ring_attn_bwd_noalloc(q, k, v, o, lse, dO, N, causal, dq, dk, dv)  # first call of this shape: not captured
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ra.ring_attn_bwd_noalloc(q, k, v, o, lse, dO, N, causal, dq, dk, dv)
    for seed in (521, 522):
        q2, k2, v2, dO2 = (t.cuda() for t in inputs.make_inputs(B, Hq, Hkv, L, d, seed=seed))
        for dst, src in ((q, q2), (k, k2), (v, v2), (dO, dO2)):
            dst.copy_(src)
        o2, lse2 = ra.ring_attn_fwd(q, k, v, N, causal)
        o.copy_(o2)
        lse.copy_(lse2)
        for t in (dq, dk, dv):
            t.fill_(float("nan"))
        graph.replay()
        ref = ra.ring_attn_bwd(q, k, v, o, lse, dO, N, causal)
        torch.cuda.synchronize()
        st, site = ra.device_status()
        assert st == 0, f"device status {st} at {site:#x}"
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            _close(f"{name} replay seed {seed}", got, want)
