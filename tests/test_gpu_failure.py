"""Failure detection without a GPU fault.

Every wait on an mbarrier in the kernels is bounded in time; when it gives
up it raises the CTA's abort flag, records a site code in the device status
word and lets the kernel return.  The self-test kernel runs that same bounded
wait on a barrier nothing will ever arrive at, so the timeout path runs for
real: the host must read RING_ATTN_ERR_DEVICE_TIMEOUT with the self-test site,
the word must be cleared by the read, and the context must stay usable.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import capi, inputs

pytestmark = pytest.mark.gpu

SITE_SELFTEST = 0x301


def test_bounded_wait_times_out_reports_and_context_survives():
    lib_build.build()
    ra.load()
    torch.cuda.synchronize()
    assert ra.device_status() == (capi.OK, 0)
    t0 = time.perf_counter()
    ra.selftest_bounded_wait(20000)  # 20 ms
    st, site = ra.device_status()
    dt = time.perf_counter() - t0
    assert st == capi.ERR_DEVICE_TIMEOUT and site == SITE_SELFTEST, (st, hex(site))
    assert 0.015 <= dt < 5.0, dt
    assert ra.device_status() == (capi.OK, 0), "status word not cleared by the read"
    # the context still computes attention correctly
    q, k, v, _ = inputs.make_inputs(1, 2, 2, 256, 64, seed=3, with_grad=False)
    o, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), 2, True)
    torch.cuda.synchronize()
    assert ra.device_status() == (capi.OK, 0)
    o_ref, _ = oracle.fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), True)
    assert np.abs(o.float().cpu().double().numpy() - o_ref).max() < 2e-2
