"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances (bf16 outputs and gradients, fp32 accumulation): max-abs error
<= 2e-2 beyond the bf16 rounding of the output (see tolerance.py) and
mean-abs error <= 2e-3 on o, dq, dk, dv; lse within 1e-3.
Small shapes are compared element by element on every output; the large
workloads on 256 sampled query rows per head (o, lse, dq) and 256 sampled key
rows per kv head (dk, dv), with the oracle's own fp64 statistics.
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_blockwise_self_gb300 as ra
from tolerance import TOL_LSE, TOL_MAX, TOL_MEAN, check_bf16, check_fp32, note
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


def f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(name, got, want, tol_max=TOL_MAX, tol_mean=TOL_MEAN):
    if tol_max == TOL_LSE and tol_mean == TOL_LSE:
        check_fp32(name, got, want, TOL_LSE)
    else:
        check_bf16(name, got, want, tol_max, tol_mean)


def assert_status_ok():
    st, site = ra.device_status()
    assert st == 0, f"device status {st} at site {site:#x}"


def gpu_fwd_bwd(q, k, v, dO, n_chunks, causal):
    qd, kd, vd, dOd = (x.cuda() for x in (q, k, v, dO))
    o, lse = ra.ring_attn_fwd(qd, kd, vd, n_chunks, causal)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, o, lse, dOd, n_chunks, causal)
    torch.cuda.synchronize()
    assert_status_ok()
    return o, lse, dq, dk, dv


# (B, Hq, Hkv, L, d, n_chunks, causal)
SMALL = [
    (1, 2, 2, 256, 64, 1, False),     # the tiny workload, every chunk count
    (1, 2, 2, 256, 64, 2, False),
    (1, 2, 2, 256, 64, 4, False),
    (1, 4, 2, 512, 128, 1, True),     # GQA causal, sub-chunks of 256 / 128 / 64
    (1, 4, 2, 512, 128, 2, True),
    (1, 4, 2, 512, 128, 4, True),
    (2, 2, 1, 384, 64, 3, True),      # MQA, odd tile count, c = 64
    (2, 8, 2, 768, 128, 3, False),    # GQA G = 4, N = 3
    (1, 2, 2, 200, 128, 2, False),    # ragged: L not a multiple of the tile
    (1, 2, 2, 200, 64, 2, True),
    (1, 3, 1, 1000, 128, 5, True),    # ragged, chunks of 100 rows
    (1, 2, 2, 1024, 128, 8, True),
    (1, 2, 2, 128, 128, 1, True),     # a single tile
    (1, 1, 1, 2, 64, 1, True),        # degenerate: two tokens
    # d = 64 over many key tiles (the forward's own P columns and pv_done
    # hand-off, the backward's separate dQ columns): causal GQA and a ragged
    # causal MHA whose last block ends mid-tile
    (1, 8, 2, 4096, 64, 8, True),
    (2, 4, 4, 3000, 64, 5, True),
    (1, 4, 1, 2560, 64, 1, False),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}-{}L{}d{}N{}{}".format(*s[:6], "c" if s[6] else "e"))
def test_small_shapes_full_parity(shape):
    B, Hq, Hkv, L, d, N, causal = shape
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=1000 + SMALL.index(shape))
    o, lse, dq, dk, dv = gpu_fwd_bwd(q, k, v, dO, N, causal)
    o_ref, lse_ref = oracle.fwd(f64(q), f64(k), f64(v), causal)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(f64(q), f64(k), f64(v), f64(dO), causal)
    assert_close("o", f64(o), o_ref)
    assert_close("lse", f64(lse), lse_ref, TOL_LSE, TOL_LSE)
    assert_close("dq", f64(dq), dq_ref)
    assert_close("dk", f64(dk), dk_ref)
    assert_close("dv", f64(dv), dv_ref)


def test_chunk_count_changes_only_rounding():
    """The same inputs through N = 1, 2, 4, 8: outputs agree to fp32
    summation-order differences (well inside the bf16 tolerance)."""
    B, Hq, Hkv, L, d = 1, 4, 2, 1024, 128
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=77)
    outs = [gpu_fwd_bwd(q, k, v, dO, N, True) for N in (1, 2, 4, 8)]
    for other in outs[1:]:
        for a, b, name in zip(outs[0], other, ("o", "lse", "dq", "dk", "dv")):
            if name == "lse":
                check_fp32(name, f64(b), f64(a), 1e-3)
            else:
                check_bf16(name, f64(b), f64(a), 1e-2, 1e-3, ulps=2)


@pytest.mark.parametrize("d", [64, 128])
def test_causal_row_zero_is_exact(d):
    """Query 0 of a causal model sees only key 0, so P = 1: o_0 must equal v_0
    bit for bit, lse_0 = q_0.k_0/sqrt(d), and dq_0 = 0 up to fp32 rounding."""
    B, Hq, Hkv, L = 2, 8, 2, 1024
    q, k, v, dO = inputs.make_inputs(B, Hq, Hkv, L, d, seed=31)
    o, lse, dq, dk, dv = gpu_fwd_bwd(q, k, v, dO, 4, True)
    G = Hq // Hkv
    v0 = v[:, :, 0].repeat_interleave(G, dim=1)
    assert torch.equal(o[:, :, 0].cpu(), v0), "o_0 differs from v_0"
    s00 = (f64(q[:, :, 0]) * f64(k[:, :, 0].repeat_interleave(G, dim=1))).sum(-1) / np.sqrt(d)
    check_fp32("lse_0", f64(lse[:, :, 0]), s00, 1e-5)
    # dq_0 = P_00 (dP_00 - D_0): both terms are dO_0 . v_0, summed in different
    # orders (tensor core vs the pre-pass), so only fp32 rounding remains
    assert dq[:, :, 0].float().abs().max().item() <= 1e-3, "dq_0 is not ~0"


def test_repeat_calls_are_deterministic_in_forward():
    q, k, v, dO = inputs.make_inputs(1, 2, 2, 512, 128, seed=5)
    o1, l1, *_ = gpu_fwd_bwd(q, k, v, dO, 2, True)
    o2, l2, *_ = gpu_fwd_bwd(q, k, v, dO, 2, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_problem_is_a_no_op():
    q = torch.empty((0, 2, 128, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = ra.ring_attn_fwd(q, q[:, :2], q[:, :2], 1, False)
    assert o.numel() == 0 and lse.numel() == 0


# ------------------------------------------------------------ full workloads

# Key rows for dk/dv.  A key row's gradient sums over every query that sees
# it, so its fp64 reference needs lse_i and D_i of all those queries: the
# oracle's row-sampled backward runs its own full statistics pass over them
# (never the GPU's lse).  The keys are sampled over the whole sequence (row 0
# and every chunk / sub-chunk boundary included), so key tiles that
# accumulate over every query tile, all G query heads of a group and every
# ring step are compared.  At 128k the statistics of every row would take
# about an hour of fp64 CPU time, so there the keys come from the last 8192
# positions (four sub-chunks of different ranks; each such key still
# gathers up to 64 query tiles over 7 heads) and two of the four kv groups.
KEY_WINDOW = {"gqa_128k": 8192}
KEY_GROUPS = {"gqa_128k": (0, 3)}


def _oracle_key_grads(w, qf, kf, vf, dOf, k_rows):
    """fp64 dk, dv on k_rows ([B, Hkv, R, d]; kv groups not in KEY_GROUPS are
    NaN and skipped by the comparison)."""
    groups = KEY_GROUPS.get(w.name)
    if groups is None:
        _, dk, dv = oracle.bwd_rows(qf, kf, vf, dOf, w.causal, np.zeros(0, np.int32), k_rows)
        return dk, dv, list(range(w.Hkv))
    G = w.Hq // w.Hkv
    dk = np.full((w.B, w.Hkv, k_rows.size, w.d), np.nan)
    dv = np.full_like(dk, np.nan)
    for g in groups:
        sl = slice(g * G, (g + 1) * G)
        _, dk_g, dv_g = oracle.bwd_rows(qf[:, sl], kf[:, g:g + 1], vf[:, g:g + 1], dOf[:, sl], w.causal,
                                        np.zeros(0, np.int32), k_rows)
        dk[:, g], dv[:, g] = dk_g[:, 0], dv_g[:, 0]
    return dk, dv, list(groups)


def _sampled_parity(w: inputs.Workload, chunk_counts):
    import time
    q, k, v, dO = inputs.workload_inputs(w)
    seed = inputs.WORKLOAD_SEEDS[w.name]
    rows = inputs.sample_rows(w.L, w.n_chunks, w.causal, 256, seed)
    k_lo = max(0, w.L - KEY_WINDOW.get(w.name, w.L))
    k_rows = inputs.sample_rows(w.L, w.n_chunks, w.causal, 256, seed + 1, lo=k_lo)
    qf, kf, vf, dOf = f64(q), f64(k), f64(v), f64(dO)
    t0 = time.perf_counter()
    o_ref, lse_ref, _ = oracle.fwd_rows(qf, kf, vf, w.causal, rows)
    dq_ref, _, _ = oracle.bwd_rows(qf, kf, vf, dOf, w.causal, rows, np.zeros(0, np.int32))
    dk_ref, dv_ref, groups = _oracle_key_grads(w, qf, kf, vf, dOf, k_rows)
    note(f"{w.name}: fp64 oracle on {rows.size} query rows and {k_rows.size} key rows "
         f"(keys from {k_lo}, kv groups {groups}): {time.perf_counter() - t0:.1f} s")
    del qf, dOf
    gi = torch.tensor(groups).long()
    for N in chunk_counts:
        o, lse, dq, dk, dv = gpu_fwd_bwd(q, k, v, dO, N, w.causal)
        ri = torch.from_numpy(rows).long().cuda()
        ki = torch.from_numpy(k_rows).long().cuda()
        assert_close(f"o N={N}", f64(o[:, :, ri]), o_ref)
        assert_close(f"lse N={N}", f64(lse[:, :, ri]), lse_ref, TOL_LSE, TOL_LSE)
        assert_close(f"dq N={N}", f64(dq[:, :, ri]), dq_ref)
        assert_close(f"dk N={N}", f64(dk[:, :, ki])[:, gi], dk_ref[:, gi])
        assert_close(f"dv N={N}", f64(dv[:, :, ki])[:, gi], dv_ref[:, gi])
        del o, lse, dq, dk, dv
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["encoder", "decoder_mha", "gqa_32k"])
def test_workload_sampled_parity(name):
    w = inputs.WORKLOADS[name]
    _sampled_parity(w, sorted({1, 2, 4, w.n_chunks}))


def test_workload_128k_sampled_parity():
    """The long-context workload at full size, in the benchmark's launch
    configuration (same entry points, same shapes, same chunk count)."""
    w = inputs.WORKLOADS["gqa_128k"]
    _sampled_parity(w, [w.n_chunks])


def test_past_two_to_the_31_elements():
    """Causal GQA with 136 query heads of 131072 rows at d = 128: q, o, dO and
    dq hold 2.28e9 elements each, past 2^31 (the fp32 dQ accumulator 9.1
    GB), so any 32-bit element index on the path would wrap.  o, lse and dq
    on the sampled rows of heads 0, 127, 128 (whose first element is element
    2^31) and 135 against the fp64 oracle, which draws those heads again on
    the CPU from their own seeds."""
    B, Hq, Hkv, L, d, N, causal = 1, 136, 8, 131072, 128, 32, True
    assert Hq * L * d > 2 ** 31
    seed = 2 ** 31 % 1000
    q, k, v, dO = inputs.make_inputs_by_head(B, Hq, Hkv, L, d, seed, "cuda")
    o, lse = ra.ring_attn_fwd(q, k, v, N, causal)
    dq, dk, dv = ra.ring_attn_bwd(q, k, v, o, lse, dO, N, causal)
    torch.cuda.synchronize()
    assert_status_ok()
    del q, k, v, dO, dk, dv
    rows = inputs.sample_rows(L, N, causal, 64, seed)
    ri = torch.from_numpy(rows).long().cuda()
    G = Hq // Hkv
    for h in (0, 127, 128, 135):
        g = h // G
        one = lambda t, hh: inputs.head_rows(L, d, inputs.head_seed(seed, t, 0, hh)).double().numpy()[None, None]  # noqa: E731
        qh, kg, vg, dOh = one(0, h), one(1, g), one(2, g), one(3, h)
        o_ref, lse_ref, _ = oracle.fwd_rows(qh, kg, vg, causal, rows)
        dq_ref, _, _ = oracle.bwd_rows(qh, kg, vg, dOh, causal, rows, np.zeros(0, np.int32))
        assert_close(f"o head {h}", f64(o[:, h:h + 1, ri]), o_ref)
        assert_close(f"lse head {h}", f64(lse[:, h:h + 1, ri]), lse_ref, TOL_LSE, TOL_LSE)
        assert_close(f"dq head {h}", f64(dq[:, h:h + 1, ri]), dq_ref)


def test_tiny_workload_full_parity():
    w = inputs.WORKLOADS["tiny"]
    q, k, v, dO = inputs.workload_inputs(w)
    o, lse, dq, dk, dv = gpu_fwd_bwd(q, k, v, dO, w.n_chunks, w.causal)
    o_ref, lse_ref = oracle.fwd(f64(q), f64(k), f64(v), w.causal)
    dq_ref, dk_ref, dv_ref, _, _ = oracle.bwd(f64(q), f64(k), f64(v), f64(dO), w.causal)
    for name, g, r in (("o", o, o_ref), ("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        assert_close(name, f64(g), r)
    assert_close("lse", f64(lse), lse_ref, TOL_LSE, TOL_LSE)
