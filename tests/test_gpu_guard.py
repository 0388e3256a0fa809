"""Out-of-bounds writes, caught by guard bands (compute-sanitizer is not
available on this pool, so this is the check that kernels write only inside
their outputs and workspaces).

Every input, output and workspace of a call lives in a device buffer of its
own between two 4 KiB guard bands filled with seeded random bytes (the
padding after a tensor up to the next 256 bytes counts as guard too).
After the call: every guard band is byte-identical, every input is
byte-identical (except x of the in-place FFN, which is its output), and the
outputs equal those of the same call on plain allocations.  The shapes are
the ones where a clipped store or a padded accumulator would spill: ragged
L (200, 1000) with two batches, ring mode, Ulysses/USP shards, the FFN with
a ragged last block (and in place), the BPT layer, and the allocation-free
backward.
"""
import math

import pytest
import torch

import sequence_blockwise_self_gb300 as ra
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import inputs
from tolerance import check_bf16

pytestmark = pytest.mark.gpu

GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    ra.load()


class Arena:
    """Device tensors, each between guard bands of seeded random bytes."""

    def __init__(self, seed):
        self.gen = torch.Generator().manual_seed(seed)
        self.items = []

    def alloc(self, name, shape, dtype, init=None, is_input=False):
        itemsize = torch.empty((), dtype=dtype).element_size()
        n = math.prod(shape) * itemsize
        body = -(-max(n, 1) // 256) * 256
        pattern = torch.randint(0, 256, (GUARD + body + GUARD,), generator=self.gen, dtype=torch.uint8)
        raw = pattern.cuda()
        t = raw[GUARD:GUARD + n].view(dtype).view(shape)
        if init is not None:
            t.copy_(init)
        self.items.append((name, raw, pattern, n, is_input))
        return t

    def like(self, name, x, is_input=True):
        return self.alloc(name, tuple(x.shape), x.dtype, init=x, is_input=is_input)

    def workspace(self, name, nbytes):
        return self.alloc(name, (max(int(nbytes), 1),), torch.uint8)

    def check(self, changed_inputs=()):
        torch.cuda.synchronize()
        st, site = ra.device_status()
        assert st == 0, f"device status {st} at site {site:#x}"
        for name, raw, pattern, n, is_input in self.items:
            host = raw.cpu()
            front = torch.equal(host[:GUARD], pattern[:GUARD])
            back = torch.equal(host[GUARD + n:], pattern[GUARD + n:])
            assert front and back, f"{name}: guard band overwritten ({'front' if not front else 'back'})"
            if is_input and name not in changed_inputs:
                self._snap_check(name, host[GUARD:GUARD + n])

    def snapshot(self):
        torch.cuda.synchronize()
        self.snaps = {name: raw[GUARD:GUARD + n].cpu() for name, raw, _, n, is_input in self.items if is_input}

    def _snap_check(self, name, now):
        assert torch.equal(now, self.snaps[name]), f"{name}: input modified"


def _same_bf16(name, got, want):
    # the backward's fp32 reduce-adds run in a nondeterministic order: two
    # runs agree to fp32 rounding, far inside the parity bound
    check_bf16(name, got.float().cpu().double().numpy(), want.float().cpu().double().numpy(), 1e-2, 1e-3, ulps=2)


def _attn_inputs(arena, shape, seed):
    B, Hq, Hkv, L, d = shape
    q, k, v, dO = (t.cuda() for t in inputs.make_inputs(B, Hq, Hkv, L, d, seed=seed))
    return (q, k, v, dO), tuple(arena.like(n, t) for n, t in zip(("q", "k", "v", "dO"), (q, k, v, dO)))


# (B, Hq, Hkv, L, d, n_chunks, causal)
FUSED = [(2, 4, 2, 1000, 64, 5, True), (2, 2, 2, 200, 128, 2, False), (1, 3, 1, 1000, 128, 5, True)]


@pytest.mark.parametrize("shape", FUSED, ids=lambda s: "B{}H{}-{}L{}d{}N{}{}".format(*s[:6], "c" if s[6] else "e"))
def test_fused_forward_backward_stay_in_bounds(shape):
    B, Hq, Hkv, L, d, N, causal = shape
    arena = Arena(seed=L + d)
    (q, k, v, dO), (gq, gk, gv, gdO) = _attn_inputs(arena, (B, Hq, Hkv, L, d), seed=900 + L)
    o_ref, lse_ref = ra.ring_attn_fwd(q, k, v, N, causal)
    dq_ref, dk_ref, dv_ref = ra.ring_attn_bwd(q, k, v, o_ref, lse_ref, dO, N, causal)

    o = arena.alloc("o", (B, Hq, L, d), torch.bfloat16)
    lse = arena.alloc("lse", (B, Hq, L), torch.float32)
    dq = arena.alloc("dq", (B, Hq, L, d), torch.bfloat16)
    dk = arena.alloc("dk", (B, Hkv, L, d), torch.bfloat16)
    dv = arena.alloc("dv", (B, Hkv, L, d), torch.bfloat16)
    ws = arena.workspace("workspace", ra.bwd_workspace_size(B, Hq, Hkv, L, d, N, causal))
    arena.snapshot()
    ra.ring_attn_fwd(gq, gk, gv, N, causal, o=o, lse=lse)
    ra.ring_attn_bwd(gq, gk, gv, o, lse, gdO, N, causal, dq=dq, dk=dk, dv=dv, workspace=ws)
    arena.check()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    for name, a, b in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        _same_bf16(name, a, b)

    # the allocation-free backward writes only its three outputs
    arena2 = Arena(seed=L + d + 1)
    ins = [arena2.like(n, t) for n, t in zip(("q", "k", "v", "o", "lse", "dO"), (q, k, v, o_ref, lse_ref, dO))]
    grads = [arena2.alloc(n, tuple(t.shape), torch.bfloat16) for n, t in (("dq", q), ("dk", k), ("dv", v))]
    arena2.snapshot()
    ra.ring_attn_bwd_noalloc(*ins, N, causal, *grads)
    arena2.check()
    for name, a, b in zip(("dq", "dk", "dv"), grads, (dq_ref, dk_ref, dv_ref)):
        _same_bf16(name, a, b)


# (B, Hq, Hkv, L, d, n_chunks, causal, schedule)
RING = [(2, 4, 2, 1024, 128, 4, True, "fold"), (1, 2, 2, 768, 64, 3, False, "fold"),
        (2, 2, 1, 768, 128, 3, True, "striped"), (2, 2, 1, 1280, 64, 5, True, "dfa")]


@pytest.mark.parametrize("shape", RING, ids=lambda s: "B{}H{}-{}L{}d{}N{}{}-{}".format(
    *s[:6], "c" if s[6] else "e", s[7]))
def test_ring_mode_stays_in_bounds(shape):
    B, Hq, Hkv, L, d, N, causal, schedule = shape
    arena = Arena(seed=7 + L)
    (q, k, v, dO), (gq, gk, gv, gdO) = _attn_inputs(arena, (B, Hq, Hkv, L, d), seed=910 + L)
    o_ref, lse_ref = ra.ring_attn_ring_fwd(q, k, v, N, causal, schedule=schedule)
    dq_ref, dk_ref, dv_ref = ra.ring_attn_ring_bwd(q, k, v, o_ref, lse_ref, dO, N, causal, schedule=schedule)
    o = arena.alloc("o", (B, Hq, L, d), torch.bfloat16)
    lse = arena.alloc("lse", (B, Hq, L), torch.float32)
    dq = arena.alloc("dq", (B, Hq, L, d), torch.bfloat16)
    dk = arena.alloc("dk", (B, Hkv, L, d), torch.bfloat16)
    dv = arena.alloc("dv", (B, Hkv, L, d), torch.bfloat16)
    wf = arena.workspace("fwd workspace", ra.ring_fwd_workspace_size(B, Hq, Hkv, L, d, N, causal, schedule=schedule))
    wb = arena.workspace("bwd workspace", ra.ring_bwd_workspace_size(B, Hq, Hkv, L, d, N, causal, schedule=schedule))
    arena.snapshot()
    ra.ring_attn_ring_fwd(gq, gk, gv, N, causal, o=o, lse=lse, workspace=wf, schedule=schedule)
    ra.ring_attn_ring_bwd(gq, gk, gv, o, lse, gdO, N, causal, dq=dq, dk=dk, dv=dv, workspace=wb, schedule=schedule)
    arena.check()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    for name, a, b in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        _same_bf16(name, a, b)


# (B, Hq, Hkv, L, d, ulysses degree U, ring degree R, causal)
USP = [(2, 4, 2, 512, 128, 2, 1, True), (1, 4, 2, 1024, 64, 2, 2, True), (1, 4, 4, 384, 128, 4, 1, False)]


@pytest.mark.parametrize("shape", USP, ids=lambda s: "B{}H{}-{}L{}d{}U{}R{}{}".format(*s[:7], "c" if s[7] else "e"))
def test_ulysses_usp_stay_in_bounds(shape):
    B, Hq, Hkv, L, d, U, R, causal = shape
    N = U * R
    C = L // N
    arena = Arena(seed=11 + L + U)
    gen = torch.Generator().manual_seed(920 + L)
    mk = lambda H: torch.randn((N, B, H, C, d), generator=gen).to(torch.bfloat16).cuda()  # noqa: E731
    q, k, v, dO = mk(Hq), mk(Hkv), mk(Hkv), mk(Hq)
    gq, gk, gv, gdO = (arena.like(n, t) for n, t in zip(("q", "k", "v", "dO"), (q, k, v, dO)))
    o_ref, lse_ref = ra.ring_attn_usp_fwd(q, k, v, U, causal)
    dq_ref, dk_ref, dv_ref = ra.ring_attn_usp_bwd(q, k, v, o_ref, lse_ref, dO, U, causal)
    o = arena.alloc("o", tuple(q.shape), torch.bfloat16)
    lse = arena.alloc("lse", (N, B, Hq, C), torch.float32)
    dq = arena.alloc("dq", tuple(q.shape), torch.bfloat16)
    dk = arena.alloc("dk", tuple(k.shape), torch.bfloat16)
    dv = arena.alloc("dv", tuple(v.shape), torch.bfloat16)
    ws = arena.workspace("workspace", ra.usp_workspace_size(B, Hq, Hkv, L, d, U, R, causal))
    arena.snapshot()
    ra.ring_attn_usp_fwd(gq, gk, gv, U, causal, o=o, lse=lse, workspace=ws)
    ra.ring_attn_usp_bwd(gq, gk, gv, o, lse, gdO, U, causal, dq=dq, dk=dk, dv=dv, workspace=ws)
    arena.check()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    for name, a, b in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        _same_bf16(name, a, b)


@pytest.mark.parametrize("in_place", [False, True], ids=["y", "in_place"])
def test_ffn_stays_in_bounds(in_place):
    M, D, F, R = 1000, 256, 512, 384  # last block ragged: 232 rows
    arena = Arena(seed=13 + int(in_place))
    x, w1, b1, w2, b2 = (t.cuda() for t in inputs.make_ffn_inputs(M, D, F, seed=930))
    dy = torch.randn((M, D), generator=torch.Generator().manual_seed(931)).to(torch.bfloat16).cuda()
    y_ref = ra.ring_attn_ffn_fwd(x, w1, b1, w2, b2, block_rows=R)
    g_ref = ra.ring_attn_ffn_bwd(x, w1, b1, w2, dy, block_rows=R)
    gx, gw1, gb1, gw2, gb2, gdy = (arena.like(n, t) for n, t in
                                   zip(("x", "w1", "b1", "w2", "b2", "dy"), (x, w1, b1, w2, b2, dy)))
    y = gx if in_place else arena.alloc("y", (M, D), torch.bfloat16)
    wsf = arena.workspace("fwd workspace", ra.ffn_workspace_size(D, F, R))
    wsb = arena.workspace("bwd workspace", ra.ffn_bwd_workspace_size(D, F, R))
    outs = [arena.alloc("dx", (M, D), torch.bfloat16), arena.alloc("dw1", (F, D), torch.float32),
            arena.alloc("db1", (F,), torch.float32), arena.alloc("dw2", (D, F), torch.float32),
            arena.alloc("db2", (D,), torch.float32)]
    arena.snapshot()
    ra.ring_attn_ffn_bwd(gx, gw1, gb1, gw2, gdy, block_rows=R, workspace=wsb, dx=outs[0], dw1=outs[1], db1=outs[2],
                         dw2=outs[3], db2=outs[4])
    ra.ring_attn_ffn_fwd(gx, gw1, gb1, gw2, gb2, block_rows=R, y=y, workspace=wsf)
    arena.check(changed_inputs=("x",) if in_place else ())
    assert torch.equal(y, y_ref)
    _same_bf16("dx", outs[0], g_ref[0])
    for name, a, b in zip(("dw1", "db1", "dw2", "db2"), outs[1:], g_ref[1:]):
        # fp32 sums with atomics in the column sums: agree to fp32 rounding
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-4), name


def test_bpt_stays_in_bounds():
    B, Hq, Hkv, L, d, N, causal, F, R = 2, 4, 2, 1000, 64, 4, True, 512, 512  # ragged L, two batches
    D = Hq * d
    arena = Arena(seed=17)
    q, k, v, _ = (t.cuda() if t is not None else None for t in
                  inputs.make_inputs(B, Hq, Hkv, L, d, seed=940, with_grad=False))
    _, w1, b1, w2, b2 = (t.cuda() for t in inputs.make_ffn_inputs(1, D, F, seed=941))
    dy = torch.randn((B, L, D), generator=torch.Generator().manual_seed(942)).to(torch.bfloat16).cuda()
    a_ref, lse_ref, y_ref = ra.ring_attn_bpt_fwd(q, k, v, w1, b1, w2, b2, N, causal, block_rows=R)
    g_ref = ra.ring_attn_bpt_bwd(q, k, v, a_ref, lse_ref, w1, b1, w2, dy, N, causal, block_rows=R)
    gq, gk, gv, gw1, gb1, gw2, gb2, gdy = (arena.like(n, t) for n, t in zip(
        ("q", "k", "v", "w1", "b1", "w2", "b2", "dy"), (q, k, v, w1, b1, w2, b2, dy)))
    a_tok = arena.alloc("a_tok", (B, L, D), torch.bfloat16)
    lse = arena.alloc("lse", (B, Hq, L), torch.float32)
    y = arena.alloc("y", (B, L, D), torch.bfloat16)
    wsf = arena.workspace("fwd workspace", ra.bpt_workspace_size(Hq, d, F, R))
    wsb = arena.workspace("bwd workspace", ra.bpt_bwd_workspace_size(B, Hq, Hkv, L, d, N, causal, F, R))
    outs = (arena.alloc("dq", (B, Hq, L, d), torch.bfloat16), arena.alloc("dk", (B, Hkv, L, d), torch.bfloat16),
            arena.alloc("dv", (B, Hkv, L, d), torch.bfloat16), arena.alloc("dw1", (F, D), torch.float32),
            arena.alloc("db1", (F,), torch.float32), arena.alloc("dw2", (D, F), torch.float32),
            arena.alloc("db2", (D,), torch.float32))
    arena.snapshot()
    ra.ring_attn_bpt_fwd(gq, gk, gv, gw1, gb1, gw2, gb2, N, causal, block_rows=R, a_tok=a_tok, lse=lse, y=y,
                         workspace=wsf)
    ra.ring_attn_bpt_bwd(gq, gk, gv, a_tok, lse, gw1, gb1, gw2, gdy, N, causal, block_rows=R, workspace=wsb,
                         outs=outs)
    arena.check()
    assert torch.equal(a_tok, a_ref) and torch.equal(lse, lse_ref) and torch.equal(y, y_ref)
    for name, a, b in zip(("dq", "dk", "dv"), outs[:3], g_ref[:3]):
        _same_bf16(name, a, b)
    for name, a, b in zip(("dw1", "db1", "dw2", "db2"), outs[3:], g_ref[3:]):
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-4), name
