"""Ring mode on the host (no GPU): the step planner and the argument checks
of the ring-mode entry points of include/ring_attn.h."""
import ctypes

import numpy as np
import pytest

import oracle
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import capi


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return capi.load()


def _chunk_positions(L, N, causal, r, striped=False, schedule=None):
    """Sequence positions of rank r's rows in chunk order (ascending: for the
    fold that is sub-chunk r, then sub-chunk 2N-1-r; r, r+N, ... striped;
    rows [rC, (r+1)C) for the contiguous schedules)."""
    return np.array([p for p in range(L) if oracle.owner_rank(L, N, causal, p, striped, schedule) == r])


CASES = [(1024, 4, True, False), (1024, 4, False, False), (2048, 4, True, False), (1536, 3, True, False),
         (3072, 8, False, False), (4096, 8, True, False), (1024, 4, True, True), (1536, 3, True, True),
         (2048, 8, True, True), (1024, 8, False, True)]


@pytest.mark.parametrize("L,N,causal,striped", CASES)
def test_step_plan_lists_exactly_the_visible_tile_pairs(lib, L, N, causal, striped):
    C = L // N
    nt = C // 128
    for r in range(N):
        qpos = _chunk_positions(L, N, causal, r, striped)
        for s in range(N):
            src = (r - s) % N
            kpos = _chunk_positions(L, N, causal, src, striped)
            plan = capi.step_plan(L, N, causal, s, r, striped)
            assert len(plan["visits"]) == (C + 255) // 256
            assert sorted(plan["order"].tolist()) == list(range(len(plan["visits"])))
            for u, visits in enumerate(plan["visits"]):
                listed = [kt for b, e in visits for kt in range(b, e)]
                assert listed == sorted(set(listed))
                qts = [qt for qt in (2 * u, 2 * u + 1) if qt < nt]
                want = set()
                for qt in qts:
                    qmax = qpos[qt * 128:(qt + 1) * 128].max()
                    for kt in range(nt):
                        if not causal or kpos[kt * 128:(kt + 1) * 128].min() <= qmax:
                            want.add(kt)
                assert set(listed) == want, (r, s, u)


@pytest.mark.parametrize("striped", [False, True])
@pytest.mark.parametrize("N", [2, 4, 8])
def test_fold_and_stripes_give_every_causal_step_the_same_work(lib, N, striped):
    """Section 8.2 of the pages: with the fold every rank does the same work
    at every step s > 0 (half of a chunk pair's tiles); step 0 is the
    diagonal pair.  With stripes every step is the same tile triangle."""
    L = 256 * N
    nt = L // N // 128
    works = {}
    for s in range(N):
        for r in range(N):
            qpos = _chunk_positions(L, N, True, r, striped)
            kpos = _chunk_positions(L, N, True, (r - s) % N, striped)
            plan = capi.step_plan(L, N, True, s, r, striped)
            pairs = 0  # (query tile, listed key tile) pairs with a visible position pair
            for u, visits in enumerate(plan["visits"]):
                for qt in (2 * u, 2 * u + 1):
                    if qt >= nt:
                        continue
                    qmax = qpos[qt * 128:(qt + 1) * 128].max()
                    pairs += sum(1 for b, e in visits for kt in range(b, e)
                                 if kpos[kt * 128:(kt + 1) * 128].min() <= qmax)
            works[(s, r)] = pairs
    for s in range(1, N):
        assert len({works[(s, r)] for r in range(N)}) == 1


I = ctypes.c_int
NUL = ctypes.c_void_p(0)
P256 = ctypes.c_void_p(256)


def test_step_rejects_bad_arguments(lib):
    def step(L=1024, N=4, causal=1, rank=0, src=0, d=64, ptr=P256, striped=0):
        return lib.ring_attn_fwd_step(ptr, ptr, ptr, ptr, ptr, 1, 2, 1, L, d, N, causal, striped, rank, src, NUL)
    assert step(rank=4) == capi.ERR_SHAPE
    assert step(src=-1) == capi.ERR_SHAPE
    assert step(L=1001) == capi.ERR_SHAPE                 # L % 2N
    assert step(L=1000) == capi.ERR_UNSUPPORTED           # sub-chunks of 125 rows: not whole tiles
    assert step(L=512, N=4) == capi.ERR_UNSUPPORTED       # sub-chunks of 64 rows
    assert step(L=512, N=4, causal=0, ptr=NUL) == capi.ERR_NULL  # chunks of 128 rows: whole tiles
    assert step(d=96) == capi.ERR_UNSUPPORTED
    assert step(ptr=ctypes.c_void_p(8)) == capi.ERR_UNSUPPORTED
    assert lib.ring_attn_fwd_step(NUL, NUL, NUL, NUL, NUL, 0, 2, 1, 1024, 64, 4, 1, 0, 0, 0, NUL) == capi.OK
    # stripes need L % N only, and chunks of whole tiles
    assert step(L=1536, N=4) == capi.ERR_UNSUPPORTED                     # fold: sub-chunks of 192 rows
    assert step(L=1536, N=4, striped=1, ptr=NUL) == capi.ERR_NULL        # stripes: chunks of 384 rows
    assert step(L=1280, N=5, striped=1, ptr=NUL) == capi.ERR_NULL        # L % 2N != 0 is fine for stripes
    assert step(L=1000, N=4, striped=1) == capi.ERR_UNSUPPORTED          # chunks of 250 rows
    assert step(L=1001, N=4, striped=1) == capi.ERR_SHAPE                # L % N



def test_merge_rejects_bad_arguments(lib):
    assert lib.ring_attn_merge(P256, P256, P256, P256, -1, 128, NUL, NUL) == capi.ERR_SHAPE
    assert lib.ring_attn_merge(P256, P256, P256, P256, 10, 96, NUL, NUL) == capi.ERR_UNSUPPORTED
    assert lib.ring_attn_merge(NUL, P256, P256, P256, 10, 128, NUL, NUL) == capi.ERR_NULL
    assert lib.ring_attn_merge(P256, P256, P256, P256, 10, 128, ctypes.c_void_p(4), NUL) == capi.ERR_UNSUPPORTED
    assert lib.ring_attn_merge(NUL, NUL, NUL, NUL, 0, 128, NUL, NUL) == capi.OK


def test_ring_fwd_workspace_and_arguments(lib):
    ws = lib.ring_attn_ring_fwd_workspace_size(1, 2, 1, 1024, 64, 4, 1, 0)
    # q, k, v in chunk order (bf16) and the running result (fp32 o + lse)
    rows_q, rows_kv = 2 * 1024, 1024
    assert ws == rows_q * 64 * 2 + 2 * rows_kv * 64 * 2 + rows_q * 64 * 4 + rows_q * 4
    assert lib.ring_attn_ring_fwd_workspace_size(1, 2, 1, 512, 64, 4, 1, 0) == 0  # not whole tiles
    assert lib.ring_attn_ring_fwd_workspace_size(1, 2, 1, 512, 64, 4, 1, 1) == ws // 2  # stripes of 128 rows
    args = [P256] * 5
    assert lib.ring_attn_ring_fwd(*args, 1, 2, 1, 1024, 64, 4, 1, 0, NUL, ws, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_ring_fwd(*args, 1, 2, 1, 1024, 64, 4, 1, 0, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_ring_fwd(*args, 1, 2, 1, 1024, 64, 4, 1, 0, ctypes.c_void_p(272), ws, NUL) == \
        capi.ERR_WORKSPACE
    assert lib.ring_attn_ring_fwd(*([NUL] * 5), 1, 2, 1, 1024, 64, 4, 1, 0, P256, ws, NUL) == capi.ERR_NULL


def test_ulysses_rejects_bad_arguments(lib):
    ws = lib.ring_attn_ulysses_workspace_size(1, 4, 2, 512, 64, 2, 1)
    assert ws > 0
    assert lib.ring_attn_ulysses_workspace_size(1, 6, 3, 512, 64, 4, 1) == 0   # heads do not split
    assert lib.ring_attn_ulysses_workspace_size(1, 8, 2, 512, 64, 4, 1) == 0   # kv heads do not split
    assert lib.ring_attn_ulysses_workspace_size(1, 4, 4, 510, 64, 4, 1) == 0   # tokens do not split
    args = [P256] * 5
    assert lib.ring_attn_ulysses_fwd(*args, 1, 4, 2, 512, 64, 0, 1, P256, ws, NUL) == capi.ERR_SHAPE
    assert lib.ring_attn_ulysses_fwd(*([NUL] * 5), 1, 4, 2, 512, 64, 2, 1, P256, ws, NUL) == capi.ERR_NULL
    assert lib.ring_attn_ulysses_fwd(*args, 1, 4, 2, 512, 64, 2, 1, NUL, ws, NUL) == capi.ERR_WORKSPACE
    bargs = [P256] * 9
    assert lib.ring_attn_ulysses_bwd(*bargs, 1, 4, 2, 512, 64, 2, 1, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_ulysses_bwd(*bargs, 1, 4, 2, 512, 96, 2, 1, P256, ws, NUL) == capi.ERR_UNSUPPORTED


def test_ring_bwd_workspace_and_arguments(lib):
    ws = lib.ring_attn_ring_bwd_workspace_size(1, 2, 1, 1024, 64, 4, 1, 0)
    rows_q, rows_kv = 2 * 1024, 1024
    # q, o, dO, k, v in chunk order (bf16); lse, -lse log2 e, -D; fp32 dq, dk, dv accumulators
    assert ws == 3 * rows_q * 64 * 2 + 2 * rows_kv * 64 * 2 + 3 * rows_q * 4 + rows_q * 64 * 4 + 2 * rows_kv * 64 * 4
    assert lib.ring_attn_ring_bwd_workspace_size(1, 2, 1, 512, 64, 4, 1, 0) == 0  # not whole tiles
    args = [P256] * 9
    assert lib.ring_attn_ring_bwd(*args, 1, 2, 1, 1024, 64, 4, 1, 0, NUL, ws, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_ring_bwd(*args, 1, 2, 1, 1024, 64, 4, 1, 0, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_ring_bwd(*([NUL] * 9), 1, 2, 1, 1024, 64, 4, 1, 0, P256, ws, NUL) == capi.ERR_NULL


def test_usp_workspace_and_arguments(lib):
    # (B, Hq, Hkv, L, d, U, R, causal)
    assert lib.ring_attn_usp_workspace_size(1, 4, 2, 512, 64, 2, 1, 1) == lib.ring_attn_ulysses_workspace_size(
        1, 4, 2, 512, 64, 2, 1)
    assert lib.ring_attn_usp_workspace_size(1, 4, 2, 1024, 64, 2, 2, 1) > 0
    assert lib.ring_attn_usp_workspace_size(1, 4, 2, 1028, 64, 2, 2, 1) == 0   # causal ring: L % 2UR
    assert lib.ring_attn_usp_workspace_size(1, 6, 3, 1024, 64, 4, 2, 1) == 0   # heads do not split by U
    assert lib.ring_attn_usp_workspace_size(1, 4, 2, 1024, 64, 2, 0, 1) == 0   # no ring groups
    ws = lib.ring_attn_usp_workspace_size(1, 4, 2, 1024, 64, 2, 2, 1)
    args = [P256] * 5
    assert lib.ring_attn_usp_fwd(*args, 1, 4, 2, 1024, 64, 0, 2, 1, P256, ws, NUL) == capi.ERR_SHAPE
    assert lib.ring_attn_usp_fwd(*([NUL] * 5), 1, 4, 2, 1024, 64, 2, 2, 1, P256, ws, NUL) == capi.ERR_NULL
    assert lib.ring_attn_usp_fwd(*args, 1, 4, 2, 1024, 64, 2, 2, 1, NUL, ws, NUL) == capi.ERR_WORKSPACE
    bargs = [P256] * 9
    assert lib.ring_attn_usp_bwd(*bargs, 1, 4, 2, 1024, 64, 2, 2, 1, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_usp_bwd(*bargs, 1, 4, 2, 1024, 96, 2, 2, 1, P256, ws, NUL) == capi.ERR_UNSUPPORTED


# ------------------------------------------------ schedules (DistFlashAttention)

@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 16, 32])
def test_schedule_pairs_match_the_oracle(lib, N):
    """The library's schedule (include/ring_attn.h) against the oracle's
    reading of the pages: DistFlashAttention's launches (section 7.2), and
    ring steps (w, (w - s) mod N) for the ring schedules."""
    assert capi.schedule_pairs(N, "dfa") == oracle.dfa_schedule(N)
    assert capi.schedule_launches(N, "dfa") == N // 2 + 1
    for sched in ("fold", "striped", "contiguous"):
        assert capi.schedule_launches(N, sched) == N
        assert capi.schedule_pairs(N, sched) == [[(w, w, (w - s) % N) for w in range(N)] for s in range(N)]


DFA_CASES = [(1024, 4), (1280, 5), (2048, 8), (768, 3), (256, 2)]


@pytest.mark.parametrize("schedule", ["contiguous", "dfa"])
@pytest.mark.parametrize("L,N", DFA_CASES)
def test_contiguous_step_plans_list_exactly_the_visible_tile_pairs(lib, L, N, schedule):
    C = L // N
    nt = C // 128
    pairs = {(t, w): (a, b) for t, launch in enumerate(capi.schedule_pairs(N, schedule)) for w, a, b in launch}
    for t in range(capi.schedule_launches(N, schedule)):
        for w in range(N):
            plan = capi.step_plan(L, N, True, t, w, schedule=schedule)
            assert len(plan["visits"]) == (C + 255) // 256
            if (t, w) not in pairs:  # idle worker: nothing listed
                assert all(not v for v in plan["visits"])
                continue
            a, b = pairs[(t, w)]
            qpos = _chunk_positions(L, N, True, a, schedule=schedule)
            kpos = _chunk_positions(L, N, True, b, schedule=schedule)
            assert np.array_equal(qpos, np.arange(a * C, (a + 1) * C))
            for u, visits in enumerate(plan["visits"]):
                listed = [kt for lo, hi in visits for kt in range(lo, hi)]
                want = set()
                for qt in (2 * u, 2 * u + 1):
                    if qt >= nt:
                        continue
                    qmax = qpos[qt * 128:(qt + 1) * 128].max()
                    want |= {kt for kt in range(nt) if kpos[kt * 128:(kt + 1) * 128].min() <= qmax}
                assert listed == sorted(want), (t, w, u)


@pytest.mark.parametrize("N", [2, 3, 4, 8])
def test_dfa_launches_after_the_first_give_every_busy_worker_a_whole_block(lib, N):
    """After the diagonal launch every busy worker runs one whole C x C block
    (its key chunk lies before its query chunk), so the launches are
    balanced; the plain contiguous ring leaves worker w idle from step w + 1
    on (the waiting the pages' figure shows)."""
    L = 256 * N
    nt = L // N // 128
    for t in range(1, N // 2 + 1):
        for w in range(N):
            plan = capi.step_plan(L, N, True, t, w, schedule="dfa")
            listed = sum(hi - lo for v in plan["visits"] for lo, hi in v)
            busy = w >= t or t < N - t
            assert listed == (nt if busy else 0)  # the block's one 256-row item visits every key tile
    for s in range(N):
        for w in range(N):
            plan = capi.step_plan(L, N, True, s, w, schedule="contiguous")
            listed = sum(hi - lo for v in plan["visits"] for lo, hi in v)
            assert (listed > 0) == (s <= w)


def test_contiguous_schedules_reject_bad_arguments(lib):
    def step(L=1024, N=4, causal=1, sched=3, ptr=P256):
        return lib.ring_attn_fwd_step(ptr, ptr, ptr, ptr, ptr, 1, 2, 1, L, 64, N, causal, sched, 0, 0, NUL)
    assert step(causal=0) == capi.ERR_UNSUPPORTED           # defined for causal attention only
    assert step(causal=0, sched=2) == capi.ERR_UNSUPPORTED
    assert step(sched=4) == capi.ERR_UNSUPPORTED
    assert step(L=1280, N=5, ptr=NUL) == capi.ERR_NULL      # L % N suffices (chunks of 256 rows)
    assert step(L=600, N=5) == capi.ERR_UNSUPPORTED          # chunks of 120 rows: not whole tiles
    assert lib.ring_attn_schedule_launches(0, 3) == capi.ERR_SHAPE
    a, b = ctypes.c_int(), ctypes.c_int()
    assert lib.ring_attn_schedule_pair(4, 3, 3, 0, ctypes.byref(a), ctypes.byref(b)) == capi.ERR_SHAPE
    assert lib.ring_attn_schedule_pair(4, 3, 2, 0, ctypes.byref(a), ctypes.byref(b)) == 0   # middle launch: idle
    assert lib.ring_attn_schedule_pair(4, 3, 1, 0, ctypes.byref(a), ctypes.byref(b)) == 1
    assert (a.value, b.value) == (3, 0)
    assert lib.ring_attn_ring_fwd_workspace_size(1, 2, 1, 1280, 64, 5, 1, 3) > 0
    assert lib.ring_attn_ring_fwd_workspace_size(1, 2, 1, 1280, 64, 5, 0, 3) == 0


def test_rank_backward_workspace_and_arguments(lib):
    # statistics (2 floats a row) and the fp32 dQ accumulator of the rank's rows
    ws = lib.ring_attn_bwd_rank_workspace_size(1, 2, 1, 1024, 64, 4, 1, 0)
    rows = 2 * 256
    assert ws == rows * 4 * 2 + rows * 64 * 4
    assert lib.ring_attn_bwd_rank_workspace_size(1, 2, 1, 512, 64, 4, 1, 0) == 0    # sub-chunks of 64 rows
    assert lib.ring_attn_bwd_rank_workspace_size(1, 2, 1, 1024, 64, 4, 0, 3) == 0   # DistFlashAttention needs causal
    I, P = ctypes.c_int, ctypes.c_void_p
    args = (1, 2, 1, 1024, 64, 4, 1, 0)
    assert lib.ring_attn_bwd_rank_begin(P256, P256, P256, *args, NUL, ws, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_bwd_rank_begin(P256, P256, P256, *args, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_bwd_rank_begin(NUL, P256, P256, *args, P256, ws, NUL) == capi.ERR_NULL
    six = [P256] * 6
    assert lib.ring_attn_bwd_rank_step(*six, *args, 4, 0, P256, ws, NUL) == capi.ERR_SHAPE   # rank out of range
    assert lib.ring_attn_bwd_rank_step(*([NUL] * 6), *args, 0, 0, P256, ws, NUL) == capi.ERR_NULL
    assert lib.ring_attn_bwd_rank_step(*six[:5], ctypes.c_void_p(8), *args, 0, 0, P256, ws, NUL) == \
        capi.ERR_UNSUPPORTED
    assert lib.ring_attn_bwd_rank_end(NUL, *args, P256, ws, NUL) == capi.ERR_NULL
    assert lib.ring_attn_grad_to_bf16(P256, P256, 100, ctypes.c_float(1.0), NUL) == capi.ERR_SHAPE
    assert lib.ring_attn_grad_to_bf16(NUL, P256, 128, ctypes.c_float(1.0), NUL) == capi.ERR_NULL
    assert lib.ring_attn_grad_to_bf16(NUL, NUL, 0, ctypes.c_float(1.0), NUL) == capi.OK


def test_rank_backward_dq_accumulator_and_partial_adds(lib):
    """The dQ accumulator's place in the rank workspace (DistFlashAttention's
    helpers send it to the owner), and the fp32 add's argument checks."""
    args = (1, 2, 1, 1024, 64, 4, 1, 3)
    ws = lib.ring_attn_bwd_rank_workspace_size(*args)
    off = lib.ring_attn_bwd_rank_dq_offset(*args)
    rows = 2 * 256
    assert off == 2 * rows * 4 and off % 256 == 0  # after the two per-row statistics
    assert off + rows * 64 * 4 == ws                # and runs to the workspace's end
    assert lib.ring_attn_bwd_rank_dq_offset(1, 2, 1, 1024, 64, 4, 0, 3) == 0  # rejected shape
    assert lib.ring_attn_add_f32(P256, P256, 6, NUL) == capi.ERR_SHAPE          # not a multiple of 4
    assert lib.ring_attn_add_f32(P256, P256, -4, NUL) == capi.ERR_SHAPE
    assert lib.ring_attn_add_f32(NUL, P256, 8, NUL) == capi.ERR_NULL
    assert lib.ring_attn_add_f32(ctypes.c_void_p(8), P256, 8, NUL) == capi.ERR_UNSUPPORTED
    assert lib.ring_attn_add_f32(NUL, NUL, 0, NUL) == capi.OK                   # nothing to add
