"""Host-side tests of the C ABI library: it builds, loads, exports every
symbol include/*.h declares, rejects bad arguments before touching a GPU,
and its chunk scheduler visits exactly the visible tiles in ring order.
No GPU needed (no compute call is made).
"""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return capi.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ring_attn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("ring_attn_fwd", "ring_attn_bwd", "ring_attn_bwd_workspace_size", "ring_attn_strerror",
              "ring_attn_device_status", "ring_attn_fwd_plan", "ring_attn_bwd_plan", "ring_attn_owner_rank"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_strerror_covers_codes(lib):
    for code in range(-6, 1):
        assert capi.strerror(code) != "unknown status"
    assert capi.strerror(-99) == "unknown status"


I = ctypes.c_int
NUL = ctypes.c_void_p(0)


def _fwd(lib, B=1, Hq=2, Hkv=2, L=256, d=64, N=4, causal=0, ptr=NUL):
    return lib.ring_attn_fwd(ptr, ptr, ptr, ptr, ptr, B, Hq, Hkv, L, d, N, causal, NUL)


def test_fwd_rejects_bad_arguments_without_launching(lib):
    assert _fwd(lib) == capi.ERR_NULL                    # valid shape, null pointers
    assert _fwd(lib, Hq=3, Hkv=2) == capi.ERR_SHAPE       # Hq % Hkv
    assert _fwd(lib, d=96) == capi.ERR_UNSUPPORTED        # head dim
    assert _fwd(lib, L=250, N=4) == capi.ERR_SHAPE        # L % N
    assert _fwd(lib, L=256, N=3, causal=1) == capi.ERR_SHAPE  # L % 2N
    assert _fwd(lib, N=0) == capi.ERR_SHAPE
    assert _fwd(lib, B=-1) == capi.ERR_SHAPE
    assert _fwd(lib, B=70000) == capi.ERR_UNSUPPORTED     # too many (batch, head) pairs
    # empty problems are a no-op, even with null pointers
    assert _fwd(lib, B=0) == capi.OK
    assert _fwd(lib, L=0) == capi.OK
    # misaligned pointers are rejected before any CUDA call
    assert _fwd(lib, ptr=ctypes.c_void_p(8)) == capi.ERR_UNSUPPORTED


def test_selftest_rejects_bad_timeout_without_launching(lib):
    assert lib.ring_attn_selftest_bounded_wait(0, NUL) == capi.ERR_SHAPE
    assert lib.ring_attn_selftest_bounded_wait(10000001, NUL) == capi.ERR_SHAPE


def test_bwd_rejects_bad_arguments_and_workspace(lib):
    args = [NUL] * 9
    ws = lib.ring_attn_bwd_workspace_size(1, 2, 2, 256, 64, 4, 0)
    # rows padded to 128: lse2 + D (2 * B*Hq*Lpad fp32) + dq accumulator (fp32)
    assert ws == 2 * 2 * 256 * 4 + 2 * 256 * 64 * 4
    assert lib.ring_attn_bwd_workspace_size(1, 2, 2, 250, 64, 4, 0) == 0
    assert lib.ring_attn_bwd(*args, 1, 2, 2, 256, 64, 4, 0, NUL, 0, NUL) == capi.ERR_NULL
    fake = [ctypes.c_void_p(256)] * 9
    assert lib.ring_attn_bwd(*fake, 1, 2, 2, 256, 64, 4, 0, NUL, ws, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_bwd(*fake, 1, 2, 2, 256, 64, 4, 0, ctypes.c_void_p(512), ws - 1, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_bwd(*fake, 1, 2, 2, 256, 64, 4, 0, ctypes.c_void_p(100), ws, NUL) == capi.ERR_WORKSPACE
    assert lib.ring_attn_bwd(*args, 0, 2, 2, 256, 64, 4, 0, NUL, 0, NUL) == capi.OK


# ------------------------------------------------------------- scheduler

CASES = [(256, 4, False), (256, 1, False), (256, 2, True), (1024, 4, True), (4096, 8, False),
         (8192, 8, True), (200, 2, False), (200, 2, True), (640, 5, True), (32768, 16, True)]


@pytest.mark.parametrize("L,N,causal", CASES)
def test_owner_rank_matches_the_oracle_chunk_map(lib, L, N, causal):
    for p in sorted({0, L - 1, L // 2, L // 3, L // (2 * N), L // N - 1} | set(range(0, L, max(1, L // 97)))):
        assert capi.owner_rank(L, N, causal, p) == oracle.owner_rank(L, N, causal, p)


def _tiles(visits):
    out = []
    for b, e in visits:
        out.extend(range(b, e))
    return out


@pytest.mark.parametrize("L,N,causal", CASES)
def test_fwd_plan_covers_each_visible_tile_once_in_ring_order(lib, L, N, causal):
    plan = capi.fwd_plan(L, N, causal)
    nb = len(plan["visits"])
    assert nb == (L + 255) // 256
    assert sorted(plan["order"].tolist()) == list(range(nb))
    vis = oracle.visible_pairs(L, causal, 128)
    seen = set()
    for u, visits in enumerate(plan["visits"]):
        tiles = _tiles(visits)
        assert len(tiles) == len(set(tiles))
        q_tiles = [t for t in (2 * u, 2 * u + 1) if t * 128 < L]
        want = {kt for qt in q_tiles for (a, kt) in vis if a == qt}
        assert set(tiles) == want
        for qt in q_tiles:
            seen |= {(qt, kt) for kt in tiles if (qt, kt) in vis}
        # ring order of the rank owning the block's first row: the step index
        # (r - src) mod N never decreases, and starts at the home chunk
        r = oracle.owner_rank(L, N, causal, 256 * u)
        srcs = oracle.ring_sources(r, N)
        steps = [srcs.index(oracle.owner_rank(L, N, causal, 128 * t)) for t in tiles]
        assert steps == sorted(steps)
    assert seen == vis


@pytest.mark.parametrize("L,N,causal", CASES)
def test_bwd_plan_covers_each_visible_tile_once_in_ring_order(lib, L, N, causal):
    plan = capi.bwd_plan(L, N, causal)
    nt = (L + 127) // 128
    assert len(plan["visits"]) == nt
    vis = oracle.visible_pairs(L, causal, 128)
    seen = set()
    for kt, visits in enumerate(plan["visits"]):
        tiles = _tiles(visits)
        assert len(tiles) == len(set(tiles))
        assert set(tiles) == {qt for (qt, k2) in vis if k2 == kt}
        seen |= {(qt, kt) for qt in tiles}
        # the block travels r -> r+1 -> ...: query owners in that order
        rk = oracle.owner_rank(L, N, causal, 128 * kt)
        steps = [(oracle.owner_rank(L, N, causal, 128 * qt) - rk) % N for qt in tiles]
        assert steps == sorted(steps)
        assert steps[0] == 0 or rk not in [oracle.owner_rank(L, N, causal, 128 * qt) for qt in tiles]
    assert seen == vis


@pytest.mark.parametrize("L,N", [(8192, 8), (32768, 16), (131072, 32)])
def test_launch_order_is_longest_first(lib, L, N):
    plan = capi.fwd_plan(L, N, True)
    work = [len(_tiles(v)) for v in plan["visits"]]
    ordered = [work[u] for u in plan["order"]]
    assert ordered == sorted(ordered, reverse=True)
    assert plan["order"][0] == len(work) - 1


@pytest.mark.parametrize("L,N", [(8192, 8), (32768, 16), (131072, 32)])
def test_folded_assignment_balances_tile_work_across_ranks(lib, L, N):
    """With the fold, every rank owns the same number of (query tile, key
    tile) pairs of the causal triangle (tile granularity, chunks of whole
    tiles)."""
    plan = capi.fwd_plan(L, N, True)
    per_rank = np.zeros(N, dtype=np.int64)
    for u, visits in enumerate(plan["visits"]):
        for qt in (2 * u, 2 * u + 1):
            r = capi.owner_rank(L, N, True, 128 * qt)
            per_rank[r] += sum(1 for kt in _tiles(visits) if kt <= qt)
    assert per_rank.max() == per_rank.min()
    # without the fold (contiguous chunks) the last rank does far more work
    contiguous = np.zeros(N, dtype=np.int64)
    for qt in range(L // 128):
        contiguous[qt * 128 // (L // N)] += qt + 1
    assert contiguous.max() > 1.5 * contiguous.mean()


def test_profile_kinds_match_the_header(lib):
    """The binding's kernel-kind list has RING_ATTN_N_KERNELS entries, and a
    read with nothing recorded (no CUDA call) returns every kind at zero."""
    text = open(os.path.join(ROOT, "include", "ring_attn.h")).read()
    n = int(re.search(r"RING_ATTN_N_KERNELS\s*=\s*(\d+)", text).group(1))
    assert len(capi.KERNEL_NAMES) == n
    got = capi.profile_read()
    assert list(got) == list(capi.KERNEL_NAMES)
    assert all(v == (0.0, 0) for v in got.values())
