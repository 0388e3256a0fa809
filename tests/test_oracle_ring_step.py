"""Pins of the oracle's ring-step and merge routines (CPU).

One ring step is rank r's query rows against the keys/values of rank src
("Large-scale distributed AI model training series: sequence parallelism",
section 2.3 Ring Self-Attention and section 6.2 Ring Attention); the merge
is the log-sum-exp rule that combines partial results of the same rows
(section 6.2).  They are pinned to the plain definition (every rank's steps
merged in ring order give the full attention), to the structure of the
fold (section 8.2) and to closed forms of the merge.
"""
import math

import numpy as np
import pytest

import oracle


def _problem(B, Hq, Hkv, L, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, L, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    return q, k, v


def _rows_of(L, N, causal, r, striped=False):
    return np.array([p for p in range(L) if oracle.owner_rank(L, N, causal, p, striped) == r])


@pytest.mark.parametrize("striped", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L,N", [(48, 2), (48, 3), (64, 4)])
def test_steps_merged_in_ring_order_equal_plain(L, N, causal, striped):
    if causal and not striped and L % (2 * N):
        pytest.skip("fold needs L % 2N == 0")
    q, k, v = _problem(1, 4, 2, L, 8, seed=10 * L + N + causal)
    o_ref, lse_ref = oracle.fwd(q, k, v, causal)
    for r in range(N):
        rows = _rows_of(L, N, causal, r, striped)
        o = np.zeros((1, 4, L, 8))
        lse = np.full((1, 4, L), -np.inf)
        for src in oracle.ring_sources(r, N):
            o_s, lse_s = oracle.ring_step(q, k, v, causal, N, r, src, striped=striped)
            o, lse = oracle.merge(o, lse, o_s, lse_s)
        np.testing.assert_allclose(o[:, :, rows], o_ref[:, :, rows], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, rows], lse_ref[:, :, rows], rtol=0, atol=1e-12)
        others = np.setdiff1d(np.arange(L), rows)
        assert np.all(lse[:, :, others] == -np.inf) and np.all(o[:, :, others] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_single_chunk_step_is_plain(causal):
    q, k, v = _problem(2, 2, 1, 24, 16, seed=3 + causal)
    o_ref, lse_ref = oracle.fwd(q, k, v, causal)
    o, lse = oracle.ring_step(q, k, v, causal, 1, 0, 0)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("N", [2, 3, 4])
def test_causal_fold_visibility_per_step(N):
    """With the fold, rank r's first sub-chunk (r) sees src's keys only if
    src <= r; its second sub-chunk (2N-1-r) sees every rank's keys."""
    c = 8
    L = 2 * N * c
    q, k, v = _problem(1, 1, 1, L, 4, seed=N)
    for r in range(N):
        first = np.arange(r * c, (r + 1) * c)
        second = np.arange((2 * N - 1 - r) * c, (2 * N - r) * c)
        for src in range(N):
            _, lse = oracle.ring_step(q, k, v, True, N, r, src)
            assert np.all(np.isfinite(lse[0, 0, second]))
            if src <= r:
                assert np.all(np.isfinite(lse[0, 0, first]))
            else:
                assert np.all(lse[0, 0, first] == -np.inf)


def test_merge_with_itself_adds_log2():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((5, 7))
    lse = rng.standard_normal(5) * 10
    o2, lse2 = oracle.merge(o, lse, o, lse)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse2, lse + math.log(2.0), rtol=0, atol=1e-13)


def test_merge_neutral_element():
    rng = np.random.default_rng(1)
    o = rng.standard_normal((4, 3))
    lse = rng.standard_normal(4)
    empty_o, empty_lse = np.zeros((4, 3)), np.full(4, -np.inf)
    for a, b in (((o, lse), (empty_o, empty_lse)), ((empty_o, empty_lse), (o, lse))):
        o2, lse2 = oracle.merge(*a, *b)
        assert np.array_equal(o2, o) and np.array_equal(lse2, lse)


def test_merge_weights_are_a_sigmoid_of_the_lse_gap():
    """Merging the unit vectors e0 (weight of side a) and e1 (side b) exposes
    the weights: 1 / (1 + e^(lse_b - lse_a)) and its complement."""
    gaps = np.array([-30.0, -3.0, -0.5, 0.0, 0.25, 2.0, 40.0])
    lse_a = np.full(gaps.size, 1.5)
    lse_b = lse_a + gaps
    o_a = np.tile([1.0, 0.0], (gaps.size, 1))
    o_b = np.tile([0.0, 1.0], (gaps.size, 1))
    o, lse = oracle.merge(o_a, lse_a, o_b, lse_b)
    for n, g in enumerate(gaps):
        wa = 1.0 / (1.0 + math.exp(g))
        assert abs(o[n, 0] - wa) < 1e-14 and abs(o[n, 1] - (1.0 - wa)) < 1e-14
        assert abs(lse[n] - (1.5 + math.log1p(math.exp(g)))) < 1e-12


def test_merge_is_symmetric_and_order_free():
    rng = np.random.default_rng(2)
    parts = [(rng.standard_normal((6, 5)), rng.standard_normal(6) * 3) for _ in range(4)]
    ab = oracle.merge(*parts[0], *parts[1])
    ba = oracle.merge(*parts[1], *parts[0])
    np.testing.assert_allclose(ab[0], ba[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(ab[1], ba[1], rtol=0, atol=1e-14)
    acc = parts[0]
    for p in parts[1:]:
        acc = oracle.merge(*acc, *p)
    acc2 = parts[3]
    for p in (parts[1], parts[0], parts[2]):
        acc2 = oracle.merge(*acc2, *p)
    np.testing.assert_allclose(acc[0], acc2[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(acc[1], acc2[1], rtol=0, atol=1e-13)


@pytest.mark.parametrize("L", [36, 60])
def test_striped_ring_form_invariant_in_chunk_count(L):
    """Striped attention: rank r owns positions r, r+N, ...; the ring form
    still equals the plain definition for every N dividing L."""
    q, k, v = _problem(1, 2, 1, L, 8, seed=L)
    o, lse = oracle.fwd(q, k, v, True)
    for n in [n for n in range(1, L + 1) if L % n == 0]:
        o_r, lse_r = oracle.ring_fwd(q, k, v, True, n, striped=True)
        np.testing.assert_allclose(o_r, o, rtol=0, atol=1e-12, err_msg=f"N={n}")
        np.testing.assert_allclose(lse_r, lse, rtol=0, atol=1e-12, err_msg=f"N={n}")


@pytest.mark.parametrize("N", [2, 3, 5])
def test_striped_step_with_zero_queries_closed_form(N):
    """q = 0 makes every score 0: a step's partial result is the mean of the
    visible v rows and lse_s = log(their count).  With stripes, row i of
    rank r (position r + N i) sees keys src + N j for j <= i if src <= r,
    j <= i - 1 if src > r: the same triangle at every step, one diagonal
    apart."""
    C = 7
    L = N * C
    rng = np.random.default_rng(N)
    q = np.zeros((1, 1, L, 4))
    k = rng.standard_normal((1, 1, L, 4))
    v = rng.standard_normal((1, 1, L, 4))
    for r in range(N):
        for src in range(N):
            o_s, lse_s = oracle.ring_step(q, k, v, True, N, r, src, striped=True)
            for i in range(C):
                count = i + 1 if src <= r else i
                pos = r + N * i
                if count == 0:
                    assert lse_s[0, 0, pos] == -np.inf and np.all(o_s[0, 0, pos] == 0)
                    continue
                keys = [src + N * j for j in range(count)]
                assert abs(lse_s[0, 0, pos] - math.log(count)) < 1e-13
                np.testing.assert_allclose(o_s[0, 0, pos], v[0, 0, keys].mean(axis=0), rtol=0, atol=1e-13)


# ------------------------------------------ contiguous causal chunks, DistFlashAttention

@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 9])
def test_dfa_schedule_runs_every_causal_block_once(N):
    """DistFlashAttention's balanced schedule (section 7.2): over its launches
    every block (query chunk a, key chunk b <= a) is computed exactly once,
    no worker holds two blocks in one launch, the keys a helper uses are its
    own chunk, and the launch count is N//2 + 1 -- every launch but an even
    N's middle one keeps all N workers busy (the pages' example: N = 8, 8
    ring steps become 5)."""
    sched = oracle.dfa_schedule(N)
    assert len(sched) == N // 2 + 1
    seen = []
    for t, launch in enumerate(sched):
        workers = [w for w, _, _ in launch]
        assert len(set(workers)) == len(workers)
        busy = len(launch)
        assert busy == (N // 2 if (N % 2 == 0 and t == N // 2 and N > 1) else N)
        for w, a, b in launch:
            assert b <= a
            if w != a:  # a helper: a later worker's block, on the helper's own keys
                assert b == w and a > w
            seen.append((a, b))
    want = sorted((a, b) for a in range(N) for b in range(a + 1))
    assert sorted(seen) == want
    if N == 8:
        assert len(sched) == 5


@pytest.mark.parametrize("schedule", ["contiguous", "dfa"])
@pytest.mark.parametrize("L,N", [(48, 2), (48, 3), (64, 4), (60, 5), (64, 8)])
def test_contiguous_causal_ring_forms_equal_plain(L, N, schedule):
    """Contiguous causal chunks, merged in plain ring order or in
    DistFlashAttention's launch order: the plain definition to 1e-12."""
    q, k, v = _problem(1, 4, 2, L, 8, seed=7 * L + N)
    o_ref, lse_ref = oracle.fwd(q, k, v, True)
    o, lse = oracle.ring_fwd(q, k, v, True, N, schedule=schedule)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("N", [2, 4, 5])
def test_dfa_blocks_merged_in_launch_order_equal_plain(N):
    """The launches run block by block: every block of the schedule as a ring
    step of the oracle (query chunk a against key chunk b), merged into its
    query chunk in launch order, gives the plain definition."""
    C = 6
    L = N * C
    q, k, v = _problem(1, 2, 1, L, 8, seed=N)
    o_ref, lse_ref = oracle.fwd(q, k, v, True)
    o = np.zeros((1, 2, L, 8))
    lse = np.full((1, 2, L), -np.inf)
    for launch in oracle.dfa_schedule(N):
        for _, a, b in launch:
            o_s, lse_s = oracle.ring_step(q, k, v, True, N, a, b, schedule="dfa")
            o, lse = oracle.merge(o, lse, o_s, lse_s)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("N", [2, 3, 4])
def test_contiguous_step_with_zero_queries_closed_form(N):
    """q = 0: chunk a against key chunk b < a sees all C keys of b (mean of
    them, lse = log C); against itself a prefix (row i of the chunk sees i+1
    keys); against b > a nothing (lse = -inf)."""
    C = 5
    L = N * C
    rng = np.random.default_rng(10 + N)
    q = np.zeros((1, 1, L, 4))
    k = rng.standard_normal((1, 1, L, 4))
    v = rng.standard_normal((1, 1, L, 4))
    for a in range(N):
        assert [oracle.owner_rank(L, N, True, p, schedule="dfa") for p in range(a * C, a * C + C)] == [a] * C
        for b in range(N):
            o_s, lse_s = oracle.ring_step(q, k, v, True, N, a, b, schedule="contiguous")
            for i in range(C):
                pos = a * C + i
                count = C if b < a else (i + 1 if b == a else 0)
                if count == 0:
                    assert lse_s[0, 0, pos] == -np.inf and np.all(o_s[0, 0, pos] == 0)
                    continue
                keys = list(range(b * C, b * C + count))
                assert abs(lse_s[0, 0, pos] - math.log(count)) < 1e-13
                np.testing.assert_allclose(o_s[0, 0, pos], v[0, 0, keys].mean(axis=0), rtol=0, atol=1e-13)


def test_contiguous_schedules_need_causal():
    q, k, v = _problem(1, 1, 1, 16, 4, seed=0)
    for schedule in ("contiguous", "dfa"):
        with pytest.raises(ValueError):
            oracle.ring_fwd(q, k, v, False, 2, schedule=schedule)


# ------------------------------------------------------------- backward blocks

@pytest.mark.parametrize("schedule", ["fold", "striped", "contiguous"])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_blocks_sum_to_the_plain_backward(schedule, causal):
    """Section 6.2's backward block by block: every (rank, src) block's dq
    (rank's rows) and dk, dv (src's rows), summed, equal the plain backward
    (itself pinned to torch's autograd)."""
    if schedule == "contiguous" and not causal:
        pytest.skip("the contiguous causal schedule needs causal attention")
    L, N = 48, 3
    q, k, v = _problem(1, 4, 2, L, 8, seed=41 + causal)
    dO = np.random.default_rng(42).standard_normal(q.shape)
    dq_ref, dk_ref, dv_ref, lse, D = oracle.bwd(q, k, v, dO, causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r in range(N):
        rows = _rows_of_sched(L, N, causal, r, schedule)
        for src in range(N):
            a, b, c = oracle.ring_step_bwd(q, k, v, dO, lse, D, causal, N, r, src, schedule=schedule)
            others = np.setdiff1d(np.arange(L), rows)
            assert np.all(a[:, :, others] == 0)
            dq += a
            dk += b
            dv += c
    np.testing.assert_allclose(dq, dq_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, dk_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, rtol=0, atol=1e-12)


def _rows_of_sched(L, N, causal, r, schedule):
    return np.array([p for p in range(L) if oracle.owner_rank(L, N, causal, p, schedule=schedule) == r])


def test_backward_block_a_key_chunk_after_the_queries_gives_nothing():
    """Causal, contiguous chunks: rank 0's queries see none of rank 1's keys,
    so that block contributes exactly zero to every gradient."""
    L, N = 32, 2
    q, k, v = _problem(1, 2, 1, L, 4, seed=7)
    dO = np.random.default_rng(8).standard_normal(q.shape)
    _, _, _, lse, D = oracle.bwd(q, k, v, dO, True)
    a, b, c = oracle.ring_step_bwd(q, k, v, dO, lse, D, True, N, 0, 1, schedule="contiguous")
    assert not a.any() and not b.any() and not c.any()
