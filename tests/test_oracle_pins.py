"""Pins for the fp64 oracle: every check here compares the oracle with
something other than itself -- a library routine (torch's scaled dot product
attention and autograd, in fp64 on the CPU), finite differences, closed forms,
invariants of attention, the ring form with its log-sum-exp merge, and a
hand-worked example.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _problem(B, Hq, Hkv, L, d, seed=0, scale_in=1.0):
    rng = np.random.default_rng(seed)
    q = scale_in * _rand((B, Hq, L, d), rng)
    k = scale_in * _rand((B, Hkv, L, d), rng)
    v = _rand((B, Hkv, L, d), rng)
    dO = _rand((B, Hq, L, d), rng)
    return q, k, v, dO


def _sdpa(q, k, v, causal, dO=None):
    """Library special case: torch SDPA in fp64 with the kv heads repeated
    consecutively (head h uses kv head h // G)."""
    G = q.shape[1] // k.shape[1]
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1), is_causal=causal)
    if dO is None:
        return o.detach().numpy()
    (o * torch.tensor(dO)).sum().backward()
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


SHAPES = [
    (1, 2, 2, 17, 8),    # odd length
    (2, 4, 2, 33, 16),   # GQA, G = 2
    (1, 6, 2, 40, 32),   # GQA, G = 3
    (1, 2, 1, 64, 64),   # MQA
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_fwd_matches_torch_sdpa(shape, causal):
    q, k, v, _ = _problem(*shape, seed=sum(shape))
    o, lse = oracle.fwd(q, k, v, causal)
    ref = _sdpa(q, k, v, causal)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-10)
    assert np.all(np.isfinite(lse))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_bwd_matches_torch_autograd(shape, causal):
    q, k, v, dO = _problem(*shape, seed=7 + sum(shape))
    dq, dk, dv, lse, D = oracle.bwd(q, k, v, dO, causal)
    o_ref, dq_ref, dk_ref, dv_ref = _sdpa(q, k, v, causal, dO)
    np.testing.assert_allclose(dq, dq_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, dk_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, dv_ref, rtol=0, atol=1e-10)
    # D_i = dO_i . o_i with the library's o
    np.testing.assert_allclose(D, (dO * o_ref).sum(-1), rtol=0, atol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_finite_differences(causal):
    """Central differences (h = 1e-6) of l = sum(dO * O) through the oracle's
    own forward pin its hand-derived backward."""
    B, Hq, Hkv, L, d = 1, 2, 1, 9, 4
    q, k, v, dO = _problem(B, Hq, Hkv, L, d, seed=11)
    dq, dk, dv, _, _ = oracle.bwd(q, k, v, dO, causal)

    def loss(args):
        o, _ = oracle.fwd(args["q"], args["k"], args["v"], causal, threads=1)
        return float((o * dO).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            num[idx] = (loss({"q": q, "k": k, "v": v, name: xp})
                        - loss({"q": q, "k": k, "v": v, name: xm})) / (2 * h)
        err = np.abs(num - g).max() / max(1.0, np.abs(g).max())
        assert err <= 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    """With v = 1 every output element is sum_j P_ij, which must be 1."""
    q, k, _, _ = _problem(2, 4, 2, 50, 16, seed=3, scale_in=2.0)
    v = np.ones((2, 2, 50, 16))
    o, _ = oracle.fwd(q, k, v, causal)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [48, 96])
def test_ring_form_invariant_in_chunk_count(L, causal):
    """The ring form (per-step partial results merged by log-sum-exp) equals
    the plain definition for every chunk count N that divides the sequence."""
    q, k, v, _ = _problem(1, 4, 2, L, 16, seed=L + causal)
    o, lse = oracle.fwd(q, k, v, causal)
    parts = [n for n in range(1, L + 1) if L % (2 * n if causal else n) == 0]
    assert len(parts) >= 4
    for n in parts:
        o_r, lse_r = oracle.ring_fwd(q, k, v, causal, n)
        np.testing.assert_allclose(o_r, o, rtol=0, atol=1e-12, err_msg=f"N={n}")
        np.testing.assert_allclose(lse_r, lse, rtol=0, atol=1e-12, err_msg=f"N={n}")


def test_causal_row_zero_closed_form():
    """Row 0 of a causal model sees only key 0: o_0 = v_0, lse_0 = s_00 and
    dq_0 = 0."""
    B, Hq, Hkv, L, d = 2, 6, 3, 20, 8
    q, k, v, dO = _problem(B, Hq, Hkv, L, d, seed=5)
    o, lse = oracle.fwd(q, k, v, True)
    dq, _, _, _, _ = oracle.bwd(q, k, v, dO, True)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            g = h // G
            np.testing.assert_allclose(o[b, h, 0], v[b, g, 0], atol=1e-14)
            s00 = sum(q[b, h, 0, c] * k[b, g, 0, c] for c in range(d)) / math.sqrt(d)
            assert abs(lse[b, h, 0] - s00) < 1e-13
            np.testing.assert_allclose(dq[b, h, 0], 0.0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_closed_form(causal):
    """q = 0 makes every score 0: o_i is the mean of the visible v_j and
    lse_i = log |V(i)|."""
    B, Hq, Hkv, L, d = 1, 2, 2, 30, 8
    _, k, v, _ = _problem(B, Hq, Hkv, L, d, seed=9)
    q = np.zeros((B, Hq, L, d))
    o, lse = oracle.fwd(q, k, v, causal)
    for i in range(L):
        n = i + 1 if causal else L
        np.testing.assert_allclose(o[:, :, i], v[:, :, :n].mean(axis=2), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_mha(causal):
    """Grouped-query attention equals MHA with k, v repeated per group, and
    its dk, dv equal the group sums of the MHA gradients."""
    B, Hq, Hkv, L, d = 1, 6, 2, 24, 8
    q, k, v, dO = _problem(B, Hq, Hkv, L, d, seed=13)
    G = Hq // Hkv
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    o, lse = oracle.fwd(q, k, v, causal)
    o2, lse2 = oracle.fwd(q, kr, vr, causal)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)
    dq, dk, dv, _, _ = oracle.bwd(q, k, v, dO, causal)
    dq2, dk2, dv2, _, _ = oracle.bwd(q, kr, vr, dO, causal)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, G, L, d).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, G, L, d).sum(2), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding one vector c to every key adds q_i . c / sqrt(d) to every score
    of row i: o is unchanged and lse_i moves by exactly that amount."""
    B, Hq, Hkv, L, d = 1, 2, 1, 21, 8
    q, k, v, _ = _problem(B, Hq, Hkv, L, d, seed=17)
    c = np.random.default_rng(99).standard_normal(d)
    o, lse = oracle.fwd(q, k, v, causal)
    o2, lse2 = oracle.fwd(q, k + c, v, causal)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2 - lse, (q @ c) / math.sqrt(d), atol=1e-12)


def test_key_permutation_equivariance_encoder():
    """Without a mask, permuting key/value rows together leaves o unchanged,
    and permuting query rows permutes o and lse."""
    q, k, v, _ = _problem(1, 2, 2, 25, 8, seed=21)
    o, lse = oracle.fwd(q, k, v, False)
    perm = np.random.default_rng(5).permutation(25)
    o2, lse2 = oracle.fwd(q, k[:, :, perm], v[:, :, perm], False)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    o3, lse3 = oracle.fwd(q[:, :, perm], k, v, False)
    np.testing.assert_allclose(o3, o[:, :, perm], atol=1e-13)
    np.testing.assert_allclose(lse3, lse[:, :, perm], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_row_sampled_routines_agree_with_full(causal):
    B, Hq, Hkv, L, d = 1, 4, 2, 64, 16
    q, k, v, dO = _problem(B, Hq, Hkv, L, d, seed=23)
    o, lse = oracle.fwd(q, k, v, causal)
    dq, dk, dv, _, _ = oracle.bwd(q, k, v, dO, causal)
    rows = np.array([0, 1, 17, 31, 32, 63], dtype=np.int32)
    o_r, lse_r, _ = oracle.fwd_rows(q, k, v, causal, rows)
    np.testing.assert_array_equal(o_r, o[:, :, rows])
    np.testing.assert_array_equal(lse_r, lse[:, :, rows])
    krows = np.array([5, 40, 62, 63], dtype=np.int32)
    dq_r, dk_r, dv_r = oracle.bwd_rows(q, k, v, dO, causal, rows, krows)
    np.testing.assert_allclose(dq_r, dq[:, :, rows], atol=1e-14)
    np.testing.assert_allclose(dk_r, dk[:, :, krows], atol=1e-14)
    np.testing.assert_allclose(dv_r, dv[:, :, krows], atol=1e-14)


def _golden():
    inputs = {"q": [], "k": [], "v": [], "dO": []}
    expect = {}
    with open(os.path.join(GOLDEN, "hand_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split(None, 3)
            if parts[0] in inputs:
                inputs[parts[0]].append([float(x) for x in line.split()[1:]])
            else:
                mode, name, row, expr = parts
                expect[(mode, name, int(row))] = expr
    arr = {n: np.array(r)[None, None] for n, r in inputs.items()}
    return arr, expect


@pytest.mark.parametrize("mode", ["enc", "cau"])
def test_hand_worked_example(mode):
    arr, expect = _golden()
    causal = mode == "cau"
    o, lse = oracle.fwd(arr["q"], arr["k"], arr["v"], causal)
    dq, dk, dv, _, _ = oracle.bwd(arr["q"], arr["k"], arr["v"], arr["dO"], causal)
    E = math.e
    env = {"a": E / (E + 1), "b": 1 / (E + 1), "E": E, "log": math.log}
    got = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    n = 0
    for (m, name, row), expr in expect.items():
        if m != mode:
            continue
        want = np.array(eval(expr, {"__builtins__": {}}, env), dtype=np.float64)  # noqa: S307
        np.testing.assert_allclose(got[name][0, 0, row], want, atol=1e-14, err_msg=f"{name}[{row}]")
        n += 1
    assert n == 10


# --------------------------------------------------------------- chunk map

@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
def test_ring_visits_every_block_once_starting_at_home(N):
    for r in range(N):
        src = oracle.ring_sources(r, N)
        assert src[0] == r
        assert sorted(src) == list(range(N))
        # K/V move to the next rank each step: what r holds at step s+1 is
        # what r-1 held at step s.
        for s in range(N - 1):
            assert oracle.ring_sources(r, N)[s + 1] == oracle.ring_sources((r - 1) % N, N)[s]


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_fold_gives_every_rank_equal_causal_work(N):
    """Rank r owns sub-chunks r and 2N-1-r; every rank then owns the same
    number of visible (i, j) pairs of the causal triangle."""
    L = 2 * N * 12
    c = L // (2 * N)
    own = {r: [] for r in range(N)}
    for p in range(L):
        own[oracle.owner_rank(L, N, True, p)].append(p)
    for r in range(N):
        assert own[r] == list(range(r * c, (r + 1) * c)) + list(range((2 * N - 1 - r) * c, (2 * N - r) * c))
    work = {r: sum(i + 1 for i in own[r]) for r in range(N)}
    assert len(set(work.values())) == 1
    # the encoder map is contiguous chunks
    for p in range(L):
        assert oracle.owner_rank(L, N, False, p) == p // (L // N)
