"""Pins of the oracle's blockwise-FFN routine (CPU).

The BPT section of the pages ("Large-scale distributed AI model training
series: sequence parallelism", section 4.2) runs, for each query block,
attention and then the FFN with its residual connection; the FFN is the
GPT-style two linear layers with a 4x up-projection (section 8).  The oracle
computes y = x + gelu(x W1 + b1) W2 + b2 with the exact GELU.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _weights(D, F, seed):
    rng = np.random.default_rng(seed)
    w1 = rng.standard_normal((D, F)) / math.sqrt(D)
    w2 = rng.standard_normal((F, D)) / math.sqrt(F)
    return w1, rng.standard_normal(F) * 0.1, w2, rng.standard_normal(D) * 0.1


@pytest.mark.parametrize("M,D,F", [(7, 16, 64), (33, 24, 96)])
def test_ffn_matches_torch(M, D, F):
    """Library special case: torch in fp64 (erf GELU, matmul)."""
    rng = np.random.default_rng(M)
    x = rng.standard_normal((M, D))
    w1, b1, w2, b2 = _weights(D, F, M + 1)
    got = oracle.ffn(x, w1, b1, w2, b2)
    tx = torch.tensor(x)
    h = torch.nn.functional.gelu(tx @ torch.tensor(w1) + torch.tensor(b1), approximate="none")
    want = (tx + h @ torch.tensor(w2) + torch.tensor(b2)).numpy()
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_gelu_odd_part_closed_form():
    """gelu(a) - gelu(-a) = a exactly (a Phi(a) + a Phi(-a) = a): with hidden
    units a and -a weighted +1 and -1 the block adds its pre-activation."""
    rng = np.random.default_rng(3)
    M, D = 9, 5
    x = rng.standard_normal((M, D)) * 3
    u = rng.standard_normal(D)
    w1 = np.stack([u, -u], axis=1)          # [D, 2]: a = x.u, then -a
    b1 = np.zeros(2)
    w2 = np.zeros((2, D))
    w2[0, :] = 1.0
    w2[1, :] = -1.0
    b2 = rng.standard_normal(D)
    y = oracle.ffn(x, w1, b1, w2, b2)
    want = x + (x @ u)[:, None] + b2
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


def test_zero_second_layer_leaves_the_residual():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 8))
    w1, b1, _, b2 = _weights(8, 32, 5)
    y = oracle.ffn(x, w1, b1, np.zeros((32, 8)), b2)
    np.testing.assert_array_equal(y, x + b2)


def test_gelu_values():
    """A single hidden unit exposes gelu: gelu(0) = 0, gelu(x) -> x for large
    x, -> 0 for very negative x; gelu(1) = Phi(1) = 0.841344746..."""
    for a, want in ((0.0, 0.0), (1.0, 0.8413447460685429), (12.0, 12.0), (-12.0, 0.0)):
        y = oracle.ffn(np.array([[a]]), np.array([[1.0]]), np.zeros(1), np.array([[1.0]]), np.zeros(1))
        assert abs(y[0, 0] - (a + want)) < 1e-13


def test_gelu_tail_keeps_relative_accuracy():
    """Far below zero gelu(a) = a Phi(a) is tiny but not zero: the hidden
    output matches a 40-digit evaluation of a erfc(-a / sqrt 2) / 2 to 1e-12
    relative down to a = -30 (where Phi is 5e-198)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    for a in (-3.0, -8.0, -8.5, -10.0, -20.0, -30.0):
        _, h = oracle.ffn(np.array([[a]]), np.array([[1.0]]), np.zeros(1), np.array([[1.0]]), np.zeros(1),
                          hidden=True)
        want = float(mpmath.mpf(a) * mpmath.erfc(-mpmath.mpf(a) / mpmath.sqrt(2)) / 2)
        assert want < 0 and abs(h[0, 0] / want - 1) < 1e-12, (a, h[0, 0], want)


def test_hidden_activation_and_row_subsets():
    """The hidden output is gelu(x W1 + b1) (torch fp64, erf GELU) and
    feeds y; a row subset gives exactly those rows of the full result."""
    rng = np.random.default_rng(6)
    M, D, F = 11, 12, 40
    x = rng.standard_normal((M, D))
    w1, b1, w2, b2 = _weights(D, F, 7)
    y, h = oracle.ffn(x, w1, b1, w2, b2, hidden=True)
    th = torch.nn.functional.gelu(torch.tensor(x) @ torch.tensor(w1) + torch.tensor(b1), approximate="none")
    np.testing.assert_allclose(h, th.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(y, x + h @ w2 + b2, rtol=0, atol=1e-12)
    rows = [10, 0, 4, 4]
    ys, hs = oracle.ffn(x, w1, b1, w2, b2, rows=rows, hidden=True)
    np.testing.assert_array_equal(ys, y[rows])
    np.testing.assert_array_equal(hs, h[rows])


def _problem(M, D, F, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, D))
    w1, b1, w2, b2 = _weights(D, F, seed + 1)
    dy = rng.standard_normal((M, D))
    return x, w1, b1, w2, b2, dy


@pytest.mark.parametrize("M,D,F", [(5, 8, 24), (13, 12, 40)])
def test_ffn_backward_matches_torch_autograd(M, D, F):
    """Library special case: torch autograd in fp64 through the exact GELU."""
    x, w1, b1, w2, b2, dy = _problem(M, D, F, M)
    got = oracle.ffn_bwd(x, w1, b1, w2, dy)
    tx, tw1, tb1, tw2, tb2 = (torch.tensor(a, requires_grad=True) for a in (x, w1, b1, w2, b2))
    y = tx + torch.nn.functional.gelu(tx @ tw1 + tb1, approximate="none") @ tw2 + tb2
    (y * torch.tensor(dy)).sum().backward()
    for name, g, t in zip(("dx", "dW1", "db1", "dW2", "db2"), got, (tx, tw1, tb1, tw2, tb2)):
        np.testing.assert_allclose(g, t.grad.numpy(), rtol=0, atol=1e-11, err_msg=name)


def test_ffn_backward_finite_differences():
    """Central differences of the oracle's own forward (loss sum(dy * y)) on a
    few entries of every argument."""
    M, D, F = 4, 6, 16
    x, w1, b1, w2, b2, dy = _problem(M, D, F, 9)
    grads = dict(zip(("x", "w1", "b1", "w2", "b2"), oracle.ffn_bwd(x, w1, b1, w2, dy)))
    args = {"x": x, "w1": w1, "b1": b1, "w2": w2, "b2": b2}
    loss = lambda a: float((oracle.ffn(a["x"], a["w1"], a["b1"], a["w2"], a["b2"]) * dy).sum())  # noqa: E731
    rng = np.random.default_rng(10)
    step = 1e-6
    for name, arr in args.items():
        for _ in range(4):
            idx = tuple(int(rng.integers(n)) for n in arr.shape)
            plus = {k: v.copy() for k, v in args.items()}
            minus = {k: v.copy() for k, v in args.items()}
            plus[name][idx] += step
            minus[name][idx] -= step
            fd = (loss(plus) - loss(minus)) / (2 * step)
            assert abs(fd - grads[name][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grads[name][idx])


def test_ffn_backward_with_zero_second_layer():
    """W2 = 0: no gradient reaches the first layer; dx = dy, dW2 = h^T dy with
    h = gelu(x W1 + b1), db2 = the column sums of dy."""
    M, D, F = 7, 5, 12
    x, w1, b1, _, _, dy = _problem(M, D, F, 11)
    dx, dw1, db1, dw2, db2 = oracle.ffn_bwd(x, w1, b1, np.zeros((F, D)), dy)
    assert np.array_equal(dx, dy) and not dw1.any() and not db1.any()
    h = torch.nn.functional.gelu(torch.tensor(x @ w1 + b1), approximate="none").numpy()
    np.testing.assert_allclose(dw2, h.T @ dy, rtol=0, atol=1e-12)
    np.testing.assert_allclose(db2, dy.sum(axis=0), rtol=0, atol=1e-12)


def test_ffn_backward_hidden_outputs():
    """The returned h is the forward's hidden activation and sum_m da is db1."""
    x, w1, b1, w2, b2, dy = _problem(6, 8, 20, 12)
    dx, dw1, db1, dw2, db2, h, da = oracle.ffn_bwd(x, w1, b1, w2, dy, hidden=True)
    _, h_fwd = oracle.ffn(x, w1, b1, w2, b2, hidden=True)
    np.testing.assert_array_equal(h, h_fwd)
    np.testing.assert_allclose(da.sum(axis=0), db1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(x.T @ da, dw1, rtol=0, atol=1e-12)
