"""The seeded row samplers the parity tests use (host logic, no GPU)."""
import numpy as np
import torch

from sequence_blockwise_self_gb300 import inputs


def test_sample_rows_cover_every_boundary_and_are_distinct():
    L, N = 32768, 16
    rows = inputs.sample_rows(L, N, True, 256, seed=4)
    assert rows.size == 256 and np.all(np.diff(rows) > 0)
    c = L // (2 * N)
    for i in range(2 * N):
        assert i * c in rows and (i + 1) * c - 1 in rows
    assert rows[0] == 0 and rows[-1] == L - 1


def test_sample_rows_within_a_window():
    L, N, lo = 131072, 32, 131072 - 8192
    rows = inputs.sample_rows(L, N, True, 256, seed=5, lo=lo)
    assert rows.size == 256 and rows.min() == lo and rows.max() == L - 1
    assert np.all(np.diff(rows) > 0)
    c = L // (2 * N)
    for start in range(lo, L, c):  # the window's four sub-chunks, both ends
        assert start in rows and start + c - 1 in rows
    # the same seed gives the same sample; another seed another one
    assert np.array_equal(rows, inputs.sample_rows(L, N, True, 256, seed=5, lo=lo))
    assert not np.array_equal(rows, inputs.sample_rows(L, N, True, 256, seed=6, lo=lo))


def test_sample_rows_small_range_returns_all_rows():
    assert np.array_equal(inputs.sample_rows(100, 2, False, 256, seed=0), np.arange(100))
    assert np.array_equal(inputs.sample_rows(100, 2, False, 256, seed=0, lo=60), np.arange(60, 100))


def test_inputs_by_head_are_seeded_per_head_and_redrawable():
    """The head-by-head generator: every (tensor, batch, head) slice has its
    own seed, the result is reproducible, and any head drawn again alone
    equals its slice of the whole."""
    B, Hq, Hkv, L, d = 2, 4, 2, 64, 16
    a = inputs.make_inputs_by_head(B, Hq, Hkv, L, d, 7, "cpu")
    b = inputs.make_inputs_by_head(B, Hq, Hkv, L, d, 7, "cpu")
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q, k, v, dO = a
    assert q.shape == (B, Hq, L, d) and k.shape == (B, Hkv, L, d) and dO.shape == q.shape
    assert torch.equal(q[1, 3], inputs.head_rows(L, d, inputs.head_seed(7, 0, 1, 3)))
    assert torch.equal(v[0, 1], inputs.head_rows(L, d, inputs.head_seed(7, 2, 0, 1)))
    seeds = {inputs.head_seed(7, t, bb, h) for t in range(4) for bb in range(B) for h in range(Hq)}
    assert len(seeds) == 4 * B * Hq
    assert not torch.equal(q[0, 0], dO[0, 0]) and not torch.equal(k[0, 0], v[0, 0])
    assert abs(float(q.float().mean())) < 0.05 and abs(float(q.float().std()) - 1.0) < 0.05
