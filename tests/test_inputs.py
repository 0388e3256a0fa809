"""The seeded row samplers the parity tests use (host logic, no GPU)."""
import numpy as np

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
