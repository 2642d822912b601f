"""Pins of the oracle's standalone row reductions ("TIRx Metal reduction
lowering" §8: row sums at widths 127, 257, 1024 and 4096; minimum and maximum
together at 7x1024) and of the canonical OT-1024 min."""
import math

import numpy as np

import oracle


def test_row_sum_closed_forms():
    # 1..n sums to n(n+1)/2 exactly in FP64 and in any FP32 order below 2^24
    for n in (127, 257, 1024, 4096):
        x = np.arange(1, n + 1, dtype=np.float32)[None, :]
        assert oracle.row_sum(x)[0] == n * (n + 1) / 2
        assert oracle.ot_row_sum(x)[0] == np.float32(n * (n + 1) / 2)


def test_ot_sum_is_a_fixed_tree_within_the_bound():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 4097)).astype(np.float32)
    exact = oracle.row_sum(x)
    got = oracle.ot_row_sum(x).astype(np.float64)
    # OT-1024: each element passes through at most 5 leaf adds + 2 + 5 + 3 tree levels
    depth = math.ceil(4097 / 1024) + 2 + 5 + 3
    bound = depth * 2.0 ** -24 * np.abs(x.astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(got - exact) <= bound)


def test_max_min_are_exact_and_canonical():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 1024)).astype(np.float32)
    assert np.array_equal(oracle.ot_row_max(x), x.max(axis=1))
    assert np.array_equal(oracle.ot_row_min(x), x.min(axis=1))
    z = np.array([[0.0, -0.0, -1.0], [-0.0, 0.0, -1.0]], np.float32)
    assert not np.signbit(oracle.ot_row_max(z)).any()          # +0 over -0 for the max
    z = -z
    assert np.signbit(oracle.ot_row_min(z)).all()              # -0 over +0 for the min
    n = np.array([[1.0, np.nan, 2.0]], np.float32)
    assert np.isnan(oracle.ot_row_min(n)[0]) and np.isnan(oracle.ot_row_max(n)[0])


def test_single_column_rows():
    x = np.array([[3.5], [-2.0]], np.float32)
    assert np.array_equal(oracle.ot_row_sum(x), x[:, 0])
    assert np.array_equal(oracle.ot_row_min(x), x[:, 0])
    assert np.array_equal(oracle.row_sum(x), x[:, 0].astype(np.float64))
