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


# ---- the unordered maximum and minimum (oracle.c Part 5). The page fixes the
# reducers and leaves NaN undefined; the reading: NaN elements are skipped, a
# vector of NaN only gives NaN, the sign of a zero extreme met with both signs
# is not fixed. Every expected value below is written out by hand.

NAN, INF = np.float32(np.nan), np.float32(np.inf)


def test_skipnan_row_extremes_hand_written():
    x = np.array([
        [1.0, NAN, 3.0, -2.0],        # NaN in the middle: skipped
        [NAN, NAN, NAN, NAN],         # only NaN: NaN
        [NAN, 5.0, 7.0, NAN],         # NaN first and last
        [-INF, NAN, -INF, -INF],      # infinities are values
        [INF, 5.0, NAN, -1.5],
        [2.5, 2.5, 2.5, 2.5],
    ], np.float32)
    want_max = np.array([3.0, NAN, 7.0, -INF, INF, 2.5], np.float32)
    want_min = np.array([-2.0, NAN, 5.0, -INF, -1.5, 2.5], np.float32)
    got_max, got_min = oracle.row_max_skipnan(x), oracle.row_min_skipnan(x)
    assert np.array_equal(np.isnan(got_max), np.isnan(want_max))
    assert np.array_equal(np.isnan(got_min), np.isnan(want_min))
    ok = ~np.isnan(want_max)
    assert np.array_equal(got_max[ok], want_max[ok]) and np.array_equal(got_min[ok], want_min[ok])


def test_skipnan_zero_extremes_have_value_zero():
    # a zero maximum met as -0 and +0: either sign is a correct result
    x = np.array([[-1.0, -0.0, NAN, 0.0], [NAN, 0.0, 1.0, -0.0]], np.float32)
    assert oracle.row_max_skipnan(x)[0] == 0.0
    assert oracle.row_min_skipnan(x)[1] == 0.0


def test_skipnan_differs_from_propagating_reducers():
    # the reading is not numpy's NaN-propagating max / min
    x = np.array([[1.0, NAN, 3.0]], np.float32)
    assert np.isnan(x.max(axis=1)[0]) and oracle.row_max_skipnan(x)[0] == 3.0
    assert np.isnan(x.min(axis=1)[0]) and oracle.row_min_skipnan(x)[0] == 1.0


def test_skipnan_axis_extremes_hand_written():
    # x[o, r, i] with outer 2, extent 3, inner 2; the reduction runs over r
    x = np.array([[[1.0, NAN], [4.0, NAN], [-3.0, NAN]],
                  [[NAN, 0.5], [NAN, -INF], [2.0, 9.0]]], np.float32)
    got_max = oracle.axis_max_skipnan(x, 1)
    got_min = oracle.axis_min_skipnan(x, 1)
    assert got_max[0, 0] == 4.0 and np.isnan(got_max[0, 1])
    assert got_max[1, 0] == 2.0 and got_max[1, 1] == 9.0
    assert got_min[0, 0] == -3.0 and np.isnan(got_min[0, 1])
    assert got_min[1, 0] == 2.0 and got_min[1, 1] == -INF
    # the same values reduced over axis 0 (outer) and axis 2 (inner)
    assert oracle.axis_max_skipnan(x, 0)[0, 0] == 1.0 and oracle.axis_max_skipnan(x, 0)[2, 1] == 9.0
    assert oracle.axis_min_skipnan(x, 2)[1, 1] == -INF and oracle.axis_max_skipnan(x, 2)[0, 0] == 1.0
