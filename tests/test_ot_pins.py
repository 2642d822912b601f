"""Pins for the OT-1024 ordered-tree emulation and its own exp/log.

The ordered policy ("TIRx Metal reduction lowering" §1: an ordered tree stays
ordered and needs precise math) has no tree shape on the page; this library
defines OT-1024 (leaf fold_left mod 1024, pairwise quads, 16-8-4-2-1 xor
butterfly, balanced 8-way top).  The pins below fix that shape with hand-derived
float32 cases whose answer changes under any other pairing or order, fix the
exp/log to within 1 ulp of the true functions, and tie each emulated operator
to the FP64 oracle within the unordered tolerance.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(99)
T24 = float(2 ** 24)


# ------------------------------------------------------------------ exp / log

def test_ot_expf_special_values():
    assert oracle.ot_expf(0.0) == 1.0
    assert oracle.ot_expf(-0.0) == 1.0
    assert oracle.ot_expf(200.0) == np.inf
    assert oracle.ot_expf(-200.0) == 0.0
    assert oracle.ot_expf(-np.inf) == 0.0
    assert np.isnan(oracle.ot_expf(np.nan))
    assert oracle.ot_expf(89.0) == np.inf          # exp(89) > FLT_MAX
    assert 0 < oracle.ot_expf(-100.0) < np.finfo(np.float32).tiny  # subnormal result


def test_ot_expf_within_one_ulp():
    x = np.linspace(-87.0, 88.5, 2_000_003, dtype=np.float64).astype(np.float32)
    x = np.concatenate([x, RNG.uniform(-20, 0, 500_000).astype(np.float32),
                        np.float32(np.arange(-150, 128)) * np.float32(math.log(2))])
    got = oracle.ot_expf_array(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - ref) / ulp) <= 1.0


def test_ot_expf_subnormal_range():
    x = np.linspace(-103.9, -87.4, 100_001).astype(np.float32)
    got = oracle.ot_expf_array(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    assert np.max(np.abs(got - ref)) <= 2.0 * 2.0 ** -149 + 1e-7 * 2.0 ** -126


def test_ot_logf_special_values():
    assert oracle.ot_logf(1.0) == 0.0
    assert oracle.ot_logf(0.0) == -np.inf
    assert oracle.ot_logf(np.inf) == np.inf
    assert np.isnan(oracle.ot_logf(-1.0))
    assert np.isnan(oracle.ot_logf(np.nan))


def test_ot_logf_within_one_ulp():
    x = np.concatenate([
        np.exp(np.linspace(math.log(1e-37), math.log(3e38), 2_000_001)).astype(np.float32),
        np.linspace(0.5, 2.0, 1_000_001, dtype=np.float32),
        np.linspace(1.0, 60000.0, 500_001, dtype=np.float32),
        np.float32(2.0) ** np.arange(-126, 128, dtype=np.float32),
    ])
    got = oracle.ot_logf_array(x).astype(np.float64)
    ref = np.log(x.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    ulp[ref == 0] = 2.0 ** -149
    assert np.max(np.abs(got - ref) / ulp) <= 1.0


def test_ot_logf_subnormal_arguments():
    x = (np.arange(1, 5000, dtype=np.float64) * 2.0 ** -149 * 977).astype(np.float32)
    got = oracle.ot_logf_array(x).astype(np.float64)
    ref = np.log(x.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - ref) / ulp) <= 1.0


# ----------------------------------------------------------------- tree shape

def test_ot_sum_exact_on_small_integers():
    # every partial sum of small integers is exact, so any order gives the exact sum
    for n in (1, 3, 1023, 1024, 1025, 4096, 6144, 50257):
        v = RNG.integers(-100, 101, n).astype(np.float32)
        assert float(oracle.ot_sum(v)) == float(v.astype(np.int64).sum())


def test_ot_max_matches_maximum():
    for n in (1, 5, 1024, 3000):
        v = RNG.standard_normal(n).astype(np.float32)
        assert oracle.ot_max(v) == v.max()


def test_ot_max_signed_zero_is_canonical():
    assert np.signbit(oracle.ot_max(np.array([-0.0, 0.0], np.float32))) == False  # noqa: E712
    assert np.signbit(oracle.ot_max(np.array([0.0, -0.0], np.float32))) == False  # noqa: E712
    assert np.signbit(oracle.ot_max(np.array([-0.0], np.float32))) == True  # noqa: E712


def test_ot_leaf_is_fold_left_in_column_order():
    # column 0, 1024, 2048 share leaf 0: ((2^24 + 1) + 1) folds to 2^24 under
    # round-to-nearest-even; any tree over the three (2^24 + (1 + 1)) gives 2^24 + 2.
    v = np.zeros(2049, np.float32)
    v[0], v[1024], v[2048] = T24, 1.0, 1.0
    assert float(oracle.ot_sum(v)) == T24


def test_ot_quad_is_pairwise():
    # leaves 0..3 = [2^24, 1, 1, 1]: (2^24 + 1) + (1 + 1) = 2^24 + 2, while a
    # left fold ((2^24 + 1) + 1) + 1 would give 2^24.
    v = np.zeros(1024, np.float32)
    v[0:4] = [T24, 1.0, 1.0, 1.0]
    assert float(oracle.ot_sum(v)) == T24 + 2.0
    # pairing is (0,1),(2,3): [2^24, 1, -2^24, 1] -> 2^24 + (-2^24 + 1) = 1,
    # while (0,2),(1,3) would give 0 + 2 = 2.
    v[0:4] = [T24, 1.0, -T24, 1.0]
    assert float(oracle.ot_sum(v)) == 1.0


def test_ot_butterfly_offsets_descend():
    # partials of threads 0..3 (leaves 4t) = [2^24, 1, -2^24, 1].  Offsets
    # 16,8,4,2,1 combine lanes of equal parity first: (2^24 + -2^24) + (1 + 1) = 2.
    # Ascending offsets 1,2,4,... would give (2^24 + 1) + (-2^24 + 1) = 1.
    v = np.zeros(1024, np.float32)
    v[[0, 4, 8, 12]] = [T24, 1.0, -T24, 1.0]
    assert float(oracle.ot_sum(v)) == 2.0


def test_ot_group_top_is_balanced():
    # group results (threads 32g -> leaf 128g) = [2^24, 1, 1, 1, 0...]:
    # ((2^24 + 1) + (1 + 1)) = 2^24 + 2; a left fold gives 2^24.
    v = np.zeros(1024, np.float32)
    v[[0, 128, 256, 384]] = [T24, 1.0, 1.0, 1.0]
    assert float(oracle.ot_sum(v)) == T24 + 2.0
    # and the pairs are (g0,g1),(g2,g3): [2^24, 1, -2^24, 1] -> 1 (not 2)
    v[[0, 128, 256, 384]] = [T24, 1.0, -T24, 1.0]
    assert float(oracle.ot_sum(v)) == 1.0


def test_ot_sum_within_error_bound():
    # depth of OT-1024 for n columns: ceil(n/1024) leaf adds + 2 + 5 + 3 levels
    for n in (100, 1537, 6144, 65536):
        v = RNG.standard_normal(n).astype(np.float32)
        exact = math.fsum(float(t) for t in v)
        depth = math.ceil(n / 1024) + 10
        bound = depth * 2.0 ** -24 * float(np.abs(v.astype(np.float64)).sum())
        assert abs(float(oracle.ot_sum(v)) - exact) <= bound


# --------------------------------------------- emulated operators vs the oracle

def close(got, ref, rtol=2e-6, atol=1e-6):
    return np.all(np.abs(got.astype(np.float64) - ref) <= atol + rtol * np.abs(ref))


@pytest.mark.parametrize("r,c", [(3, 4096), (37, 1537), (5, 7), (2, 1)])
def test_ot_softmax_close_to_oracle(r, c):
    x = (RNG.standard_normal((r, c)) * 2).astype(np.float32)
    assert close(oracle.ot_softmax(x), oracle.softmax(x))


@pytest.mark.parametrize("r,c", [(3, 4096), (8, 3072), (4, 12289), (3, 1)])
def test_ot_norms_close_to_oracle(r, c):
    x = (RNG.standard_normal((r, c)) + RNG.uniform(-3, 3, (r, 1))).astype(np.float32)
    w = RNG.uniform(0.5, 1.5, c).astype(np.float32)
    b = (RNG.standard_normal(c) * 0.3).astype(np.float32)
    assert close(oracle.ot_rmsnorm(x, w, 1e-5), oracle.rmsnorm(x, w, 1e-5))
    assert close(oracle.ot_layernorm(x, w, b, 1e-5), oracle.layernorm(x, w, b, 1e-5))
    assert close(oracle.ot_layernorm(x, None, None, 1e-5), oracle.layernorm(x, None, None, 1e-5))


@pytest.mark.parametrize("r,c", [(7, 4096), (4, 50257), (3, 3)])
def test_ot_cross_entropy_close_to_oracle(r, c):
    x = (RNG.standard_normal((r, c)) * 3).astype(np.float32)
    lab = RNG.integers(-1, c + 1, r)
    assert close(oracle.ot_cross_entropy(x, lab), oracle.cross_entropy(x, lab))


def test_ot_softmax_constant_row_and_shift():
    x = np.full((1, 3000), 2.5, np.float32)
    assert np.all(oracle.ot_softmax(x) == np.float32(1.0) / np.float32(3000))
    g = (RNG.integers(-2048, 2049, (2, 5000)) / 1024.0).astype(np.float32)
    # x - max is exact for both, so the shifted row gives identical bits
    assert np.array_equal(oracle.ot_softmax(g), oracle.ot_softmax(g + np.float32(1.0)))


def test_ot_layernorm_constant_row_gives_beta():
    b = RNG.standard_normal(2048).astype(np.float32)
    g = RNG.uniform(0.5, 1.5, 2048).astype(np.float32)
    x = np.full((1, 2048), 3.0, np.float32)
    assert np.array_equal(oracle.ot_layernorm(x, g, b, 1e-5)[0], b)
