"""GPU parity of the reductions over a non-last axis against the CPU oracle
("TIRx Metal reduction lowering", Reductions inside composed groups: both
axis positions, extent one, ragged widths, more outputs than resident
workers).

x is [outer, extent, inner]; the library reduces the middle axis. Unordered
sums: |gpu - FP64| <= (extent / 32 + 24) * 2^-24 * sum|x| (the longest chain:
an eighth of a split's rows folded into one of four accumulators, then at most
2 + 3 + 5 tree levels); max / min exact. Ordered: bit-identical to OT-1024
applied to every column vector (a NaN sum only checked to be NaN).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp32_row_reduction_gb300 as tr

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SHAPES = [(1, 1, 1), (3, 1, 5), (2, 7, 33), (4, 257, 3), (1, 1024, 64), (3, 1025, 40), (2, 3000, 17),
          (64, 128, 1), (1, 20000, 7), (5, 4099, 128), (1, 768, 6144), (7, 300, 1000)]
OPS = ["sum", "max", "min", "minmax"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()


def make(outer, extent, inner, seed):
    x = synth.make_inputs("row_sum", outer * extent, inner, seed=seed, row_offset=True, device=DEV)["x"]
    return x.view(outer, extent, inner)


def run(x, op, order, dim=1):
    out = tr.axis_reduce(x, dim, op, order=order)
    torch.cuda.synchronize()
    if op == "minmax":
        return out[0].cpu().numpy(), out[1].cpu().numpy()
    return out.cpu().numpy()


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def same_extremes(got, want):
    """Unordered max / min (NaN elements skipped): NaN exactly where the oracle has
    NaN, every other value equal (a zero extreme of either sign)."""
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def check(x, op, order, got, dim=1):
    h = x.cpu().numpy()
    if order == "unordered":
        if op == "sum":
            exact = oracle.axis_sum(h, dim)
            bound = (h.shape[dim] / 32 + 24) * 2.0 ** -24 * np.abs(h.astype(np.float64)).sum(axis=dim)
            assert np.all(np.abs(got.astype(np.float64) - exact) <= bound)
        elif op == "max":
            same_extremes(got, oracle.axis_max_skipnan(h, dim))
        elif op == "min":
            same_extremes(got, oracle.axis_min_skipnan(h, dim))
        else:
            same_extremes(got[0], oracle.axis_min_skipnan(h, dim))
            same_extremes(got[1], oracle.axis_max_skipnan(h, dim))
        return
    if op == "sum":
        want = oracle.ot_axis_sum(h, dim)
        assert np.array_equal(np.isnan(got), np.isnan(want))
        ok = ~np.isnan(want)
        assert np.array_equal(bits(got[ok]), bits(want[ok]))
    elif op == "max":
        assert np.array_equal(bits(got), bits(oracle.ot_axis_max(h, dim)))
    elif op == "min":
        assert np.array_equal(bits(got), bits(oracle.ot_axis_min(h, dim)))
    else:
        assert np.array_equal(bits(got[0]), bits(oracle.ot_axis_min(h, dim)))
        assert np.array_equal(bits(got[1]), bits(oracle.ot_axis_max(h, dim)))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("op", OPS)
def test_axis_matches_oracle(op, shape):
    x = make(*shape, seed=sum(shape))
    for order in ("unordered", "ordered"):
        check(x, op, order, run(x, op, order))


def test_both_axis_positions_and_splits():
    # dim 0, 1, 2 and the last of a 4-D tensor; launches with and without splits
    x = make(3, 40, 6 * 50, seed=3).view(3, 40, 6, 50)
    for dim in range(4):
        for order in ("unordered", "ordered"):
            for op in ("sum", "max"):
                check(x, op, order, run(x, op, order, dim), dim)
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert tr.axis_launch_shape("sum", 1, 20000, 7, sm)[0] > 1
    assert tr.axis_launch_shape("sum", 1, 768, 6144, sm)[0] >= 1


def test_repeated_split_launches_reset_their_tickets():
    x = make(1, 20000, 7, seed=4)
    first = run(x, "sum", "ordered")
    for _ in range(3):
        assert np.array_equal(bits(run(x, "sum", "ordered")), bits(first))
    check(x, "minmax", "unordered", run(x, "minmax", "unordered"))


def test_axis_equals_row_reduction_of_the_same_vectors():
    # inner = 1: each column vector is a row; the ordered results share the tree
    x = make(37, 1537, 1, seed=6)
    rows = x.view(37, 1537)
    for op in ("sum", "max", "min"):
        a = tr.axis_reduce(x, 1, op, order="ordered")
        b = tr.row_reduce(rows, "row_" + op, order="ordered")
        torch.cuda.synchronize()
        assert np.array_equal(bits(a.view(-1).cpu().numpy()), bits(b.cpu().numpy()))


def test_ordered_nan_payloads_and_zeros():
    rng = np.random.default_rng(17)
    h = rng.standard_normal((2, 3000, 40)).astype(np.float32)
    b = h.view(np.uint32)
    for i in range(0, 40, 3):
        k = int(rng.integers(1, 4))
        rows = rng.choice(3000, k, replace=False)
        b[i % 2, rows, i] = (rng.integers(0, 2, k).astype(np.uint32) << 31) | np.uint32(0x7fc00000) | \
            rng.integers(1, 1 << 22, k).astype(np.uint32)
    h[:, :, 1] = 0.0
    h[:, ::7, 1] = -0.0
    h[0, :, 2] = np.nan
    x = torch.from_numpy(h.copy()).to(DEV)
    for op in ("max", "min", "minmax"):
        check(x, op, "ordered", run(x, op, "ordered"))
        check(x, op, "unordered", run(x, op, "unordered"))


def test_axis_argument_errors():
    x = make(2, 3, 4, seed=1)
    lib = tr.load()
    s = torch.cuda.current_stream().cuda_stream
    out = torch.empty(8, device=DEV)
    assert lib.tr_axis_sum_f32(x.data_ptr(), out.data_ptr(), 2, 0, 4, 0, s) == tr.TR_ERR_INVALID_ARG
    assert lib.tr_axis_sum_f32(x.data_ptr(), out.data_ptr(), 2, 3, 0, 0, s) == tr.TR_ERR_INVALID_ARG
    assert lib.tr_axis_sum_f32(x.data_ptr(), x.data_ptr() + 4, 2, 3, 4, 0, s) == tr.TR_ERR_INVALID_ARG
    assert lib.tr_axis_sum_f32(x.data_ptr(), out.data_ptr(), 0, 3, 4, 0, s) == tr.TR_OK   # nothing to do
    assert lib.tr_axis_sum_f32(x.data_ptr(), out.data_ptr(), 2, 3, 4, 7, s) == tr.TR_ERR_INVALID_ARG


def test_full_size_768x6144_column_sums():
    x = synth.workload_inputs("axis_sum_768x6144", device=DEV)["x"].view(1, 768, 6144)
    for op in ("sum", "minmax"):
        for order in ("unordered", "ordered"):
            check(x, op, order, run(x, op, order))


@pytest.mark.parametrize("off", [1, 2, 3])
def test_unaligned_x_takes_the_scalar_columns(off):
    outer, extent, inner = 3, 1500, 64
    x0 = make(outer, extent, inner, seed=off)
    big = torch.empty(x0.numel() + 8, device=DEV)
    x = big[off:off + x0.numel()].view(outer, extent, inner)
    x.copy_(x0)
    for op in ("sum", "minmax"):
        for order in ("unordered", "ordered"):
            check(x, op, order, run(x, op, order))


@pytest.mark.parametrize("shape", [(2, 3000, 40), (1, 20000, 7), (3, 64, 129), (4, 9, 256)])
def test_unordered_axis_extremes_skip_nan(shape):
    # NaN at random places of some columns, all-NaN columns, infinities, signed
    # zeros; with and without splits of the reduced axis, scalar and quad columns
    outer, extent, inner = shape
    rng = np.random.default_rng(sum(shape))
    h = (rng.standard_normal(shape) * 2.0).astype(np.float32)
    for i in range(inner):
        kind = i % 6
        o = i % outer
        if kind == 1:
            h[o, rng.choice(extent, min(extent, 3), replace=False), i] = np.nan
        elif kind == 2:
            h[o, :, i] = np.nan
        elif kind == 3:
            h[o, rng.random(extent) < 0.8, i] = np.nan
        elif kind == 4:
            h[o, rng.integers(0, extent), i] = np.inf
            h[o, rng.integers(0, extent), i] = -np.inf
        elif kind == 5:
            h[o, :, i] = -np.abs(h[o, :, i]) - 1.0
            h[o, 0, i], h[o, extent - 1, i] = -0.0, 0.0
    x = torch.from_numpy(h).to(DEV)
    for op in ("max", "min", "minmax"):
        check(x, op, "unordered", run(x, op, "unordered"))
