"""GPU parity of the standalone row reductions (sum, max, min, min and max
together) against the CPU oracle ("TIRx Metal reduction lowering" §8: row sums
at widths 127, 257, 1024 and 4096; minimum and maximum together at 7x1024).

Unordered sum: |gpu - FP64 sum| <= (cols/4 + 16) * 2^-24 * sum|x|, the
rounding bound of a sum in which every element passes through at most
cols/4 + 16 additions (the longest chain of any plan: a 4-lane worker's
sequential fold, then the tree). Max and min are exact in any order; under
the unordered policy they skip NaN elements (oracle.row_max_skipnan /
row_min_skipnan), so they must give NaN exactly where the oracle does and the
oracle's value everywhere else (a zero extreme met with both signs may come
out with either sign). Ordered: bit-identical to the OT-1024
emulation; max and min keep NaN payloads (they only select), a sum that
becomes NaN is only checked to be NaN.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp32_row_reduction_gb300 as tr

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SHAPES = [(1, 1), (5, 3), (3, 127), (3, 257), (3, 1024), (3, 4096), (7, 1024), (17, 257), (37, 1537),
          (9, 20000), (1000, 96), (4, 70001)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()
    yield
    tr.tr_plan_override(None)


def run(op, x, order="unordered"):
    out = tr.row_reduce(x, op, order=order)
    torch.cuda.synchronize()
    if op == "row_minmax":
        return out[0].cpu().numpy(), out[1].cpu().numpy()
    return out.cpu().numpy()


def same_extremes(got, want):
    """NaN exactly where `want` has NaN; every other value equal (+0 == -0)."""
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def check_unordered(op, x, got):
    h = x.cpu().numpy()
    if op == "row_sum":
        exact = oracle.row_sum(h)
        cols = h.shape[1]
        bound = (cols / 4 + 16) * 2.0 ** -24 * np.abs(h.astype(np.float64)).sum(axis=1)
        assert np.all(np.abs(got.astype(np.float64) - exact) <= bound)
    elif op == "row_max":
        same_extremes(got, oracle.row_max_skipnan(h))
    elif op == "row_min":
        same_extremes(got, oracle.row_min_skipnan(h))
    else:
        same_extremes(got[0], oracle.row_min_skipnan(h))
        same_extremes(got[1], oracle.row_max_skipnan(h))


def check_ordered(op, x, got):
    h = x.cpu().numpy()
    bits = lambda a: np.asarray(a, np.float32).view(np.uint32)
    if op == "row_sum":
        # a NaN produced by arithmetic has no portable payload: NaN positions must
        # agree, every other result bit for bit
        want = oracle.ot_row_sum(h)
        assert np.array_equal(np.isnan(got), np.isnan(want))
        ok = ~np.isnan(want)
        assert np.array_equal(bits(got[ok]), bits(want[ok]))
    elif op == "row_max":
        assert np.array_equal(bits(got), bits(oracle.ot_row_max(h)))
    elif op == "row_min":
        assert np.array_equal(bits(got), bits(oracle.ot_row_min(h)))
    else:
        assert np.array_equal(bits(got[0]), bits(oracle.ot_row_min(h)))
        assert np.array_equal(bits(got[1]), bits(oracle.ot_row_max(h)))


OPS = ["row_sum", "row_max", "row_min", "row_minmax"]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", OPS)
def test_row_reductions_match_oracle(op, rows, cols):
    x = synth.make_inputs(op, rows, cols, seed=rows * 7 + cols, row_offset=True, device=DEV)["x"]
    check_unordered(op, x, run(op, x))
    check_ordered(op, x, run(op, x, "ordered"))


@pytest.mark.parametrize("xoff", [1, 2, 3])
@pytest.mark.parametrize("op", OPS)
def test_unaligned_rows(op, xoff):
    rows, cols = 6, 1027
    x0 = synth.make_inputs(op, rows, cols, seed=xoff, device=DEV)["x"]
    big = torch.empty(rows * cols + 8, device=DEV)
    x = big[xoff:xoff + rows * cols].view(rows, cols)
    x.copy_(x0)
    check_unordered(op, x, run(op, x))
    check_ordered(op, x, run(op, x, "ordered"))


def test_integer_rows_sum_exactly():
    # small integers: every partial sum is exact, so both policies give the exact sum
    g = torch.Generator().manual_seed(8)
    x = torch.randint(-100, 101, (7, 4099), generator=g).float().to(DEV)
    exact = x.cpu().numpy().astype(np.float64).sum(axis=1)
    assert np.array_equal(run("row_sum", x).astype(np.float64), exact)
    assert np.array_equal(run("row_sum", x, "ordered").astype(np.float64), exact)


def test_special_rows():
    x = torch.randn(6, 3000, generator=torch.Generator().manual_seed(9))
    x[0] = float("nan")                   # all NaN
    x[1, 17] = float("nan")               # one NaN
    x[2] = -x[2].abs() - 1.0
    x[2, 5], x[2, 2000] = -0.0, 0.0       # maximum a tie of -0 and +0
    x[3] = x[3].abs() + 1.0
    x[3, 9], x[3, 99] = 0.0, -0.0         # minimum a tie of +0 and -0
    x[4, 100] = float("inf")
    x[5, 200] = float("-inf")
    x = x.to(DEV)
    for op in ("row_max", "row_min", "row_minmax", "row_sum"):
        check_ordered(op, x, run(op, x, "ordered"))
    for op in ("row_max", "row_min", "row_minmax"):
        check_unordered(op, x, run(op, x))


def reduce_plans(op, rows, cols):
    code = tr.OPS[op]
    plans = []
    for g in (4, 8, 16):
        plans.append(dict(lanes_per_row=g, warps_per_row=1, rows_per_cta=128 // g, vec_slots=2, block_threads=128))
    for s in (1, 3, 8, 32):
        for q in (1, 2):
            if 32 * s * q > 1024:
                continue
            for k in (2, 4, 8):
                plans.append(dict(lanes_per_row=32, warps_per_row=s, rows_per_cta=q, vec_slots=k,
                                  block_threads=32 * s * q))
    ok = []
    for p in plans:
        assert tr.tr_plan_override(tr.tr_plan(op=code, order=0, kind=tr.TR_PLAN_XENT, cluster_ctas=1, **p)) == tr.TR_OK
        try:
            tr.tr_plan_describe(code, rows, cols, 0)
            ok.append(p)
        except tr.TrError as e:
            assert e.status == tr.TR_ERR_UNSUPPORTED
    tr.tr_plan_override(None)
    return ok


@pytest.mark.parametrize("rows,cols", [(5, 3), (7, 1024), (3, 4099)])
@pytest.mark.parametrize("op", OPS)
def test_every_reduction_plan(op, rows, cols):
    x = synth.make_inputs(op, rows, cols, seed=11, device=DEV)["x"]
    plans = reduce_plans(op, rows, cols)
    assert plans
    try:
        for p in plans:
            assert tr.tr_plan_override(tr.tr_plan(op=tr.OPS[op], order=0, kind=tr.TR_PLAN_XENT, cluster_ctas=1,
                                                  **p)) == tr.TR_OK
            check_unordered(op, x, run(op, x))
    finally:
        tr.tr_plan_override(None)


@pytest.mark.parametrize("op", ["row_sum", "row_minmax"])
def test_full_size_768x6144(op):
    x = synth.workload_inputs(f"{op}_768x6144", device=DEV)["x"]
    check_unordered(op, x, run(op, x))
    check_ordered(op, x, run(op, x, "ordered"))


def test_ordered_nan_payloads_and_signed_zeros():
    # quiet NaNs of both signs with distinct payloads: the ordered max and min keep
    # the one the canonical tree selects, bit for bit; rows without NaN take the
    # integer-key path and must still give +0 (max) and -0 (min) for mixed zeros
    rng = np.random.default_rng(12)
    h = rng.standard_normal((10, 5003)).astype(np.float32)
    b = h.view(np.uint32)
    for r in range(6):
        k = int(rng.integers(1, 6))
        cols = rng.choice(5003 if r else 40, k, replace=False)
        payload = rng.integers(1, 1 << 22, k).astype(np.uint32)
        sign = (rng.integers(0, 2, k).astype(np.uint32) << 31)
        b[r, cols] = sign | np.uint32(0x7fc00000) | payload
    h[6] = 0.0
    h[6, ::3] = -0.0
    h[7] = -np.abs(h[7]) - 1.0
    h[7, 4999] = -0.0
    h[8] = np.abs(h[8]) + 1.0
    h[8, 3] = 0.0
    h[9, 11] = np.float32(np.inf)
    h[9, 12] = np.float32(-np.inf)
    x = torch.from_numpy(h.copy()).to(DEV)
    for op in ("row_max", "row_min", "row_minmax"):
        check_ordered(op, x, run(op, x, "ordered"))


def nan_rows(rows, cols, seed):
    """Rows with NaN at random places (none, a few, most, all), infinities and signed zeros."""
    rng = np.random.default_rng(seed)
    h = (rng.standard_normal((rows, cols)) * 3.0).astype(np.float32)
    for r in range(rows):
        kind = r % 8
        if kind == 1:
            h[r, rng.choice(cols, min(cols, 3), replace=False)] = np.nan
        elif kind == 2:
            h[r, rng.random(cols) < 0.9] = np.nan
        elif kind == 3:
            h[r] = np.nan
        elif kind == 4:
            h[r, rng.integers(0, cols)] = np.inf
            h[r, rng.integers(0, cols)] = -np.inf
            h[r, rng.integers(0, cols)] = np.nan
        elif kind == 5:
            h[r] = -np.abs(h[r]) - 1.0
            h[r, rng.choice(cols, min(cols, 2), replace=False)] = [-0.0, 0.0][:min(cols, 2)]
            h[r, rng.integers(0, cols)] = np.nan
        elif kind == 6:
            h[r] = np.abs(h[r]) + 1.0
            h[r, rng.integers(0, cols)] = -0.0
        elif kind == 7:
            h[r, 0] = np.nan
            h[r, cols - 1] = np.nan
    return h


@pytest.mark.parametrize("rows,cols", [(8, 1), (16, 5), (24, 257), (16, 1024), (8, 4099), (16, 20000)])
def test_unordered_extremes_skip_nan(rows, cols):
    # the unordered max / min against the oracle's NaN-skipping definition
    h = nan_rows(rows, cols, seed=rows * 31 + cols)
    x = torch.from_numpy(h).to(DEV)
    for op in ("row_max", "row_min", "row_minmax"):
        check_unordered(op, x, run(op, x))


def test_unordered_extremes_skip_nan_in_every_plan():
    h = nan_rows(24, 1031, seed=77)
    x = torch.from_numpy(h).to(DEV)
    for op in ("row_max", "row_min", "row_minmax"):
        plans = reduce_plans(op, 24, 1031)
        assert plans
        try:
            for p in plans:
                assert tr.tr_plan_override(tr.tr_plan(op=tr.OPS[op], order=0, kind=tr.TR_PLAN_XENT, cluster_ctas=1,
                                                      **p)) == tr.TR_OK
                check_unordered(op, x, run(op, x))
        finally:
            tr.tr_plan_override(None)
