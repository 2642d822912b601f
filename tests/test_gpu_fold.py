"""GPU parity of the fold policies ("TIRx Metal reduction lowering" §1,
ReductionPolicy fold_left / fold_right) against the CPU emulation: every
operator and row reduction bit-identical, both directions, ragged and
unaligned rows, rows holding NaN, and the refusal of the entry points that
take the tree policies only. A NaN produced by arithmetic has no portable
payload: NaN positions must agree, every other output bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp32_row_reduction_gb300 as tr

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DIRS = ["fold_left", "fold_right"]
SHAPES = [(1, 1), (5, 3), (4, 127), (3, 128), (17, 257), (7, 1025), (37, 1537), (3, 6144), (2, 20000)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def same(got, want, what):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), f"{what}: NaN positions differ"
    bad = bits(got[~nan]) != bits(want[~nan])
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} differ"


def direction(order):
    return "left" if order == "fold_left" else "right"


def check_ops(d, order, what):
    x = d["x"]
    h = {k: v.cpu().numpy() for k, v in d.items()}
    dr = direction(order)
    same(tr.softmax(x, order=order).cpu().numpy(), oracle.fold_softmax(h["x"], dr), f"softmax {what}")
    same(tr.rmsnorm(x, d["w"], 1e-5, order=order).cpu().numpy(), oracle.fold_rmsnorm(h["x"], h["w"], 1e-5, dr),
         f"rmsnorm {what}")
    same(tr.layernorm(x, d["w"], d["b"], 1e-5, order=order).cpu().numpy(),
         oracle.fold_layernorm(h["x"], h["w"], h["b"], 1e-5, dr), f"layernorm {what}")
    same(tr.layernorm(x, None, None, 1e-5, order=order).cpu().numpy(),
         oracle.fold_layernorm(h["x"], None, None, 1e-5, dr), f"layernorm no affine {what}")
    same(tr.row_reduce(x, "row_sum", order=order).cpu().numpy(), oracle.fold_row_sum(h["x"], dr), f"row_sum {what}")
    same(tr.row_reduce(x, "row_max", order=order).cpu().numpy(), oracle.fold_row_max(h["x"], dr), f"row_max {what}")
    same(tr.row_reduce(x, "row_min", order=order).cpu().numpy(), oracle.fold_row_min(h["x"], dr), f"row_min {what}")
    lo, hi = tr.row_reduce(x, "row_minmax", order=order)
    same(lo.cpu().numpy(), oracle.fold_row_min(h["x"], dr), f"row_minmax min {what}")
    same(hi.cpu().numpy(), oracle.fold_row_max(h["x"], dr), f"row_minmax max {what}")


@pytest.mark.parametrize("order", DIRS)
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_fold_matches_emulation(rows, cols, order):
    d = synth.make_inputs("layernorm", rows, cols, seed=rows * 5 + cols, row_offset=True, device=DEV)
    check_ops(d, order, f"{order} {rows}x{cols}")
    c = synth.make_inputs("cross_entropy", rows, cols, seed=rows + cols, var=9.0, device=DEV)
    lab = c["labels"].clone()
    if rows > 1:
        lab[0] = -1
    got = tr.cross_entropy(c["x"], lab, order=order).cpu().numpy()
    same(got, oracle.fold_cross_entropy(c["x"].cpu().numpy(), lab.cpu().numpy(), direction(order)),
         f"cross_entropy {order} {rows}x{cols}")


@pytest.mark.parametrize("order", DIRS)
@pytest.mark.parametrize("off", [1, 2, 3])
def test_fold_unaligned_rows(order, off):
    rows, cols = 6, 1031
    d0 = synth.make_inputs("layernorm", rows, cols, seed=off, row_offset=True, device=DEV)
    big = torch.empty(rows * cols + 8, device=DEV)
    x = big[off:off + rows * cols].view(rows, cols)
    x.copy_(d0["x"])
    check_ops(dict(d0, x=x), order, f"{order} offset {off}")


@pytest.mark.parametrize("order", DIRS)
def test_fold_rows_with_nan_and_signed_zeros(order):
    rng = np.random.default_rng(41)
    h = rng.standard_normal((6, 700)).astype(np.float32)
    b = h.view(np.uint32)
    b[0, [5, 600]] = np.array([0x7fc00011, 0xffc00022], np.uint32)   # two NaN payloads, both signs
    b[1, 350] = np.uint32(0xffc00033)
    h[2] = 0.0
    h[2, ::3] = -0.0
    h[3, 0] = np.inf
    h[4, 699] = -np.inf
    x = torch.from_numpy(h.copy()).to(DEV)
    dr = direction(order)
    same(tr.row_reduce(x, "row_max", order=order).cpu().numpy(), oracle.fold_row_max(h, dr), "max")
    same(tr.row_reduce(x, "row_min", order=order).cpu().numpy(), oracle.fold_row_min(h, dr), "min")
    same(tr.row_reduce(x, "row_sum", order=order).cpu().numpy(), oracle.fold_row_sum(h, dr), "sum")
    same(tr.softmax(x, order=order).cpu().numpy(), oracle.fold_softmax(h, dr), "softmax")


def test_fold_refusals():
    d = synth.make_inputs("add_layernorm", 4, 300, seed=1, device=DEV)
    for order in DIRS:
        with pytest.raises(tr.TrError) as e:
            tr.add_layernorm(d["x"], d["r"], d["w"], d["b"], order=order)
        assert e.value.status == tr.TR_ERR_UNSUPPORTED
        with pytest.raises(tr.TrError) as e:
            tr.softmax_backward(d["x"], d["r"], order=order)
        assert e.value.status == tr.TR_ERR_UNSUPPORTED
        with pytest.raises(tr.TrError) as e:
            tr.axis_reduce(d["x"], 0, "sum", order=order)
        assert e.value.status == tr.TR_ERR_UNSUPPORTED
        p = tr.tr_plan_describe(tr.TR_OP_SOFTMAX, 100, 6144, tr.ORDERS[order])
        assert p.kind == tr.TR_PLAN_FOLD and p.grid_ctas == 50


def test_fold_full_size_768x6144():
    d = synth.workload_inputs("layernorm_768x6144", device=DEV)
    idx = torch.arange(0, 768, 16, device=DEV)
    for order in DIRS:
        y = tr.layernorm(d["x"], d["w"], d["b"], 1e-5, order=order)[idx].cpu().numpy()
        sub = d["x"][idx].cpu().numpy()
        same(y, oracle.fold_layernorm(sub, d["w"].cpu().numpy(), d["b"].cpu().numpy(), 1e-5, direction(order)),
             f"layernorm 768x6144 {order}")
