"""GPU parity of the fused residual norms (y = norm(x + r), h = x + r) against
the CPU oracle ("TIRx Metal reduction lowering" §5.1: LayerNorm over combined =
X + residual, each input loaded once).

h must equal the FP32 sum bit for bit in both policies; y must be within the
unordered tolerance of the FP64 oracle (unordered), or bit-identical to the
OT-1024 emulation (ordered). Every legal plan of the family is checked.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp32_row_reduction_gb300 as tr

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-6, 1e-6
DEV = "cuda:0"
OPS = ["add_rmsnorm", "add_layernorm"]
SHAPES = [(1, 1), (5, 3), (4, 127), (17, 257), (3, 4096), (7, 1024), (37, 1537), (9, 20000), (64, 12289)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()
    yield
    tr.tr_plan_override(None)


def make(op, rows, cols, seed, affine=True):
    d = synth.make_inputs(op, rows, cols, seed, row_offset=True, device=DEV)
    if not affine:
        d = {"x": d["x"], "r": d["r"]}
    return d


def reference(op, d, order):
    h = {k: v.cpu().numpy() for k, v in d.items()}
    if op == "add_rmsnorm":
        f = oracle.ot_add_rmsnorm if order == "ordered" else oracle.add_rmsnorm
        return f(h["x"], h["r"], h.get("w"), 1e-5)
    f = oracle.ot_add_layernorm if order == "ordered" else oracle.add_layernorm
    return f(h["x"], h["r"], h.get("w"), h.get("b"), 1e-5)


def run(op, d, order="unordered", y=None, h=None):
    y = torch.empty_like(d["x"]) if y is None else y
    h = torch.empty_like(d["x"]) if h is None else h
    tr.run_op(op, d, out=y, order=order, h_out=h)
    torch.cuda.synchronize()
    return y, h


def check(op, d, y, h, order, what):
    want_y, want_h = reference(op, d, order)
    got_h = h.cpu().numpy()
    assert np.array_equal(got_h.view(np.uint32), want_h.view(np.uint32)), f"{what}: h differs"
    got = y.cpu().numpy()
    if order == "ordered":
        assert np.array_equal(got.view(np.uint32), want_y.view(np.uint32)), f"{what}: y differs from the emulation"
    else:
        err = np.abs(got.astype(np.float64) - want_y)
        bad = ~(err <= ATOL + RTOL * np.abs(want_y))
        assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"


@pytest.mark.parametrize("order", ["unordered", "ordered"])
@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", OPS)
def test_fused_matches_oracle(op, rows, cols, order):
    d = make(op, rows, cols, seed=rows * 13 + cols)
    if order == "ordered" and cols > 16 * 1024:
        # the fused ordered plans cache the row: longer rows are refused, not clamped
        with pytest.raises(tr.TrError) as e:
            run(op, d, order)
        assert e.value.status == tr.TR_ERR_UNSUPPORTED
        return
    y, h = run(op, d, order)
    check(op, d, y, h, order, f"{op} {order} {rows}x{cols}")


@pytest.mark.parametrize("op", OPS)
def test_fused_without_affine_and_without_h(op):
    d = make(op, 11, 3000, seed=5, affine=False)
    y = torch.empty_like(d["x"])
    tr.run_op(op, d, out=y)
    torch.cuda.synchronize()
    want_y, _ = reference(op, d, "unordered")
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want_y) <= ATOL + RTOL * np.abs(want_y))


@pytest.mark.parametrize("offs", [(1, 0, 0, 0), (0, 2, 0, 3), (3, 1, 2, 1), (2, 2, 2, 2)])
@pytest.mark.parametrize("op", OPS)
def test_fused_unaligned_tensors(op, offs):
    # x, r, y, h each placed at an offset of 0..3 floats from a 16-byte boundary
    rows, cols = 6, 2051
    d = make(op, rows, cols, seed=sum(offs) + 40)
    n = rows * cols
    views = []
    for src, off in zip((d["x"], d["r"]), offs[:2]):
        big = torch.empty(n + 8, device=DEV)
        v = big[off:off + n].view(rows, cols)
        v.copy_(src)
        views.append(v)
    outs = []
    for off in offs[2:]:
        big = torch.zeros(n + 8, device=DEV)
        outs.append(big[off:off + n].view(rows, cols))
    d2 = dict(d, x=views[0], r=views[1])
    for order in ("unordered", "ordered"):
        y, h = run(op, d2, order, y=outs[0], h=outs[1])
        check(op, d, y, h, order, f"{op} {order} offsets {offs}")


def fused_plans(op, rows, cols):
    """Every plan the library accepts for the fused op at this shape (unordered)."""
    code = tr.OPS[op]
    plans = []
    for g in (4, 8, 16):
        for k in (1, 2, 4):
            plans.append(dict(kind=tr.TR_PLAN_ROWS, lanes_per_row=g, warps_per_row=1, rows_per_cta=64 // g,
                              cluster_ctas=1, vec_slots=k, block_threads=64))
    for s in (1, 3, 8):
        for q in (1, 2):
            for k in (1, 2, 4, 6, 8, 16):
                for flags in (0, tr.TR_PLAN_FLAG_PARAMS_IN_SHARED):
                    plans.append(dict(kind=tr.TR_PLAN_ROWS, lanes_per_row=32, warps_per_row=s, rows_per_cta=q,
                                      cluster_ctas=1, vec_slots=k, block_threads=32 * s * q, flags=flags))
    for c in (2, 5):
        for k in (4, 8, 16):
            plans.append(dict(kind=tr.TR_PLAN_CLUSTER, lanes_per_row=32, warps_per_row=8, rows_per_cta=1,
                              cluster_ctas=c, vec_slots=k, block_threads=256))
    ok = []
    for p in plans:
        assert tr.tr_plan_override(tr.tr_plan(op=code, order=0, **p)) == tr.TR_OK
        try:
            tr.tr_plan_describe(code, rows, cols, 0)
            ok.append(p)
        except tr.TrError as e:
            assert e.status == tr.TR_ERR_UNSUPPORTED
    tr.tr_plan_override(None)
    return ok


@pytest.mark.parametrize("rows,cols", [(5, 3), (7, 1024), (3, 4100), (2, 20001)])
@pytest.mark.parametrize("op", OPS)
def test_every_fused_plan_matches_oracle(op, rows, cols):
    d = make(op, rows, cols, seed=rows + cols)
    plans = fused_plans(op, rows, cols)
    assert plans
    try:
        for p in plans:
            assert tr.tr_plan_override(tr.tr_plan(op=tr.OPS[op], order=0, **p)) == tr.TR_OK
            y, h = run(op, d)
            check(op, d, y, h, "unordered", f"{op} {rows}x{cols} plan {p}")
    finally:
        tr.tr_plan_override(None)


@pytest.mark.parametrize("op", OPS)
def test_fused_plans_exclude_streaming_kinds(op):
    # the residual is added at load time: staged, stream and split plans are refused
    code = tr.OPS[op]
    for kind, extra in ((tr.TR_PLAN_STREAM, dict(cluster_ctas=2, vec_slots=0)),
                        (tr.TR_PLAN_SPLIT, dict(cluster_ctas=4, vec_slots=2)),
                        (tr.TR_PLAN_STAGED, dict(cluster_ctas=1, vec_slots=2))):
        p = tr.tr_plan(op=code, order=0, kind=kind, lanes_per_row=32, warps_per_row=8, rows_per_cta=1,
                       block_threads=256, **extra)
        assert tr.tr_plan_override(p) == tr.TR_OK
        try:
            with pytest.raises(tr.TrError) as e:
                tr.tr_plan_describe(code, 16, 8192, 0)
            assert e.value.status == tr.TR_ERR_UNSUPPORTED
        finally:
            tr.tr_plan_override(None)


def test_fused_refusals():
    d = make("add_layernorm", 4, 20000, seed=1)
    with pytest.raises(tr.TrError) as e:        # ordered fused rows must fit 1024 * 16 columns
        run("add_layernorm", d, "ordered")
    assert e.value.status == tr.TR_ERR_UNSUPPORTED
    x = d["x"]
    with pytest.raises(tr.TrError) as e:        # h may not alias x
        tr.add_layernorm(x, d["r"], d["w"], d["b"], h_out=x)
    assert e.value.status == tr.TR_ERR_INVALID_ARG


@pytest.mark.parametrize("order", ["unordered", "ordered"])
@pytest.mark.parametrize("op", OPS)
def test_fused_full_size_768x6144(op, order):
    d = synth.workload_inputs(f"{op}_768x6144", device=DEV)
    y, h = run(op, d, order)
    idx = np.unique(np.linspace(0, 767, 48).astype(np.int64))
    it = torch.as_tensor(idx, device=DEV)
    sub = {k: (v[it] if v.dim() == 2 else v) for k, v in d.items()}
    check(op, sub, y[it], h[it], order, f"{op} {order} 768x6144 sampled rows")
