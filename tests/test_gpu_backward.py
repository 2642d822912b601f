"""GPU parity of the backward passes against the CPU oracle.

Ordered policy: dx and every column gradient bit-identical to the OT-1024
emulation. Unordered policy: within bounds derived from the arithmetic, with
u = 2^-24 and L = ceil(cols / 1024) + 24 (the longest chain of one row sum:
the leaf folds, 2 quad levels, 5 butterfly levels, 3 group levels, plus the
rounding of the steps around it):
  softmax   |e_i| <= L u y_i (sum|dy y| + |dy_i| + |s|)
  xent      |e_i| <= dloss (4e-6 p_i + 2 u |d_i|)   (hardware exp2: 2^-22 plus
            the rounding of the shifted argument)
  RMSNorm   |e_i| <= L u r (|g_i| + |x_i| r^2 (|mean gx| + mean|gx|))
  LayerNorm |e_i| <= L u r (|g_i| + mean|g| + |xh_i| (|b| + mean|g xh|) + |b| r mean|x|)
Column gradients sum per-row terms over the rows (partial folds, then a column
reduction): |e| <= (rows / 8 + L + 40) u sum over rows of |term| (+ the error
of xh, bounded the same way, for dgamma).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import fp32_row_reduction_gb300 as tr

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
U = 2.0 ** -24
SHAPES = [(1, 1), (5, 3), (4, 127), (17, 257), (3, 1024), (7, 1025), (37, 1537), (2, 4096), (9, 6144),
          (3, 8193), (2, 20000), (2, 60000), (1100, 64),
          # the norms' one-pass kernel (aligned rows of 1024 .. 8192 columns): row counts
          # 1, 2, 3 past a leaf quad, the ordered limit of 1024 rows, and 1030 rows (the
          # ordered policy then takes the two-pass kernels; the unordered one more than 256 quads)
          (5, 2048), (6, 3000), (13, 8192), (1024, 1028), (1030, 1024)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def same_bits(got, want, what):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), f"{what}: NaN positions differ"
    bad = bits(got[~nan]) != bits(want[~nan])
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} differ from the emulation"


def within(got, want, bound, what):
    err = np.abs(np.asarray(got, np.float64) - want)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside the bound (worst {np.max(err - bound):.3g})"


def chain(cols):
    return math.ceil(cols / 1024) + 24


def norm_inputs(rows, cols, seed):
    d = synth.make_inputs("layernorm", rows, cols, seed, row_offset=True)
    return d["x"].numpy(), d["w"].numpy(), synth.grad_f32(rows, cols, seed).numpy()


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_softmax_backward(rows, cols):
    x = synth.make_inputs("softmax", rows, cols, seed=rows + cols, var=4.0)["x"].numpy()
    y = oracle.ot_softmax(x)
    dy = synth.grad_f32(rows, cols, rows + cols).numpy()
    for order in ("unordered", "ordered"):
        dx = tr.softmax_backward(dev(y), dev(dy), order=order)
        torch.cuda.synchronize()
        got = dx.cpu().numpy()
        if order == "ordered":
            same_bits(got, oracle.ot_softmax_backward(y, dy), f"softmax bwd {rows}x{cols}")
        else:
            want = oracle.softmax_backward(y, dy)
            y64, d64 = y.astype(np.float64), dy.astype(np.float64)
            s = (y64 * d64).sum(1, keepdims=True)
            bound = chain(cols) * U * y64 * (np.abs(y64 * d64).sum(1, keepdims=True) + np.abs(d64) + np.abs(s))
            within(got, want, bound, f"softmax bwd {rows}x{cols}")


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("scaled", [True, False])
def test_cross_entropy_backward(rows, cols, scaled):
    d = synth.make_inputs("cross_entropy", rows, cols, seed=rows * 3 + cols, var=9.0)
    x, labels = d["x"].numpy(), d["labels"].numpy().copy()
    if rows > 2:
        labels[1] = -1        # outside [0, cols): no one-hot term
        labels[2] = cols
    dl = synth.dloss_f32(rows, seed=rows).numpy() if scaled else None
    for order in ("unordered", "ordered"):
        dx = tr.cross_entropy_backward(dev(x), dev(labels), dev(dl), order=order)
        torch.cuda.synchronize()
        got = dx.cpu().numpy()
        if order == "ordered":
            same_bits(got, oracle.ot_cross_entropy_backward(x, labels, dl), f"xent bwd {rows}x{cols}")
        else:
            want = oracle.cross_entropy_backward(x, labels, dl)
            p = oracle.softmax(x)
            scale = np.ones((rows, 1)) if dl is None else dl.astype(np.float64)[:, None]
            bound = scale * (4e-6 * p + 2 * U * np.abs(want / scale))
            within(got, want, bound, f"xent bwd {rows}x{cols}")


def rms_bounds(x, w, dy, eps):
    x64, d64 = x.astype(np.float64), dy.astype(np.float64)
    n = x.shape[1]
    g = d64 * (1.0 if w is None else w.astype(np.float64))
    r = 1.0 / np.sqrt((x64 * x64).mean(1, keepdims=True) + eps)
    gx = g * x64
    bx = chain(n) * U * r * (np.abs(g) + np.abs(x64) * r * r * (np.abs(gx.mean(1, keepdims=True)) + np.abs(gx).mean(1, keepdims=True)))
    rows = x.shape[0]
    bw = (rows / 8 + chain(n) + 40) * U * np.abs(d64 * x64 * r).sum(0)
    return bx, bw


def ln_bounds(x, gam, dy, eps):
    x64, d64 = x.astype(np.float64), dy.astype(np.float64)
    n = x.shape[1]
    g = d64 * (1.0 if gam is None else gam.astype(np.float64))
    mu = x64.mean(1, keepdims=True)
    r = 1.0 / np.sqrt(((x64 - mu) ** 2).mean(1, keepdims=True) + eps)
    xh = (x64 - mu) * r
    b = (g * xh).mean(1, keepdims=True)
    mx = np.abs(x64).mean(1, keepdims=True)
    L = chain(n)
    bx = L * U * r * (np.abs(g) + np.abs(g).mean(1, keepdims=True) + np.abs(xh) * (np.abs(b) + np.abs(g * xh).mean(1, keepdims=True))
                      + np.abs(b) * r * mx)
    rows = x.shape[0]
    k = rows / 8 + L + 40
    bg = k * U * (np.abs(d64) * (np.abs(xh) + r * mx)).sum(0)
    bb = k * U * np.abs(d64).sum(0)
    return bx, bg, bb


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("affine", [True, False])
def test_rmsnorm_backward(rows, cols, affine):
    x, w, dy = norm_inputs(rows, cols, seed=rows + 5 * cols)
    w = w if affine else None
    for order in ("unordered", "ordered"):
        dx, dw = tr.rmsnorm_backward(dev(x), dev(w), dev(dy), 1e-5, order=order)
        torch.cuda.synchronize()
        gx, gw = dx.cpu().numpy(), dw.cpu().numpy()
        if order == "ordered":
            ex, ew = oracle.ot_rmsnorm_backward(x, w, dy, 1e-5)
            same_bits(gx, ex, f"rms bwd dx {rows}x{cols}")
            same_bits(gw, ew, f"rms bwd dw {rows}x{cols}")
        else:
            ex, ew = oracle.rmsnorm_backward(x, w, dy, 1e-5)
            bx, bw = rms_bounds(x, w, dy, 1e-5)
            within(gx, ex, bx, f"rms bwd dx {rows}x{cols}")
            within(gw, ew, bw, f"rms bwd dw {rows}x{cols}")


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("affine", [True, False])
def test_layernorm_backward(rows, cols, affine):
    x, g, dy = norm_inputs(rows, cols, seed=rows + 7 * cols)
    g = g if affine else None
    for order in ("unordered", "ordered"):
        dx, dg, db = tr.layernorm_backward(dev(x), dev(g), dev(dy), 1e-5, order=order)
        torch.cuda.synchronize()
        got = [t.cpu().numpy() for t in (dx, dg, db)]
        if order == "ordered":
            want = oracle.ot_layernorm_backward(x, g, dy, 1e-5)
            for a, b, nm in zip(got, want, ("dx", "dgamma", "dbeta")):
                same_bits(a, b, f"ln bwd {nm} {rows}x{cols}")
        else:
            want = oracle.layernorm_backward(x, g, dy, 1e-5)
            for a, b, bd, nm in zip(got, want, ln_bounds(x, g, dy, 1e-5), ("dx", "dgamma", "dbeta")):
                within(a, b, bd, f"ln bwd {nm} {rows}x{cols}")


def test_dx_only_and_workspace_errors():
    x, w, dy = norm_inputs(6, 3000, seed=1)
    dx, dw = tr.rmsnorm_backward(dev(x), dev(w), dev(dy), want_dw=False)
    dx2, dg, db = tr.layernorm_backward(dev(x), dev(w), dev(dy), want_params=False)
    torch.cuda.synchronize()
    assert dw is None and dg is None and db is None
    same_bits(tr.rmsnorm_backward(dev(x), dev(w), dev(dy), order="ordered", want_dw=False)[0].cpu().numpy(),
              oracle.ot_rmsnorm_backward(x, w, dy)[0], "rms dx only")
    lib = tr.load()
    X, W, DY = dev(x), dev(w), dev(dy)
    DX, DW = torch.empty_like(X), torch.empty(3000, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    need = tr.norm_backward_workspace_bytes(6, 3000)
    assert need == 2 * 3000 * 2 * 4            # the one-pass kernel's partials: 2 leaf quads x 3000 columns x 2
    assert tr.norm_backward_workspace_bytes(6, 3001) == 6 * 2 * 4                 # two statistics per row
    small = torch.empty(need, dtype=torch.uint8, device=DEV)
    assert lib.tr_rmsnorm_backward_f32(X.data_ptr(), W.data_ptr(), DY.data_ptr(), DX.data_ptr(), DW.data_ptr(), 6, 3000,
                                       1e-5, 0, small.data_ptr(), need - 4, s) == tr.TR_ERR_INVALID_ARG
    assert lib.tr_rmsnorm_backward_f32(X.data_ptr(), W.data_ptr(), DY.data_ptr(), X.data_ptr(), None, 6, 3000,
                                       1e-5, 0, None, 0, s) == tr.TR_ERR_INVALID_ARG     # dx aliases x
    assert lib.tr_softmax_backward_f32(X.data_ptr(), DY.data_ptr(), DY.data_ptr(), 6, 3000, 0, s) == tr.TR_ERR_INVALID_ARG


def test_full_size_768x6144():
    rows, cols = 768, 6144
    x, g, dy = norm_inputs(rows, cols, seed=2)
    for order in ("unordered", "ordered"):
        got = [t.cpu().numpy() for t in tr.layernorm_backward(dev(x), dev(g), dev(dy), 1e-5, order=order)]
        if order == "ordered":
            for a, b, nm in zip(got, oracle.ot_layernorm_backward(x, g, dy, 1e-5), ("dx", "dgamma", "dbeta")):
                same_bits(a, b, f"ln bwd {nm} 768x6144")
        else:
            want = oracle.layernorm_backward(x, g, dy, 1e-5)
            for a, b, bd, nm in zip(got, want, ln_bounds(x, g, dy, 1e-5), ("dx", "dgamma", "dbeta")):
                within(a, b, bd, f"ln bwd {nm} 768x6144")


def offset_copy(a, off):
    """A copy of the float32 array a in device memory starting `off` floats past a 16-byte boundary."""
    big = torch.empty(a.size + 8, device=DEV)
    v = big[off:off + a.size].view(*a.shape)
    v.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return v


@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 2, 3), (3, 1, 2)])
def test_unaligned_tensors(offs):
    rows, cols = 5, 3001
    x, g, dy = norm_inputs(rows, cols, seed=sum(offs) + 3)
    X, DY = offset_copy(x, offs[0]), offset_copy(dy, offs[1])
    for order in ("unordered", "ordered"):
        big = torch.zeros(rows * cols + 8, device=DEV)
        DX = big[offs[2]:offs[2] + rows * cols].view(rows, cols)
        dx, dg, db = tr.layernorm_backward(X, dev(g), DY, 1e-5, order=order, dx=DX)
        torch.cuda.synchronize()
        got = [t.cpu().numpy() for t in (dx, dg, db)]
        if order == "ordered":
            for a, b, nm in zip(got, oracle.ot_layernorm_backward(x, g, dy, 1e-5), ("dx", "dgamma", "dbeta")):
                same_bits(a, b, f"ln bwd {nm} offsets {offs}")
        else:
            want = oracle.layernorm_backward(x, g, dy, 1e-5)
            for a, b, bd, nm in zip(got, want, ln_bounds(x, g, dy, 1e-5), ("dx", "dgamma", "dbeta")):
                within(a, b, bd, f"ln bwd {nm} offsets {offs}")
        y = oracle.ot_softmax(x)
        Y = offset_copy(y, offs[0])
        big2 = torch.zeros(rows * cols + 8, device=DEV)
        DX2 = big2[offs[2]:offs[2] + rows * cols].view(rows, cols)
        tr.softmax_backward(Y, DY, out=DX2, order=order)
        torch.cuda.synchronize()
        if order == "ordered":
            same_bits(DX2.cpu().numpy(), oracle.ot_softmax_backward(y, dy), f"softmax bwd offsets {offs}")
        labels = synth.labels_i64(rows, cols, seed=7)
        L = offset_copy(x, offs[1])
        big3 = torch.zeros(rows * cols + 8, device=DEV)
        DL = big3[offs[2]:offs[2] + rows * cols].view(rows, cols)
        tr.cross_entropy_backward(L, labels.to(DEV), None, out=DL, order=order)
        torch.cuda.synchronize()
        if order == "ordered":
            same_bits(DL.cpu().numpy(), oracle.ot_cross_entropy_backward(x, labels.numpy()), f"xent bwd offsets {offs}")


@pytest.mark.parametrize("offs", [(0, 0), (1, 0), (0, 3), (2, 1)])
@pytest.mark.parametrize("rows,cols", [(3, 8193), (4, 20001), (2, 100003)])
def test_cross_entropy_backward_long_rows_unaligned(rows, cols, offs):
    # rows longer than the cached kernels take run the streaming kernel (a
    # 1024-thread CTA per row): row heads and tails of every phase, dlogits on
    # the logits' 16-byte phase or off it, labels on the head, the tail, a
    # quad's last lane and out of range; the guard floats stay untouched
    x = synth.make_inputs("cross_entropy", rows, cols, seed=cols + 11 * offs[0] + offs[1], var=9.0)["x"].numpy()
    labels = np.array([0, cols - 1, 7, -3][:rows], dtype=np.int64)
    dl = synth.dloss_f32(rows, seed=cols).numpy()
    L = offset_copy(x, offs[0])
    big = torch.zeros(rows * cols + 8, device=DEV)
    DL = big[offs[1]:offs[1] + rows * cols].view(rows, cols)
    tr.cross_entropy_backward(L, torch.from_numpy(labels).to(DEV), dev(dl), out=DL, order="unordered")
    torch.cuda.synchronize()
    want = oracle.cross_entropy_backward(x, labels, dl)
    p = oracle.softmax(x)
    scale = dl.astype(np.float64)[:, None]
    within(DL.cpu().numpy(), want, scale * (4e-6 * p + 2 * U * np.abs(want / scale)),
           f"xent bwd {rows}x{cols} offsets {offs}")
    assert float(big[:offs[1]].abs().sum()) == 0.0 and float(big[offs[1] + rows * cols:].abs().sum()) == 0.0


def test_cross_entropy_backward_full_size_sampled_rows():
    # the 4096 x 50257 workload through the streaming kernel; sampled rows
    # against the oracle, and every row of dlogits sums to 0 (in-range labels)
    rows, cols = 4096, 50257
    d = synth.make_inputs("cross_entropy", rows, cols, seed=3, var=9.0)
    dx = tr.cross_entropy_backward(d["x"].to(DEV), d["labels"].to(DEV), None, order="unordered")
    torch.cuda.synchronize()
    pick = [0, 1, 777, 2048, 4095]
    x = d["x"].numpy()[pick]
    labels = d["labels"].numpy()[pick]
    want = oracle.cross_entropy_backward(x, labels, None)
    p = oracle.softmax(x)
    within(dx[pick].cpu().numpy(), want, 4e-6 * p + 2 * U * np.abs(want), "xent bwd 4096x50257 sampled")
    sums = dx.double().sum(1).abs().max().item()
    assert sums < 1e-4, sums
