"""GPU parity of the split-row plan (TR_PLAN_SPLIT) against the CPU oracle.

A row is cut into C segments on C co-resident CTAs that exchange partial
statistics through a per-stream workspace ("TIRx Metal reduction lowering"
§4.2, the combine of cooperating workers, one level above a CTA). Covered:
segments fully cached, partly cached (overflow streamed and re-read) and not
cached; ragged and unaligned rows; up to 32 CTAs per row; repeated launches on
one workspace; two streams; CUDA-graph replay after a warm call; the refusal
of a first call under capture; and the special rows of the softmax.
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
NORM_OPS = ["softmax", "rmsnorm", "layernorm"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr.load()
    yield
    tr.tr_plan_override(None)


@pytest.fixture(autouse=True)
def _clear_override():
    yield
    tr.tr_plan_override(None)


def split(op, C, T, K):
    return tr.tr_plan(op=tr.OPS[op], order=0, kind=tr.TR_PLAN_SPLIT, lanes_per_row=32, warps_per_row=T // 32,
                      rows_per_cta=1, cluster_ctas=C, vec_slots=K, block_threads=T)


def make(op, rows, cols, seed):
    if op == "softmax":
        return synth.make_inputs(op, rows, cols, seed, var=4.0, device=DEV)
    return synth.make_inputs(op, rows, cols, seed, row_offset=True, device=DEV)


def reference(op, h, eps=1e-5):
    if op == "softmax":
        return oracle.softmax(h["x"])
    if op == "rmsnorm":
        return oracle.rmsnorm(h["x"], h.get("w"), eps)
    return oracle.layernorm(h["x"], h.get("w"), h.get("b"), eps)


def host(d):
    return {k: v.cpu().numpy() for k, v in d.items()}


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={got[i]!r} oracle={ref[i]!r}")


def run_split(op, d, C, T, K, stream=None):
    assert tr.tr_plan_override(split(op, C, T, K)) == tr.TR_OK
    y = tr.run_op(op, d, stream=stream)
    torch.cuda.synchronize()
    assert tr.tr_last_device_error() == tr.TR_OK
    return y


# (rows, cols, C, T, K): all cached, partly cached, not cached, many segments
CASES = [
    (3, 4096, 2, 256, 2),      # each segment fully cached
    (3, 70001, 4, 256, 3),     # ragged row; overflow streamed
    (5, 100003, 7, 512, 0),    # nothing cached: pure streaming
    (16, 65536, 9, 1024, 14),  # the long-row workload, one CTA per SM
    (2, 262147, 32, 256, 1),   # 32 segments, odd width
    (1, 1, 2, 64, 1),          # one element: the second segment is empty
    (4, 5, 3, 64, 1),          # fewer 16-byte slots than segments
]


@pytest.mark.parametrize("rows,cols,C,T,K", CASES)
@pytest.mark.parametrize("op", NORM_OPS)
def test_split_matches_oracle(op, rows, cols, C, T, K):
    d = make(op, rows, cols, seed=rows * 31 + cols + C)
    y = run_split(op, d, C, T, K)
    assert_close(y.cpu().numpy(), reference(op, host(d)), f"split {op} {rows}x{cols} C={C} T={T} K={K}")


@pytest.mark.parametrize("xoff,yoff,woff", [(1, 1, 0), (3, 0, 1), (2, 2, 3)])
@pytest.mark.parametrize("op", NORM_OPS)
def test_split_unaligned_rows_outputs_and_weights(op, xoff, yoff, woff):
    rows, cols = 3, 50001
    d = make(op, rows, cols, seed=11 + xoff + 4 * yoff + 16 * woff)
    ref = reference(op, host(d))
    xbig = torch.empty(rows * cols + 8, device=DEV)
    x = xbig[xoff:xoff + rows * cols].view(rows, cols)
    x.copy_(d["x"])
    ybig = torch.zeros(rows * cols + 8, device=DEV)
    y = ybig[yoff:yoff + rows * cols].view(rows, cols)
    d2 = dict(d, x=x)
    for key in ("w", "b"):
        if key in d:
            big = torch.empty(cols + 8, device=DEV)
            v = big[woff:woff + cols]
            v.copy_(d[key])
            d2[key] = v
    assert tr.tr_plan_override(split(op, 5, 256, 4)) == tr.TR_OK
    tr.run_op(op, d2, out=y)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, f"split {op} x+{xoff} y+{yoff} w+{woff}")
    assert float(ybig[:yoff].abs().sum()) == 0.0 and float(ybig[yoff + rows * cols:].abs().sum()) == 0.0


@pytest.mark.parametrize("op", NORM_OPS)
def test_split_repeated_launches_reuse_the_workspace(op):
    # the last CTA of each row clears the row's counters, so back-to-back
    # launches on one stream (no host work in between) give identical bits
    d = make(op, 16, 65536, seed=5)
    assert tr.tr_plan_override(split(op, 8, 512, 4)) == tr.TR_OK
    ys = [tr.run_op(op, d) for _ in range(6)]
    torch.cuda.synchronize()
    assert tr.tr_last_device_error() == tr.TR_OK
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32))
    assert_close(ys[-1].cpu().numpy(), reference(op, host(d)), f"split {op} repeated")


def test_split_on_two_streams():
    # each stream has its own workspace: concurrent split launches never share counters
    d1 = make("softmax", 12, 100000, seed=1)
    d2 = make("layernorm", 12, 100000, seed=2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    tr.tr_plan_override(split("softmax", 6, 256, 2))
    tr.tr_plan_override(split("layernorm", 6, 256, 2))
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            a = tr.run_op("softmax", d1, stream=s1)
        with torch.cuda.stream(s2):
            b = tr.run_op("layernorm", d2, stream=s2)
        outs.append((a, b))
    torch.cuda.synchronize()
    assert tr.tr_last_device_error() == tr.TR_OK
    ra, rb = reference("softmax", host(d1)), reference("layernorm", host(d2))
    for a, b in outs:
        assert_close(a.cpu().numpy(), ra, "split softmax on stream 1")
        assert_close(b.cpu().numpy(), rb, "split layernorm on stream 2")


def test_split_graph_replay_after_a_warm_call():
    d = make("rmsnorm", 16, 65536, seed=9)
    y = torch.empty_like(d["x"])
    s = torch.cuda.Stream()
    tr.tr_plan_override(split("rmsnorm", 9, 1024, 4))
    with torch.cuda.stream(s):
        tr.run_op("rmsnorm", d, out=y, stream=s)   # allocates this stream's workspace
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tr.run_op("rmsnorm", d, out=y, stream=s)
    ref = reference("rmsnorm", host(d))
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), ref, "split rmsnorm graph replay")
    assert tr.tr_last_device_error() == tr.TR_OK


def test_split_first_call_under_capture_is_refused():
    # the workspace is allocated on a stream's first split call; under capture
    # that is refused with an error (no allocation, no launch)
    d = make("softmax", 4, 40000, seed=4)
    y = torch.empty_like(d["x"])
    s = torch.cuda.Stream()
    tr.tr_plan_override(split("softmax", 4, 256, 2))
    tr.run_op("softmax", d, out=y)   # plan and occupancy cached; another stream's workspace
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    err = None
    with torch.cuda.graph(g, stream=s):
        try:
            tr.run_op("softmax", d, out=y, stream=s)
        except tr.TrError as e:
            err = e
    assert err is not None and err.status == tr.TR_ERR_UNSUPPORTED
    assert "captur" in str(err)


def test_split_special_softmax_rows():
    x = torch.zeros(7, 60000, device=DEV)
    x[1] = 5.0                        # constant row
    x[2, 17] = 80.0                   # one dominant logit in the first segment
    x[3] = torch.linspace(-30, 30, 60000, device=DEV)
    x[4, ::2] = -1e30                 # huge negative entries
    x[5, :30000] = float("-inf")      # first segments hold only -inf
    x[6, 59999] = 1e4                 # the maximum in the last segment's overflow
    tr.tr_plan_override(split("softmax", 4, 256, 4))
    y = tr.softmax(x)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), oracle.softmax(x.cpu().numpy()), "special softmax rows")
