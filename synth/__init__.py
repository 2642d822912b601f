"""Seeded synthetic inputs for the row-reduction workloads.

This module is shared by the tests, the benchmark and the CPU oracle checks.
It holds none of the reductions' arithmetic: it only turns (seed, tensor tag,
element index) into random numbers and shapes them into the distributions the
workloads use.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used in counter form: draw ``i`` of a stream
is ``mix64(base + (i + 1) * GOLDEN)``, so any element can be produced on its own
and a tensor can be generated in slices, on the CPU or on a GPU, with the same
integer results.  Uniforms take the top 53 bits; normals use the Box–Muller
transform (cosine branch) in float64 and are rounded to float32 once.

Distribution notation follows the workload descriptions: ``N(mu, v)`` is a
normal with mean ``mu`` and VARIANCE ``v`` (so ``N(0, 2^2)`` has sigma 2 and the
bias ``N(0, 0.1)`` has sigma sqrt(0.1)); ``U(a, b)`` is uniform on [a, b).
"""
from __future__ import annotations

import math

import torch

_MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
_MUL1 = 0xBF58476D1CE4E5B9
_MUL2 = 0x94D049BB133111EB

# tensor tags: one independent stream per (seed, tag)
TAG_X = 1
TAG_W = 2
TAG_B = 3
TAG_LABELS = 4
TAG_ROW_OFFSET = 5
TAG_RESIDUAL = 6
TAG_DY = 7
TAG_DLOSS = 8

_CHUNK = 1 << 23  # elements generated per slice (bounds temporary memory)


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit value as the signed int64 torch stores."""
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (reference form)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _MUL1) & _MASK64
    z = ((z ^ (z >> 27)) * _MUL2) & _MASK64
    return z ^ (z >> 31)


def stream_base(seed: int, tag: int) -> int:
    """Base counter of the stream for one tensor of one workload."""
    return mix64_int(mix64_int(seed) ^ (tag * 0x5851F42D4C957F2D))


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return torch.bitwise_and(torch.bitwise_right_shift(z, k), (1 << (64 - k)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = torch.bitwise_xor(z, _lsr(z, 30)) * _s64(_MUL1)
    z = torch.bitwise_xor(z, _lsr(z, 27)) * _s64(_MUL2)
    return torch.bitwise_xor(z, _lsr(z, 31))


def raw_u64(seed: int, tag: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Draws ``start .. start+count-1`` of stream (seed, tag) as int64 bit patterns."""
    base = stream_base(seed, tag)
    i = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = i * _s64(GOLDEN) + _s64(base)
    return _mix64(z)


def _unit53(z: torch.Tensor) -> torch.Tensor:
    """Top 53 bits -> float64 in [0, 1)."""
    return _lsr(z, 11).to(torch.float64) * (2.0 ** -53)


def uniform01(seed, tag, n, device="cpu", start=0) -> torch.Tensor:
    """float64 uniforms in [0, 1)."""
    out = torch.empty(n, dtype=torch.float64, device=device)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = _unit53(raw_u64(seed, tag, start + s, c, device))
    return out


def _std_normal_f64(seed, tag, start, count, device) -> torch.Tensor:
    z = raw_u64(seed, tag, 2 * start, 2 * count, device).view(count, 2)
    u1 = (_lsr(z[:, 0], 11).to(torch.float64) + 0.5) * (2.0 ** -53)  # (0, 1)
    u2 = _unit53(z[:, 1])
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal_f32(shape, seed, tag, mean=0.0, var=1.0, device="cpu") -> torch.Tensor:
    """float32 tensor of i.i.d. N(mean, var) (var is the variance)."""
    n = math.prod(shape)
    sd = math.sqrt(var)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = (mean + sd * _std_normal_f64(seed, tag, s, c, device)).to(torch.float32)
    return out.view(*shape)


def uniform_f32(shape, seed, tag, lo, hi, device="cpu") -> torch.Tensor:
    n = math.prod(shape)
    u = uniform01(seed, tag, n, device)
    return (lo + (hi - lo) * u).to(torch.float32).view(*shape)


def normal_plus_row_offset_f32(rows, cols, seed, lo=-3.0, hi=3.0, device="cpu") -> torch.Tensor:
    """x[r, c] = N(0,1) + o_r with one o_r ~ U(lo, hi) per row, summed in float64, rounded once."""
    off = lo + (hi - lo) * uniform01(seed, TAG_ROW_OFFSET, rows, device)
    out = torch.empty(rows, cols, dtype=torch.float32, device=device)
    # whole rows per slice (a row longer than a slice is split): the offsets are
    # broadcast from plain slices of `off`, no gather
    rows_per = max(1, _CHUNK // cols)
    for r0 in range(0, rows, rows_per):
        r1 = min(rows, r0 + rows_per)
        if r1 - r0 > 1 or cols <= _CHUNK:
            z = _std_normal_f64(seed, TAG_X, r0 * cols, (r1 - r0) * cols, device).view(r1 - r0, cols)
            out[r0:r1] = (z + off[r0:r1].view(-1, 1)).to(torch.float32)
        else:
            for c0 in range(0, cols, _CHUNK):
                c = min(_CHUNK, cols - c0)
                z = _std_normal_f64(seed, TAG_X, r0 * cols + c0, c, device)
                out[r0, c0:c0 + c] = (z + off[r0:r0 + 1]).to(torch.float32)
    return out


def labels_i64(rows, classes, seed, device="cpu") -> torch.Tensor:
    """int64 labels uniform in [0, classes)."""
    u = uniform01(seed, TAG_LABELS, rows, device)
    return torch.clamp(torch.floor(u * classes).to(torch.int64), max=classes - 1)


# ---------------------------------------------------------------------------
# The workloads.  Each returns a dict of float32 / int64 tensors.
# ---------------------------------------------------------------------------

def softmax_inputs(rows, cols, seed, var=1.0, device="cpu"):
    return {"x": normal_f32((rows, cols), seed, TAG_X, 0.0, var, device)}


def norm_inputs(rows, cols, seed, row_offset=False, device="cpu"):
    if row_offset:
        x = normal_plus_row_offset_f32(rows, cols, seed, device=device)
    else:
        x = normal_f32((rows, cols), seed, TAG_X, 0.0, 1.0, device)
    w = uniform_f32((cols,), seed, TAG_W, 0.5, 1.5, device)
    b = normal_f32((cols,), seed, TAG_B, 0.0, 0.1, device)
    return {"x": x, "w": w, "b": b}


def residual_norm_inputs(rows, cols, seed, row_offset=False, device="cpu"):
    """Norm inputs plus a residual r ~ N(0, 1), i.i.d. per element."""
    d = norm_inputs(rows, cols, seed, row_offset, device)
    d["r"] = normal_f32((rows, cols), seed, TAG_RESIDUAL, 0.0, 1.0, device)
    return d


def xent_inputs(rows, cols, seed, var=9.0, device="cpu"):
    return {"x": normal_f32((rows, cols), seed, TAG_X, 0.0, var, device),
            "labels": labels_i64(rows, cols, seed, device)}


# The five workload families, with the seeds and distributions they are quoted with.
WORKLOADS = {
    "softmax_37x1537": dict(op="softmax", rows=37, cols=1537, seed=0, var=4.0),
    "rmsnorm_256x3072": dict(op="rmsnorm", rows=256, cols=3072, seed=1, row_offset=True),
    "layernorm_256x3072": dict(op="layernorm", rows=256, cols=3072, seed=1, row_offset=True),
    "rmsnorm_64x12289": dict(op="rmsnorm", rows=64, cols=12289, seed=1, row_offset=True),
    "layernorm_64x12289": dict(op="layernorm", rows=64, cols=12289, seed=1, row_offset=True),
    "softmax_768x6144": dict(op="softmax", rows=768, cols=6144, seed=2, var=1.0),
    "rmsnorm_768x6144": dict(op="rmsnorm", rows=768, cols=6144, seed=2),
    "layernorm_768x6144": dict(op="layernorm", rows=768, cols=6144, seed=2),
    "cross_entropy_4096x50257": dict(op="cross_entropy", rows=4096, cols=50257, seed=3, var=9.0),
    "softmax_16x65536": dict(op="softmax", rows=16, cols=65536, seed=4, var=1.0),
    "softmax_16x262144": dict(op="softmax", rows=16, cols=262144, seed=4, var=1.0),
    "softmax_16x1048576": dict(op="softmax", rows=16, cols=1048576, seed=4, var=1.0),
    "softmax_65536x128": dict(op="softmax", rows=65536, cols=128, seed=4, var=1.0),
    "layernorm_16x65536": dict(op="layernorm", rows=16, cols=65536, seed=4),
    "layernorm_16x262144": dict(op="layernorm", rows=16, cols=262144, seed=4),
    "layernorm_16x1048576": dict(op="layernorm", rows=16, cols=1048576, seed=4),
    "layernorm_65536x128": dict(op="layernorm", rows=65536, cols=128, seed=4),
    # fused residual norms (x and w, b as the 768x6144 family, residual ~ N(0, 1))
    "add_rmsnorm_768x6144": dict(op="add_rmsnorm", rows=768, cols=6144, seed=2),
    "add_layernorm_768x6144": dict(op="add_layernorm", rows=768, cols=6144, seed=2),
    # standalone row reductions, x ~ N(0, 1)
    "row_sum_768x6144": dict(op="row_sum", rows=768, cols=6144, seed=2),
    "row_minmax_768x6144": dict(op="row_minmax", rows=768, cols=6144, seed=2),
    # backward passes: upstream gradients dy ~ N(0, 1), dloss ~ U(0.5, 1.5); the softmax
    # backward's y is the forward softmax of x ~ N(0, 1), computed by the caller
    "softmax_bwd_768x6144": dict(op="softmax_bwd", rows=768, cols=6144, seed=2, var=1.0),
    "rmsnorm_bwd_768x6144": dict(op="rmsnorm_bwd", rows=768, cols=6144, seed=2),
    "layernorm_bwd_768x6144": dict(op="layernorm_bwd", rows=768, cols=6144, seed=2),
    "cross_entropy_bwd_4096x50257": dict(op="cross_entropy_bwd", rows=4096, cols=50257, seed=3, var=9.0),
    # reductions over axis 0 (one value per column), x ~ N(0, 1)
    "axis_sum_768x6144": dict(op="axis_sum", rows=768, cols=6144, seed=2),
    "axis_minmax_768x6144": dict(op="axis_minmax", rows=768, cols=6144, seed=2),
}


def grad_f32(rows, cols, seed, device="cpu"):
    """An upstream gradient dy ~ N(0, 1), i.i.d. per element."""
    return normal_f32((rows, cols), seed, TAG_DY, 0.0, 1.0, device)


def dloss_f32(rows, seed, device="cpu"):
    """A per-row upstream loss gradient ~ U(0.5, 1.5)."""
    return uniform_f32((rows,), seed, TAG_DLOSS, 0.5, 1.5, device)


def make_inputs(op, rows, cols, seed, var=None, row_offset=False, device="cpu"):
    """Inputs of one workload: softmax/cross_entropy use ``var``; norms use ``row_offset``."""
    if op == "softmax":
        return softmax_inputs(rows, cols, seed, 1.0 if var is None else var, device)
    if op in ("rmsnorm", "layernorm"):
        return norm_inputs(rows, cols, seed, row_offset, device)
    if op == "cross_entropy":
        return xent_inputs(rows, cols, seed, 9.0 if var is None else var, device)
    if op in ("add_rmsnorm", "add_layernorm"):
        return residual_norm_inputs(rows, cols, seed, row_offset, device)
    if op == "softmax_bwd":
        return {"x": normal_f32((rows, cols), seed, TAG_X, 0.0, 1.0 if var is None else var, device),
                "dy": grad_f32(rows, cols, seed, device)}
    if op == "cross_entropy_bwd":
        d = xent_inputs(rows, cols, seed, 9.0 if var is None else var, device)
        d["dloss"] = dloss_f32(rows, seed, device)
        return d
    if op in ("rmsnorm_bwd", "layernorm_bwd"):
        d = norm_inputs(rows, cols, seed, row_offset, device)
        d.pop("b")
        d["dy"] = grad_f32(rows, cols, seed, device)
        return d
    if op in ("row_sum", "row_max", "row_min", "row_minmax", "axis_sum", "axis_max", "axis_min", "axis_minmax"):
        return {"x": normal_plus_row_offset_f32(rows, cols, seed, device=device) if row_offset
                else normal_f32((rows, cols), seed, TAG_X, 0.0, 1.0 if var is None else var, device)}
    raise ValueError(f"unknown op {op!r}")


def workload_inputs(name, device="cpu"):
    w = dict(WORKLOADS[name])
    op = w.pop("op")
    return make_inputs(op, device=device, **w)
