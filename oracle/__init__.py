"""CPU oracle for the FP32 row reductions: TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package.  The product path (the CUDA library and its
Python binding) never imports it and shares no code with it.

Wraps ``oracle.c`` (plain serial C): the FP64 definitions of softmax, RMSNorm,
LayerNorm and cross-entropy and of their gradients, and the bit-exact FP32
emulation of the ordered fixed-tree policy (OT-1024) with its own exp/log.  Arrays are numpy; inputs
are float32 (labels int64) row-major, FP64 outputs are returned as float64 and
emulated outputs as float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

# -ffp-contract=off: no a*b+c fusion (the emulation must round every op);
# no -ffast-math; -O2 keeps IEEE semantics.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-finite-math-only", "-Wall"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, a second or so)."""
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        sig = {
            "oracle_softmax_f64": [f32p, f64p, i64, i64],
            "oracle_rmsnorm_f64": [f32p, f32p, f64p, i64, i64, ctypes.c_float],
            "oracle_layernorm_f64": [f32p, f32p, f32p, f64p, i64, i64, ctypes.c_float],
            "oracle_cross_entropy_f64": [f32p, i64p, f64p, i64, i64],
            "ot_softmax_f32": [f32p, f32p, i64, i64],
            "ot_rmsnorm_f32": [f32p, f32p, f32p, i64, i64, ctypes.c_float],
            "ot_layernorm_f32": [f32p, f32p, f32p, f32p, i64, i64, ctypes.c_float],
            "ot_cross_entropy_f32": [f32p, i64p, f32p, i64, i64],
            "oracle_softmax_bwd_f64": [f32p, f32p, f64p, i64, i64],
            "oracle_cross_entropy_bwd_f64": [f32p, i64p, f32p, f64p, i64, i64],
            "oracle_rmsnorm_bwd_f64": [f32p, f32p, f32p, f64p, f64p, i64, i64, ctypes.c_float],
            "oracle_layernorm_bwd_f64": [f32p, f32p, f32p, f64p, f64p, f64p, i64, i64, ctypes.c_float],
            "ot_softmax_bwd_f32": [f32p, f32p, f32p, i64, i64],
            "ot_cross_entropy_bwd_f32": [f32p, i64p, f32p, f32p, i64, i64],
            "ot_rmsnorm_bwd_f32": [f32p, f32p, f32p, f32p, f32p, i64, i64, ctypes.c_float],
            "ot_layernorm_bwd_f32": [f32p, f32p, f32p, f32p, f32p, f32p, i64, i64, ctypes.c_float],
            "fold_softmax_f32": [f32p, f32p, i64, i64, ctypes.c_int],
            "fold_rmsnorm_f32": [f32p, f32p, f32p, i64, i64, ctypes.c_float, ctypes.c_int],
            "fold_layernorm_f32": [f32p, f32p, f32p, f32p, i64, i64, ctypes.c_float, ctypes.c_int],
            "fold_cross_entropy_f32": [f32p, i64p, f32p, i64, i64, ctypes.c_int],
            "ot_sum_f32": [f32p, i64],
            "ot_max_f32": [f32p, i64],
            "ot_min_f32": [f32p, i64],
            "skipnan_row_max_f32": [f32p, f32p, i64, i64],
            "skipnan_row_min_f32": [f32p, f32p, i64, i64],
            "skipnan_axis_max_f32": [f32p, f32p, i64, i64, i64],
            "skipnan_axis_min_f32": [f32p, f32p, i64, i64, i64],
        }
        for name, args in sig.items():
            fn = getattr(_lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_float if name in ("ot_sum_f32", "ot_max_f32", "ot_min_f32") else ctypes.c_int
        for name in ("fold_sum_f32", "fold_max_f32", "fold_min_f32"):
            fn = getattr(_lib, name)
            fn.argtypes = [f32p, i64, ctypes.c_int]
            fn.restype = ctypes.c_float
        for name in ("ot_expf", "ot_logf"):
            fn = getattr(_lib, name)
            fn.argtypes = [ctypes.c_float]
            fn.restype = ctypes.c_float
        for name in ("ot_expf_n", "ot_logf_n"):
            fn = getattr(_lib, name)
            fn.argtypes = [f32p, f32p, i64]
            fn.restype = None
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _rc(code):
    if code != 0:
        raise ValueError("oracle rejected the sizes")


# --- FP64 definitions ------------------------------------------------------

def softmax(x):
    x = _f32(x)
    r, c = x.shape
    y = np.empty((r, c), np.float64)
    _rc(lib().oracle_softmax_f64(_ptr(x, ctypes.c_float), _ptr(y, ctypes.c_double), r, c))
    return y


def rmsnorm(x, w=None, eps=1e-5):
    x = _f32(x)
    w = None if w is None else _f32(w)
    r, c = x.shape
    y = np.empty((r, c), np.float64)
    _rc(lib().oracle_rmsnorm_f64(_ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float),
                                 _ptr(y, ctypes.c_double), r, c, eps))
    return y


def layernorm(x, gamma=None, beta=None, eps=1e-5):
    x = _f32(x)
    gamma = None if gamma is None else _f32(gamma)
    beta = None if beta is None else _f32(beta)
    r, c = x.shape
    y = np.empty((r, c), np.float64)
    _rc(lib().oracle_layernorm_f64(_ptr(x, ctypes.c_float), _ptr(gamma, ctypes.c_float),
                                   _ptr(beta, ctypes.c_float), _ptr(y, ctypes.c_double),
                                   r, c, eps))
    return y


def cross_entropy(logits, labels):
    x = _f32(logits)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    r, c = x.shape
    loss = np.empty(r, np.float64)
    _rc(lib().oracle_cross_entropy_f64(_ptr(x, ctypes.c_float), _ptr(lab, ctypes.c_int64),
                                       _ptr(loss, ctypes.c_double), r, c))
    return loss


# --- OT-1024 emulation -----------------------------------------------------

def residual_sum(x, r):
    """h = x + r for the fused residual norms: one IEEE binary32 addition per
    element ("TIRx Metal reduction lowering" §5.1: combined = X + residual),
    numpy's float32 add (round to nearest even)."""
    return (_f32(x) + _f32(r)).astype(np.float32)


def add_rmsnorm(x, r, w=None, eps=1e-5):
    """RMSNorm of the FP32 row h = x + r (FP64 definition applied to h); returns (y, h)."""
    h = residual_sum(x, r)
    return rmsnorm(h, w, eps), h


def add_layernorm(x, r, gamma=None, beta=None, eps=1e-5):
    """LayerNorm of the FP32 row h = x + r (FP64 definition applied to h); returns (y, h)."""
    h = residual_sum(x, r)
    return layernorm(h, gamma, beta, eps), h


def ot_add_rmsnorm(x, r, w=None, eps=1e-5):
    """Ordered-policy emulation of the fused residual RMSNorm: OT-1024 on h = x + r."""
    h = residual_sum(x, r)
    return ot_rmsnorm(h, w, eps), h


def ot_add_layernorm(x, r, gamma=None, beta=None, eps=1e-5):
    """Ordered-policy emulation of the fused residual LayerNorm: OT-1024 on h = x + r."""
    h = residual_sum(x, r)
    return ot_layernorm(h, gamma, beta, eps), h


def ot_softmax(x):
    x = _f32(x)
    r, c = x.shape
    y = np.empty((r, c), np.float32)
    _rc(lib().ot_softmax_f32(_ptr(x, ctypes.c_float), _ptr(y, ctypes.c_float), r, c))
    return y


def ot_rmsnorm(x, w=None, eps=1e-5):
    x = _f32(x)
    w = None if w is None else _f32(w)
    r, c = x.shape
    y = np.empty((r, c), np.float32)
    _rc(lib().ot_rmsnorm_f32(_ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float),
                             _ptr(y, ctypes.c_float), r, c, eps))
    return y


def ot_layernorm(x, gamma=None, beta=None, eps=1e-5):
    x = _f32(x)
    gamma = None if gamma is None else _f32(gamma)
    beta = None if beta is None else _f32(beta)
    r, c = x.shape
    y = np.empty((r, c), np.float32)
    _rc(lib().ot_layernorm_f32(_ptr(x, ctypes.c_float), _ptr(gamma, ctypes.c_float),
                               _ptr(beta, ctypes.c_float), _ptr(y, ctypes.c_float), r, c, eps))
    return y


def ot_cross_entropy(logits, labels):
    x = _f32(logits)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    r, c = x.shape
    loss = np.empty(r, np.float32)
    _rc(lib().ot_cross_entropy_f32(_ptr(x, ctypes.c_float), _ptr(lab, ctypes.c_int64),
                                   _ptr(loss, ctypes.c_float), r, c))
    return loss


def ot_sum(v):
    v = _f32(v).ravel()
    return np.float32(lib().ot_sum_f32(_ptr(v, ctypes.c_float), v.size))


def ot_max(v):
    v = _f32(v).ravel()
    return np.float32(lib().ot_max_f32(_ptr(v, ctypes.c_float), v.size))


def ot_min(v):
    v = _f32(v).ravel()
    return np.float32(lib().ot_min_f32(_ptr(v, ctypes.c_float), v.size))


# ---- standalone row reductions ("TIRx Metal reduction lowering" §8: row sums at
# widths 127/257/1024/4096, minimum and maximum together): the plain definitions.

def row_sum(x):
    """Sum of each row in FP64 (float64 result)."""
    return _f32(x).astype(np.float64).sum(axis=1)


def row_max(x):
    """Maximum of each row (exact in any order; float32 result)."""
    return _f32(x).max(axis=1)


def row_min(x):
    """Minimum of each row (exact in any order; float32 result)."""
    return _f32(x).min(axis=1)


def _skipnan_rows(x, name):
    x = _f32(x)
    out = np.empty(x.shape[0], np.float32)
    _rc(getattr(lib(), name)(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_float), x.shape[0], x.shape[1]))
    return out


def row_max_skipnan(x):
    """Unordered-policy row maximum (oracle.c Part 5): NaN elements are skipped,
    so a row gives NaN only when all of it is NaN; a zero maximum that occurs
    with both signs may come out with either sign."""
    return _skipnan_rows(x, "skipnan_row_max_f32")


def row_min_skipnan(x):
    """Unordered-policy row minimum (oracle.c Part 5), NaN elements skipped."""
    return _skipnan_rows(x, "skipnan_row_min_f32")


def ot_row_sum(x):
    """Ordered-policy (OT-1024) emulation of the row sums."""
    return np.array([ot_sum(r) for r in _f32(x)], dtype=np.float32)


def ot_row_max(x):
    return np.array([ot_max(r) for r in _f32(x)], dtype=np.float32)


def ot_row_min(x):
    return np.array([ot_min(r) for r in _f32(x)], dtype=np.float32)


# ---- reductions over any axis ("TIRx Metal reduction lowering", Reductions
# inside composed groups: the reduced axis need not be the last memory
# dimension): the same definitions applied to the vectors along `dim`.

def _columns(x, dim):
    """x with `dim` moved last, as a 2-D float32 array of vectors (and the result shape)."""
    a = np.moveaxis(_f32(x), dim, -1)
    return np.ascontiguousarray(a.reshape(-1, a.shape[-1])), a.shape[:-1]


def axis_sum(x, dim=0):
    """Sum over `dim` in FP64 (float64 result)."""
    return _f32(x).astype(np.float64).sum(axis=dim)


def axis_max(x, dim=0):
    return _f32(x).max(axis=dim)


def axis_min(x, dim=0):
    return _f32(x).min(axis=dim)


def _skipnan_axis(x, dim, name):
    x = _f32(x)
    dim = dim % x.ndim
    outer = int(np.prod(x.shape[:dim], dtype=np.int64))
    inner = int(np.prod(x.shape[dim + 1:], dtype=np.int64))
    out = np.empty(x.shape[:dim] + x.shape[dim + 1:], np.float32)
    _rc(getattr(lib(), name)(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_float), outer, x.shape[dim], inner))
    return out


def axis_max_skipnan(x, dim=0):
    """Unordered-policy maximum over `dim` (oracle.c Part 5), NaN elements skipped."""
    return _skipnan_axis(x, dim, "skipnan_axis_max_f32")


def axis_min_skipnan(x, dim=0):
    """Unordered-policy minimum over `dim` (oracle.c Part 5), NaN elements skipped."""
    return _skipnan_axis(x, dim, "skipnan_axis_min_f32")


def ot_axis_sum(x, dim=0):
    """Ordered-policy (OT-1024) sum of every vector along `dim`."""
    v, shape = _columns(x, dim)
    return ot_row_sum(v).reshape(shape)


def ot_axis_max(x, dim=0):
    v, shape = _columns(x, dim)
    return ot_row_max(v).reshape(shape)


def ot_axis_min(x, dim=0):
    v, shape = _columns(x, dim)
    return ot_row_min(v).reshape(shape)


# ---- backward passes (the gradients of the four operators; not on the pages,
# the next rows of the same row-reduction family). FP64 definitions return
# float64 arrays, the OT-1024 emulations float32.

def softmax_backward(y, dy):
    y, dy = _f32(y), _f32(dy)
    r, c = y.shape
    dx = np.empty((r, c), np.float64)
    _rc(lib().oracle_softmax_bwd_f64(_ptr(y, ctypes.c_float), _ptr(dy, ctypes.c_float), _ptr(dx, ctypes.c_double), r, c))
    return dx


def cross_entropy_backward(logits, labels, dloss=None):
    x = _f32(logits)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    dl = None if dloss is None else _f32(dloss)
    r, c = x.shape
    dx = np.empty((r, c), np.float64)
    _rc(lib().oracle_cross_entropy_bwd_f64(_ptr(x, ctypes.c_float), _ptr(lab, ctypes.c_int64),
                                           _ptr(dl, ctypes.c_float), _ptr(dx, ctypes.c_double), r, c))
    return dx


def rmsnorm_backward(x, w, dy, eps=1e-5):
    """(dx, dw) in FP64; dw is the column sum over rows of dy * x / rms."""
    x, dy = _f32(x), _f32(dy)
    w = None if w is None else _f32(w)
    r, c = x.shape
    dx = np.empty((r, c), np.float64)
    dw = np.empty(c, np.float64)
    _rc(lib().oracle_rmsnorm_bwd_f64(_ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float), _ptr(dy, ctypes.c_float),
                                     _ptr(dx, ctypes.c_double), _ptr(dw, ctypes.c_double), r, c, eps))
    return dx, dw


def layernorm_backward(x, gamma, dy, eps=1e-5):
    """(dx, dgamma, dbeta) in FP64."""
    x, dy = _f32(x), _f32(dy)
    gamma = None if gamma is None else _f32(gamma)
    r, c = x.shape
    dx = np.empty((r, c), np.float64)
    dg = np.empty(c, np.float64)
    db = np.empty(c, np.float64)
    _rc(lib().oracle_layernorm_bwd_f64(_ptr(x, ctypes.c_float), _ptr(gamma, ctypes.c_float),
                                       _ptr(dy, ctypes.c_float), _ptr(dx, ctypes.c_double),
                                       _ptr(dg, ctypes.c_double), _ptr(db, ctypes.c_double), r, c, eps))
    return dx, dg, db


def ot_softmax_backward(y, dy):
    y, dy = _f32(y), _f32(dy)
    r, c = y.shape
    dx = np.empty((r, c), np.float32)
    _rc(lib().ot_softmax_bwd_f32(_ptr(y, ctypes.c_float), _ptr(dy, ctypes.c_float), _ptr(dx, ctypes.c_float), r, c))
    return dx


def ot_cross_entropy_backward(logits, labels, dloss=None):
    x = _f32(logits)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    dl = None if dloss is None else _f32(dloss)
    r, c = x.shape
    dx = np.empty((r, c), np.float32)
    _rc(lib().ot_cross_entropy_bwd_f32(_ptr(x, ctypes.c_float), _ptr(lab, ctypes.c_int64), _ptr(dl, ctypes.c_float),
                                       _ptr(dx, ctypes.c_float), r, c))
    return dx


def ot_rmsnorm_backward(x, w, dy, eps=1e-5):
    x, dy = _f32(x), _f32(dy)
    w = None if w is None else _f32(w)
    r, c = x.shape
    dx = np.empty((r, c), np.float32)
    dw = np.empty(c, np.float32)
    _rc(lib().ot_rmsnorm_bwd_f32(_ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float), _ptr(dy, ctypes.c_float),
                                 _ptr(dx, ctypes.c_float), _ptr(dw, ctypes.c_float), r, c, eps))
    return dx, dw


def ot_layernorm_backward(x, gamma, dy, eps=1e-5):
    x, dy = _f32(x), _f32(dy)
    gamma = None if gamma is None else _f32(gamma)
    r, c = x.shape
    dx = np.empty((r, c), np.float32)
    dg = np.empty(c, np.float32)
    db = np.empty(c, np.float32)
    _rc(lib().ot_layernorm_bwd_f32(_ptr(x, ctypes.c_float), _ptr(gamma, ctypes.c_float), _ptr(dy, ctypes.c_float),
                                   _ptr(dx, ctypes.c_float), _ptr(dg, ctypes.c_float), _ptr(db, ctypes.c_float),
                                   r, c, eps))
    return dx, dg, db


# ---- the fold policies ("TIRx Metal reduction lowering" §1, ReductionPolicy
# fold_left / fold_right): every reduction a sequential fold over the columns,
# left to right with the accumulator on the left, or right to left with the
# accumulator on the right. `direction` is "left" or "right".

def _right(direction):
    if direction not in ("left", "right"):
        raise ValueError("direction must be 'left' or 'right'")
    return 1 if direction == "right" else 0


def fold_sum(v, direction="left"):
    v = _f32(v).ravel()
    return np.float32(lib().fold_sum_f32(_ptr(v, ctypes.c_float), v.size, _right(direction)))


def fold_max(v, direction="left"):
    v = _f32(v).ravel()
    return np.float32(lib().fold_max_f32(_ptr(v, ctypes.c_float), v.size, _right(direction)))


def fold_min(v, direction="left"):
    v = _f32(v).ravel()
    return np.float32(lib().fold_min_f32(_ptr(v, ctypes.c_float), v.size, _right(direction)))


def fold_row_sum(x, direction="left"):
    return np.array([fold_sum(r, direction) for r in _f32(x)], dtype=np.float32)


def fold_row_max(x, direction="left"):
    return np.array([fold_max(r, direction) for r in _f32(x)], dtype=np.float32)


def fold_row_min(x, direction="left"):
    return np.array([fold_min(r, direction) for r in _f32(x)], dtype=np.float32)


def fold_softmax(x, direction="left"):
    x = _f32(x)
    r, c = x.shape
    y = np.empty((r, c), np.float32)
    _rc(lib().fold_softmax_f32(_ptr(x, ctypes.c_float), _ptr(y, ctypes.c_float), r, c, _right(direction)))
    return y


def fold_rmsnorm(x, w=None, eps=1e-5, direction="left"):
    x = _f32(x)
    w = None if w is None else _f32(w)
    r, c = x.shape
    y = np.empty((r, c), np.float32)
    _rc(lib().fold_rmsnorm_f32(_ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float), _ptr(y, ctypes.c_float), r, c, eps,
                               _right(direction)))
    return y


def fold_layernorm(x, gamma=None, beta=None, eps=1e-5, direction="left"):
    x = _f32(x)
    gamma = None if gamma is None else _f32(gamma)
    beta = None if beta is None else _f32(beta)
    r, c = x.shape
    y = np.empty((r, c), np.float32)
    _rc(lib().fold_layernorm_f32(_ptr(x, ctypes.c_float), _ptr(gamma, ctypes.c_float), _ptr(beta, ctypes.c_float),
                                 _ptr(y, ctypes.c_float), r, c, eps, _right(direction)))
    return y


def fold_cross_entropy(logits, labels, direction="left"):
    x = _f32(logits)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    r, c = x.shape
    loss = np.empty(r, np.float32)
    _rc(lib().fold_cross_entropy_f32(_ptr(x, ctypes.c_float), _ptr(lab, ctypes.c_int64), _ptr(loss, ctypes.c_float),
                                     r, c, _right(direction)))
    return loss


def ot_expf(x):
    return np.float32(lib().ot_expf(float(x)))


def ot_logf(x):
    return np.float32(lib().ot_logf(float(x)))


def ot_expf_array(x):
    x = _f32(x).ravel()
    y = np.empty_like(x)
    lib().ot_expf_n(_ptr(x, ctypes.c_float), _ptr(y, ctypes.c_float), x.size)
    return y


def ot_logf_array(x):
    x = _f32(x).ravel()
    y = np.empty_like(x)
    lib().ot_logf_n(_ptr(x, ctypes.c_float), _ptr(y, ctypes.c_float), x.size)
    return y
