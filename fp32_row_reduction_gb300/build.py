"""Build libtr.so in-tree: nvcc for sm_103a, one object per source, in parallel.

Usage: ``python -m fp32_row_reduction_gb300.build`` (or ``build()`` from Python).
The library links the CUDA runtime statically, so it loads on machines without
a GPU (the symbol checks run there); kernels need a GB300 (sm_103a).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtr.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}",
          "--expt-relaxed-constexpr"]
# The ordered kernels must round every step: no FMA contraction, IEEE division
# and square root, no flush to zero (nvcc's defaults for the last three).
_EXACT = ["-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false"]
EXTRA = {"k_ordered.cu": _EXACT, "k_wave_ordered.cu": _EXACT}
SOURCES = ["tr_api.cu", "tr_plan.cpp", "k_softmax.cu", "k_rmsnorm.cu", "k_layernorm.cu", "k_xent.cu",
           "k_ordered.cu", "tr_noalloc.cu", "k_add_rmsnorm.cu", "k_add_layernorm.cu",
           "k_reduce.cu", "k_axis.cu", "k_backward.cu", "k_fold.cu", "k_ot_cluster.cu", "k_xent_bwd.cu",
           "k_wave.cu", "k_wave_ordered.cu", "k_segments.cu", "k_bwd_wave.cu"]
HEADERS = ["tr_device.cuh", "tr_row_kernels.cuh", "tr_split_kernels.cuh", "tr_dispatch.cuh", "tr_internal.h",
           "tr_plan.h", "tr_ot.cuh", "tr_wave_kernels.cuh", "tr_segments_kernels.cuh"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtr.so")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "tr.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def _compile(nvcc: str, src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, *COMMON, *EXTRA.get(src, [])]
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas:
        sys.stderr.write(res.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    """Compile and link libtr.so next to this file; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    jobs = jobs or min(len(SOURCES), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, verbose_ptxas), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
