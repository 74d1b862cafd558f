"""Build ``libcausal_product.so`` in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library under ``prefix_sum_outer_gb300/_build/``.  No CMake, no torch
extension machinery: the library exports the plain C ABI of
``include/causal_product.h`` and links only the CUDA runtime.

    python -m prefix_sum_outer_gb300.build [--force]
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libcausal_product.so")
SOURCES = ["cp_api.cu", "cp_simt.cu", "cp_tc.cu", "cp_tc_dkdv.cu", "cp_decode.cu",
           "cp_selftest.cu", "cp_norm.cu", "cp_feature.cu", "cp_segscan.cu", "cp_favor.cu", "cp_favor_fwd.cu",
           "cp_tc_lookback.cu", "cp_norm_pp.cu"]
HEADERS = ["cp_internal.h", "cp_tc_common.cuh", "cp_tc_causal.cuh", "cp_tc_dkdv.cuh",
           "sm103_ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _flags():
    # hidden visibility (and no GNU-unique objects) keeps every internal symbol,
    # including function-local statics, private to this copy of the library
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden", "-Xcompiler", "-fno-gnu-unique",
                   "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "causal_product.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if any source changed; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc] + _flags() + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
