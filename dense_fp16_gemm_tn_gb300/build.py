"""Builds the C-ABI shared library ``libgemm_tn_f16.so`` in-tree.

Every ``csrc/*.cu`` translation unit is compiled by nvcc for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, and linked into
one shared library next to this file.  The CUDA runtime is linked statically
and the driver's tensor-map encoder is looked up at run time, so the library
loads on a machine without a GPU driver (the boundary tests use that).

Usage: ``python -m dense_fp16_gemm_tn_gb300.build`` (or ``build()``).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build", "gemm_tn_f16")
LIB_PATH = os.path.join(PKG, "libgemm_tn_f16.so")
# The checked build: the same sources with device-side bounds checks (-DGTN_CHECKED).
BUILD_DIR_CHECKED = os.path.join(ROOT, "_build", "gemm_tn_f16_checked")
LIB_PATH_CHECKED = os.path.join(PKG, "libgemm_tn_f16_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + \
        [os.path.join(INCLUDE, "gemm_tn_f16.h"), os.path.abspath(__file__)]


def up_to_date(checked: bool = False) -> bool:
    lib = LIB_PATH_CHECKED if checked else LIB_PATH
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link the library (or, with checked=True, its checked build); returns
    its path.  Raises on failure."""
    lib_path = LIB_PATH_CHECKED if checked else LIB_PATH
    build_dir = BUILD_DIR_CHECKED if checked else BUILD_DIR
    if not force and up_to_date(checked):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    extra = ["-DGTN_CHECKED"] if checked else []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for obj, log in results:
            sys.stderr.write(f"== {os.path.basename(obj)}\n{log}")
    objs = [o for o, _ in results]
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
