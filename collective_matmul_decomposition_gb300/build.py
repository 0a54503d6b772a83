"""Build the CUDA library in-tree: _build/libcm.so for sm_103a (nvcc, no cmake)."""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libcm.so")
# the same library with every computed index bounds-checked in the kernels
# (CM_DEBUG_BOUNDS): an index outside its buffer is reported as CM_ERR_BOUNDS
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libcm_debug.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["cm_kernel.cu", "cm_kernel_pair.cu", "cm_api.cu", "cm_plan.cpp", "cm_noalloc.cu", "cm_cost.cpp", "cm_reduce.cu"]
HEADERS = ["cm_internal.h", "cm_kernel.cuh", "cm_device.cuh", "cm_kernel_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-diag-suppress", "1160", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cuda, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile every translation unit in parallel, then link the shared library
    (debug=True: the bounds-checked build, in its own folder)."""
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "cm.h")]
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DCM_DEBUG_BOUNDS=1"] if debug else [])
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            extra = ["-x", "cu"] if src.endswith(".cu") else []
            jobs.append([nvcc] + ARCH + flags + extra + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stdout.write(r.stdout + r.stderr)

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
