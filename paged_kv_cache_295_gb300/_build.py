"""In-tree build of libpagedkv.so for sm_103a with nvcc (no cmake, no torch).

Each translation unit compiles in parallel into ``_build/``; the shared
library lands next to this file.  A rebuild happens when any source or header
is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", f"-I{INCLUDE}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")
    return exe


def sources():
    cu = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cpp = sorted(glob.glob(os.path.join(CSRC, "*.cpp")))
    deps = cu + cpp + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h")))
    return cu, cpp, deps


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in sources()[2] + [__file__])


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build_library(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile every CUDA / C++ unit for sm_103a and link ``libpagedkv.so``."""
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cu, cpp, _ = sources()
    nv = nvcc()
    jobs = []
    for src in cu:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        extra = ["-Xptxas", "-v"] if verbose_ptxas else []
        jobs.append([nv, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj])
    for src in cpp:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        jobs.append([os.environ.get("CXX", "g++"), *CXX_FLAGS, "-c", src, "-o", obj])
    logs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for out in ex.map(_run, jobs):
            logs.append(out)
    objs = [j[-1] for j in jobs]
    tmp = LIB + ".tmp"
    _run([nv, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    if verbose_ptxas:
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            f.write("\n".join(logs))
    return LIB


if __name__ == "__main__":
    import sys
    print(build_library(force=True, verbose_ptxas="-v" in sys.argv))
