"""Builds librkv.so in-tree with nvcc for sm_103a (B300).

`python -m rolling_kv_cache_buffer_b300.build` or build() from Python.  The
library links the CUDA runtime statically, so loading it needs no GPU; ptxas
register/spill reports go to lib/ptxas.log.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "librkv.so")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["rkv_api.cu", "rkv_misc.cu", "rkv_attend_fma.cu", "rkv_attend_mma.cu",
           "rkv_attend_chunk.cu", "rkv_attend_tc.cu", "rkv_attend_static.cu", "rkv_reset.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "rkv.h")]


def _compile(src):
    obj = os.path.join(LIBDIR, os.path.basename(src).replace(".cu", ".o"))
    cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in _deps())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    with open(os.path.join(LIBDIR, "ptxas.log"), "w") as f:
        for obj, log in results:
            f.write(f"== {os.path.basename(obj)}\n{log}\n")
    tmp = LIB + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", "--cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
