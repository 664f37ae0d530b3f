"""Compile the CUDA sources under ``csrc/`` into the in-tree shared library ``libmdw.so``.

sm_103a only (GB300): ``nvcc -gencode arch=compute_103a,code=sm_103a``. Each translation
unit is compiled in parallel, then linked with the CUDA runtime statically.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmdw.so")
TRACE_LIB = os.path.join(PKG, "libmdw_trace.so")     # profiling build (-DMDW_TRACE), never loaded by the API
SOURCES = ["moe.cu", "lm_head.cu", "abi.cu", "noalloc.cu", "sampler.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=default",
         "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmdw.so")
    return path


def _compile(src: str, trace: bool = False) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + (".trace.o" if trace else ".o"))
    cmd = [nvcc(), *ARCH, *FLAGS, *(["-DMDW_TRACE"] if trace else []), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False, trace: bool = False) -> str:
    """Build libmdw.so (always rebuilds); returns its path. trace=True builds the profiling
    library libmdw_trace.so instead: the same kernels with %globaltimer stamps at their phase
    boundaries (read by moe_decode_weight_gb300.phase_trace); the product library is untouched."""
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda src: _compile(src, trace), SOURCES))
    out = TRACE_LIB if trace else LIB
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(f"built {out}")
    return out


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
