"""Build the in-tree shared library librk_seg_attn.so for sm_103a with nvcc.

Each translation unit is compiled in parallel into `_build/`, then linked
into `position_independent_kv_gb300/_lib/librk_seg_attn.so` against the
shared CUDA runtime.  No CMake, one -gencode.
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
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "librk_seg_attn.so")

SOURCES = ["plan.cpp", "dense_mma.cu", "split_decode.cu", "dense_tc.cu", "dense_tc2.cu",
           "dense_tc4.cu", "dense_side.cu", "dense_tcs.cu", "noalloc.cu", "protected.cu",
           "project.cu", "seg_paged.cu"]
# test-only library: single-CTA checks of the tensor-path building blocks
SELFTEST_SOURCES = ["tc_selftest.cu"]
SELFTEST_LIB = os.path.join(LIBDIR, "librk_tc_selftest.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3",
                   "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + _flags() + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False, extra: list[str] | None = None, force: bool = False) -> str:
    lib = _build_lib(SOURCES, LIB, verbose, extra, force)
    _build_lib(SELFTEST_SOURCES, SELFTEST_LIB, verbose, extra, force)
    return lib


def _build_lib(sources, target, verbose, extra, force) -> str:
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = [s for s in sources if os.path.exists(os.path.join(CSRC, s))]
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [os.path.abspath(__file__)]
    if not force and os.path.exists(target):
        newest = max(os.path.getmtime(d) for d in deps)
        if os.path.getmtime(target) >= newest:
            return target
    extra = list(extra or [])
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), srcs))
    tmp = target + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, target)
    if verbose:
        print("built", target)
    return target


if __name__ == "__main__":
    build(verbose=True, extra=sys.argv[1:], force=True)
