"""Builds the in-tree shared library ``libmqa_attention_gb300.so`` for sm_103a.

Each CUDA translation unit is compiled by nvcc in parallel, then linked into
one shared library (CUDA runtime linked statically, so the library loads on a
machine without a GPU driver; the driver is reached at run time through the
runtime's entry-point query). Run as ``python -m mqa_attention_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libmqa_attention_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
# The debug build: every kernel checks its global indices and TMA coordinates before
# using them (GB_BOUNDS_CHECK) and reports a failed check in the device status word.
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libmqa_attention_gb300_debug.so")
SOURCES = ["api.cu", "rope.cu", "attn_fwd.cu", "attn_bwd.cu", "attn_decode.cu", "attn_delta.cu",
           "noalloc.cu"]
HEADERS = ["ptx.cuh", "kernels.h", "rope_math.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(PKG_DIR, "..", "include", "attn.h"))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    """Compiles (if out of date) and returns the path of the shared library; with
    debug=True the bounds-checking build instead."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _deps_mtime():
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug:
        extra.append("-DGB_BOUNDS_CHECK")

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
