"""Builds libsdpa_bwd.so in-tree from csrc/*.cu for sm_103a with nvcc, and its
debug-bounds twin libsdpa_bwd_debug.so (compiled with SDPA_DEBUG_BOUNDS: the
kernels check their raw-pointer global accesses and report a violation in the
status word instead of making it).

Each translation unit compiles in parallel to an object file under _build/
(_build_debug/ for the twin), then nvcc links them into a shared library (CUDA
runtime linked statically, no libcuda link: the driver API is reached through
the runtime's entry-point query, so the library loads on hosts without a GPU
driver).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsdpa_bwd.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libsdpa_bwd_debug.so")
DEBUG_FLAGS = ["-DSDPA_DEBUG_BOUNDS"]
SOURCES = ["sdpa_bwd_api.cu", "sdpa_bwd_main.cu", "sdpa_bwd_main_bias.cu", "sdpa_bwd_main_qat.cu",
           "sdpa_bwd_main_f16.cu",
           "sdpa_bwd_main_ds.cu",
           "sdpa_bwd_aux.cu",
           "sdpa_bwd_dq.cu", "sdpa_bwd_noalloc.cu", "sdpa_fwd.cu", "sdpa_fwd_shared.cu", "sdpa_fwd_wide.cu"]
HEADERS = ["common.cuh", "gqa.cuh", "ptx.cuh", "tmap.h", "sdpa_bwd_main.cuh", "nvfp4.cuh", "bias.cuh", "sdpa_fwd.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsdpa_bwd.so")
    return exe


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, h) for h in HEADERS]
            + [os.path.join(ROOT, "include", "sdpa_bwd.h")])


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile(src: str, extra, build_dir=BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def _link(objs, lib) -> str:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """libsdpa_bwd.so, or with debug=True the debug-bounds twin."""
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = list(extra_flags) + (DEBUG_FLAGS if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, build_dir), srcs))
    _link(objs, lib)
    if verbose:
        print(f"built {lib}", file=sys.stderr)
    return lib


def build_all(verbose: bool = False) -> None:
    """Both libraries, their translation units compiled side by side."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        list(ex.map(lambda d: build(verbose=verbose, debug=d), (False, True)))


if __name__ == "__main__":
    build(verbose=True, extra_flags=sys.argv[1:])
