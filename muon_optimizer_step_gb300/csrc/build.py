"""Build libmuon.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

    python -m muon_optimizer_step_gb300.csrc.build          # or build() from Python
    python -m muon_optimizer_step_gb300.csrc.build --debug  # libmuon_debug.so

Every translation unit compiles in parallel into ``_build/`` next to the package; the
shared library lands at ``muon_optimizer_step_gb300/libmuon.so``.  The debug build
(-DMUON_DEBUG: device-side range checks of every table entry the kernels use) compiles
into ``_build_debug/`` and lands at ``muon_optimizer_step_gb300/libmuon_debug.so``; the
binding loads it when MUON_LIB names it.  Host code is plain C++17 (no x86 intrinsics),
so the same sources build on x86_64 and aarch64 hosts.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
ROOT = os.path.dirname(PKG)
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libmuon.so")
BUILD_DIR_DEBUG = os.path.join(PKG, "_build_debug")
LIB_PATH_DEBUG = os.path.join(PKG, "libmuon_debug.so")

SOURCES = ["layout.cpp", "capi.cu", "stream_kernels.cu", "gemm_f32.cu", "gemm_ns.cu",
           "noalloc.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand) and shutil.which(cand) is None:
        raise RuntimeError("nvcc not found; set NVCC or put CUDA's bin directory on PATH")
    return cand


def _flags(debug=False):
    return ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O3",
            "-I" + os.path.join(ROOT, "include"), "-I" + HERE] + GENCODE + \
        (["-DMUON_DEBUG"] if debug else [])


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DIR_DEBUG if debug else BUILD_DIR, os.path.splitext(src)[0] + ".o")
    path = os.path.join(HERE, src)
    cmd = [_nvcc(), "-c", path, "-o", obj] + _flags(debug)
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(verbose: bool = False, jobs: int | None = None, debug: bool = False) -> str:
    """Compile every source and link libmuon.so (debug: libmuon_debug.so); returns the
    library path."""
    os.makedirs(BUILD_DIR_DEBUG if debug else BUILD_DIR, exist_ok=True)
    lib_path = LIB_PATH_DEBUG if debug else LIB_PATH
    jobs = jobs or min(len(SOURCES), os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [_nvcc(), "-shared", "-o", tmp] + objs + GENCODE + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
