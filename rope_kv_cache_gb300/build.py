"""Build libropekv.so (the C ABI and its sm_103a kernels) in-tree with nvcc,
and libropekv_floor.so, the copy kernel the benchmark times as the floor of
a decode-sized launch.

Each library is one translation unit compiled for sm_103a only and linked
against the static CUDA runtime, so it loads without any other file from this
package; the two compile in parallel. Output: ``rope_kv_cache_gb300/lib/``
(git-ignored).
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libropekv.so")
FLOOR_LIB_PATH = os.path.join(LIB_DIR, "libropekv_floor.so")
SOURCES = [os.path.join(CSRC, "ropekv_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ropekv_kernels.cuh"), os.path.join(INCLUDE, "ropekv.h")]
FLOOR_SOURCES = [os.path.join(CSRC, "ropekv_floor.cu")]
FLOOR_DEPS = FLOOR_SOURCES + [os.path.join(INCLUDE, "ropekv_floor.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libropekv.so")


def nvcc_command(out: str, extra=(), sources=None) -> list:
    return [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
            "-Xcompiler", "-fPIC,-fvisibility=hidden", "-cudart", "static",
            "-I", INCLUDE, "-I", CSRC, *extra, "-o", out, *(sources or SOURCES)]


def _stale(lib: str, deps) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(p) for p in deps)


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Build both libraries where stale (or always with force); returns the
    path of libropekv.so."""
    os.makedirs(LIB_DIR, exist_ok=True)
    extra = ("-Xptxas", "-v") if verbose else ()
    jobs = []
    for lib, sources, deps in ((LIB_PATH, SOURCES, DEPS),
                               (FLOOR_LIB_PATH, FLOOR_SOURCES, FLOOR_DEPS)):
        if force or _stale(lib, deps):
            tmp = lib + f".{os.getpid()}.tmp"
            jobs.append((subprocess.Popen(nvcc_command(tmp, extra, sources)), tmp, lib))
    failed = []
    for proc, tmp, lib in jobs:
        if proc.wait() != 0:
            failed.append(os.path.basename(lib))
        else:
            os.replace(tmp, lib)
    if failed:
        raise RuntimeError(f"nvcc failed for {', '.join(failed)}")
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
