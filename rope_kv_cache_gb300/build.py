"""Build libropekv.so (the C ABI and its sm_103a kernels) in-tree with nvcc.

The library is one translation unit compiled for sm_103a only and linked
against the static CUDA runtime, so it loads without any other file from this
package. Output: ``rope_kv_cache_gb300/lib/libropekv.so`` (git-ignored).
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
SOURCES = [os.path.join(CSRC, "ropekv_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ropekv_kernels.cuh"), os.path.join(INCLUDE, "ropekv.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libropekv.so")


def nvcc_command(out: str, extra=()) -> list:
    return [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
            "-Xcompiler", "-fPIC,-fvisibility=hidden", "-cudart", "static",
            "-I", INCLUDE, "-I", CSRC, *extra, "-o", out, *SOURCES]


def build_library(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(LIB_DIR, exist_ok=True)
    stale = not os.path.exists(LIB_PATH) or \
        os.path.getmtime(LIB_PATH) < max(os.path.getmtime(p) for p in DEPS)
    if force or stale:
        tmp = LIB_PATH + f".{os.getpid()}.tmp"
        extra = ("-Xptxas", "-v") if verbose else ()
        subprocess.run(nvcc_command(tmp, extra), check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
