"""The C ABI used from plain C: tests/c_abi_consumer.c is compiled with gcc
(C11, -Wall -Werror) against include/ropekv.h, linked with libropekv.so and
the CUDA runtime, and run. On the CPU it makes the host-only calls; on the GPU
it runs a packed call on seeded inputs, whose outputs must match the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_consumer.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("CUDA runtime headers not found")
    from rope_kv_cache_gb300 import build
    lib = build.build_library()
    libdir = os.path.dirname(lib)
    out = str(tmp_path_factory.mktemp("c_consumer") / "consumer")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O2",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"), SRC,
           "-L", libdir, "-lropekv", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_host_calls_from_c(consumer):
    r = subprocess.run([consumer, "host"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert lines[0] == "capacity(4096, 4096) = 0"
    assert lines[1] == "capacity(4097, 4096) = -8"        # ROPEKV_ERR_CAPACITY
    assert lines[2] == "status 0: ok"
    assert len(lines) == 14 and all(line.startswith("status -") for line in lines[3:13])
    assert lines[13] == "residency cap: default 1, after switching off 0"


@pytest.mark.gpu
@pytest.mark.parametrize("style", [workloads.NEOX, workloads.GPTJ])
def test_packed_call_from_c(consumer, tmp_path, style):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import oracle
    from parity import compare, qkv_rotated, cache_rotated
    B, S, Hq, Hkv, D, r, cap = 3, 37, 8, 2, 128, 64, 64
    case = workloads.make_packed(B, S, Hq, Hkv, D, r, cap, style, 1e4, seed=55, cache_init="zero")
    cs, qkv = tmp_path / "cs.bin", tmp_path / "qkv.bin"
    oq, oc = tmp_path / "out_qkv.bin", tmp_path / "out_cache.bin"
    np.ascontiguousarray(case.cos_sin, dtype=np.float32).tofile(cs)
    np.ascontiguousarray(case.qkv, dtype=np.uint16).tofile(qkv)
    args = [consumer, "packed"] + [str(x) for x in (B, S, Hq, Hkv, D, r, cap, style)] + \
        [str(cs), str(qkv), str(oq), str(oc)]
    res = subprocess.run(args, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr
    got_qkv = np.fromfile(oq, dtype=np.uint16).reshape(case.qkv.shape)
    got_cache = np.fromfile(oc, dtype=np.uint16).reshape(case.new_cache().shape)
    want_qkv = case.qkv.copy()
    want_cache = case.new_cache()
    oracle.packed(case.cos_sin, want_qkv, want_cache, Hq, Hkv, style)
    compare(got_qkv, want_qkv, qkv_rotated(Hq, Hkv, D, r), "C consumer qkv")
    compare(got_cache, want_cache, cache_rotated(want_cache.shape, r), "C consumer cache")
