"""The C-ABI library loads, exports every declared symbol and validates its
arguments on the host (no GPU: only calls that must be rejected before any
CUDA call, or that have nothing to do, are made)."""
import ctypes
import os
import re

import pytest

import rope_kv_cache_gb300 as rk
from rope_kv_cache_gb300 import build
from rope_kv_cache_gb300._binding import ropekv_dims

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ropekv.h")

A = ctypes.c_void_p(0x10000)        # a 16-byte aligned fake device address
MIS = ctypes.c_void_p(0x10008)      # misaligned
NUL = ctypes.c_void_p(0)

OK = 0
ERR = {n: -i for i, n in enumerate(
    ["", "NULL", "MISALIGNED", "HEAD_DIM", "ROTARY_DIM", "HEADS", "SHAPE", "COS_SIN_BATCH",
     "CAPACITY", "STYLE", "LAUNCH"])}


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return rk.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"ROPEKV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    assert names == {"rope_write_kv_packed", "rope_write_kv_continuous", "rope_write_kv_tree",
                     "paged_kv_delta_update", "paged_kv_delta_update_fused",
                     "dflash_prepare_delta_metadata", "dflash_gather_delta_rope",
                     "rope_write_kv_slot_mapping", "rope_write_kv_continuous_qknorm",
                     "rope_write_kv_continuous_fp8",
                     "rope_check_capacity", "ropekv_set_residency_cap",
                     "ropekv_status_string"}


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def _dims(**kw):
    d = dict(batch=2, seqLen=4, numQHeads=8, numKVHeads=2, headDim=128, rotaryDim=128,
             kvCapacity=16, cosSinBatch=1, cosSinSeqLen=16, style=0)
    d.update(kw)
    return ropekv_dims(**d)


@pytest.mark.parametrize("kw,want", [
    (dict(headDim=96, rotaryDim=96), "HEAD_DIM"),
    (dict(headDim=32, rotaryDim=32), "HEAD_DIM"),
    (dict(rotaryDim=8), "ROTARY_DIM"),
    (dict(rotaryDim=72), "ROTARY_DIM"),
    (dict(rotaryDim=144), "ROTARY_DIM"),
    (dict(rotaryDim=0), "ROTARY_DIM"),
    (dict(numQHeads=6, numKVHeads=4), "HEADS"),
    (dict(numKVHeads=0), "HEADS"),
    (dict(batch=-1), "SHAPE"),
    (dict(seqLen=-3), "SHAPE"),
    (dict(cosSinBatch=3), "COS_SIN_BATCH"),
    (dict(style=2), "STYLE"),
])
def test_contiguous_rejects_bad_sizes(lib, kw, want):
    d = _dims(**kw)
    assert lib.rope_write_kv_continuous(A, A, A, A, A, ctypes.byref(d), NUL) == ERR[want]
    assert lib.rope_write_kv_tree(A, A, A, A, A, A, ctypes.byref(d), NUL) == ERR[want]
    assert lib.rope_write_kv_packed(A, A, A, ctypes.byref(d), NUL) == ERR[want]


def test_null_and_misaligned_pointers(lib):
    d = _dims()
    assert lib.rope_write_kv_continuous(A, NUL, A, A, A, ctypes.byref(d), NUL) == ERR["NULL"]
    assert lib.rope_write_kv_continuous(A, A, A, A, MIS, ctypes.byref(d), NUL) == ERR["MISALIGNED"]
    assert lib.rope_write_kv_tree(A, A, NUL, A, A, A, ctypes.byref(d), NUL) == ERR["NULL"]
    assert lib.rope_write_kv_tree(A, A, MIS, A, A, A, ctypes.byref(d), NUL) == ERR["MISALIGNED"]
    assert lib.rope_write_kv_packed(A, NUL, A, ctypes.byref(d), NUL) == ERR["NULL"]
    assert lib.rope_write_kv_packed(MIS, A, A, ctypes.byref(d), NUL) == ERR["MISALIGNED"]
    assert lib.rope_write_kv_packed(A, A, A, None, NUL) == ERR["NULL"]


def test_packed_capacity_checks(lib):
    assert lib.rope_write_kv_packed(A, A, A, ctypes.byref(_dims(seqLen=17)), NUL) == ERR["CAPACITY"]
    d = _dims(seqLen=8, cosSinSeqLen=7)
    assert lib.rope_write_kv_packed(A, A, A, ctypes.byref(d), NUL) == ERR["CAPACITY"]


def test_empty_calls_launch_nothing(lib):
    # zero tokens: OK without touching a pointer (NULLs allowed)
    for d in (_dims(batch=0), _dims(seqLen=0)):
        assert lib.rope_write_kv_continuous(NUL, NUL, NUL, NUL, NUL, ctypes.byref(d), NUL) == OK
        assert lib.rope_write_kv_tree(NUL, NUL, NUL, NUL, NUL, NUL, ctypes.byref(d), NUL) == OK
        assert lib.rope_write_kv_packed(NUL, NUL, NUL, ctypes.byref(d), NUL) == OK
    assert lib.paged_kv_delta_update(NUL, NUL, NUL, NUL, NUL, NUL, NUL, 0, 4, 8, 128, 128, 16,
                                     8, 64, 0, NUL) == OK


def _paged(lib, *, ptrs=None, N=16, B=4, Hkv=8, D=128, r=128, P=16, M=8, tpp=64, style=0):
    p = ptrs or [A] * 7
    return lib.paged_kv_delta_update(*p, N, B, Hkv, D, r, P, M, tpp, style, NUL)


def test_paged_rejects_bad_arguments(lib):
    assert _paged(lib, D=80, r=80) == ERR["HEAD_DIM"]
    assert _paged(lib, r=24) == ERR["ROTARY_DIM"]
    assert _paged(lib, Hkv=0) == ERR["HEADS"]
    assert _paged(lib, tpp=0) == ERR["SHAPE"]
    assert _paged(lib, N=-1) == ERR["SHAPE"]
    assert _paged(lib, P=-2) == ERR["SHAPE"]
    assert _paged(lib, style=5) == ERR["STYLE"]
    assert _paged(lib, ptrs=[A, A, NUL, A, A, A, A]) == ERR["NULL"]
    assert _paged(lib, ptrs=[A, A, A, MIS, A, A, A]) == ERR["MISALIGNED"]
    # batchSize 0: every row names a sequence >= batchSize, nothing to launch
    assert _paged(lib, B=0) == OK


def test_capacity_check(lib):
    assert lib.rope_check_capacity(4096, 4096) == OK
    assert lib.rope_check_capacity(100, 4096) == OK
    assert lib.rope_check_capacity(4097, 4096) == ERR["CAPACITY"]
    with pytest.raises(rk.RopeKVError):
        rk.rope_check_capacity(9000, 8192)
    rk.rope_check_capacity(8192, 8192)


def test_status_strings(lib):
    for code in range(0, -11, -1):
        s = rk.ropekv_status_string(code)
        assert s and s != "unknown status"
    assert rk.ropekv_status_string(-99) == "unknown status"


def _fused(lib, *, ptrs=None, W=16, B=4, Hkv=8, D=128, r=128, P=16, M=8, tpp=64, rows=1, cap=64,
           style=0):
    p = ptrs or [A] * 9
    return lib.paged_kv_delta_update_fused(p[0], p[1], p[2], p[3], p[4], p[5], W, p[6], p[7],
                                           B, Hkv, D, r, P, M, tpp, rows, cap, style, NUL)


def test_fused_rejects_bad_arguments(lib):
    assert _fused(lib, W=-1) == ERR["SHAPE"]
    assert _fused(lib, rows=-1) == ERR["SHAPE"]
    assert _fused(lib, cap=-1) == ERR["SHAPE"]
    assert _fused(lib, W=1 << 20, B=1 << 12) == ERR["SHAPE"]  # 2^32 rows
    assert _fused(lib, D=48, r=48) == ERR["HEAD_DIM"]
    assert _fused(lib, r=200) == ERR["ROTARY_DIM"]
    assert _fused(lib, style=3) == ERR["STYLE"]
    assert _fused(lib, ptrs=[A, A, A, A, NUL, A, A, A, A]) == ERR["NULL"]
    assert _fused(lib, ptrs=[A, A, A, A, A, A, MIS, A, A]) == ERR["MISALIGNED"]
    assert _fused(lib, W=0) == OK and _fused(lib, B=0) == OK


def test_metadata_and_gather_reject_bad_arguments(lib):
    assert lib.dflash_prepare_delta_metadata(A, A, -1, A, A, 4, NUL) == ERR["SHAPE"]
    assert lib.dflash_prepare_delta_metadata(A, A, 4, A, A, -4, NUL) == ERR["SHAPE"]
    assert lib.dflash_prepare_delta_metadata(A, A, 4, NUL, A, 4, NUL) == ERR["NULL"]
    assert lib.dflash_prepare_delta_metadata(A, A, 4, A, MIS, 4, NUL) == ERR["MISALIGNED"]
    assert lib.dflash_prepare_delta_metadata(NUL, NUL, 0, NUL, NUL, 4, NUL) == OK
    assert lib.dflash_gather_delta_rope(A, A, A, A, NUL, 8, 4, 1, 64, 72, NUL) == ERR["ROTARY_DIM"]
    assert lib.dflash_gather_delta_rope(A, A, A, A, NUL, 8, 4, 1, 64, 512, NUL) == ERR["ROTARY_DIM"]
    assert lib.dflash_gather_delta_rope(A, A, A, A, NUL, -8, 4, 1, 64, 64, NUL) == ERR["SHAPE"]
    assert lib.dflash_gather_delta_rope(A, NUL, A, A, NUL, 8, 4, 1, 64, 64, NUL) == ERR["NULL"]
    assert lib.dflash_gather_delta_rope(A, A, A, A, MIS, 8, 4, 1, 64, 64, NUL) == ERR["MISALIGNED"]
    assert lib.dflash_gather_delta_rope(NUL, NUL, NUL, NUL, NUL, 0, 4, 1, 64, 64, NUL) == OK


def _slotmap(lib, *, ptrs=None, qs=48 * 128, ks=48 * 128, vs=48 * 128, T=4, Hq=32, Hkv=8, D=128,
             r=128, rows=16, blocks=4, bsz=16, style=0):
    p = ptrs or [A] * 10
    return lib.rope_write_kv_slot_mapping(p[0], p[1], p[2], qs, p[3], ks, p[4], vs, p[5], p[6],
                                          p[7], p[8], p[9], T, Hq, Hkv, D, r, rows, blocks, bsz,
                                          style, NUL)


def test_slot_mapping_rejects_bad_arguments(lib):
    assert _slotmap(lib, qs=100) == ERR["SHAPE"]          # smaller than Hq*D
    assert _slotmap(lib, ks=8 * 128 + 4) == ERR["SHAPE"]   # not a multiple of 8
    assert _slotmap(lib, bsz=0) == ERR["SHAPE"]
    assert _slotmap(lib, blocks=-1) == ERR["SHAPE"]
    assert _slotmap(lib, Hq=12, Hkv=8) == ERR["HEADS"]
    assert _slotmap(lib, D=96, r=96) == ERR["HEAD_DIM"]
    assert _slotmap(lib, style=7) == ERR["STYLE"]
    assert _slotmap(lib, ptrs=[A, A, A, A, A, NUL, A, A, A, A]) == ERR["NULL"]
    assert _slotmap(lib, ptrs=[A, A, A, A, A, A, A, A, A, MIS]) == ERR["MISALIGNED"]
    assert _slotmap(lib, T=0, ptrs=[NUL] * 10) == OK


def test_qknorm_rejects_bad_arguments(lib):
    d = _dims()
    f = lib.rope_write_kv_continuous_qknorm
    assert f(A, A, A, A, A, A, A, -1.0, ctypes.byref(d), NUL) == ERR["SHAPE"]
    assert f(A, A, A, A, A, A, A, float("nan"), ctypes.byref(d), NUL) == ERR["SHAPE"]
    assert f(A, A, A, A, A, NUL, A, 1e-6, ctypes.byref(d), NUL) == ERR["NULL"]
    assert f(A, A, A, A, A, A, MIS, 1e-6, ctypes.byref(d), NUL) == ERR["MISALIGNED"]
    assert f(A, A, A, A, A, A, A, 1e-6, ctypes.byref(_dims(headDim=80, rotaryDim=80)),
             NUL) == ERR["HEAD_DIM"]
    assert f(NUL, NUL, NUL, NUL, NUL, NUL, NUL, 1e-6, ctypes.byref(_dims(batch=0)), NUL) == OK


def test_fp8_rejects_bad_arguments(lib):
    d = _dims()
    f = lib.rope_write_kv_continuous_fp8
    assert f(A, A, A, A, A, NUL, A, ctypes.byref(d), NUL) == ERR["NULL"]
    assert f(A, A, A, MIS, A, A, A, ctypes.byref(d), NUL) == ERR["MISALIGNED"]
    assert f(A, A, A, A, A, A, A, ctypes.byref(_dims(rotaryDim=40)), NUL) == ERR["ROTARY_DIM"]
    assert f(NUL, NUL, NUL, NUL, NUL, NUL, NUL, ctypes.byref(_dims(seqLen=0)), NUL) == OK


def test_slot_mapping_rejects_slot_counts_past_int64(lib):
    # numBlocks * blockSize must not overflow: 2^40 blocks of 2^31 - 1 slots
    assert _slotmap(lib, blocks=1 << 40, bsz=(1 << 31) - 1) == ERR["SHAPE"]


def test_residency_cap_switch(lib):
    # host-only: the switch is a process-wide flag; returns the previous value
    try:
        assert lib.ropekv_set_residency_cap(0) == 1          # on by default
        assert lib.ropekv_set_residency_cap(0) == 0
        assert rk.ropekv_set_residency_cap(True) is False
        assert rk.ropekv_set_residency_cap(True) is True
    finally:
        lib.ropekv_set_residency_cap(1)


def _no_cuda_device():
    try:
        import torch
        return torch.cuda.device_count() == 0
    except Exception:
        return True


@pytest.mark.skipif(not _no_cuda_device(),
                    reason="fake device addresses must never reach a real GPU")
def test_launch_failure_is_the_launchs_own_status(lib):
    """On a host without a CUDA device every call that passes the host checks
    reaches its launch, and the failure comes back from that launch as
    ROPEKV_ERR_LAUNCH (no launch path reads CUDA's last-error state). The
    fused update accepts a NULL cos/sin source when it has no source rows,
    as the gather does."""
    d = _dims()
    assert lib.rope_write_kv_continuous(A, A, A, A, A, ctypes.byref(d), NUL) == ERR["LAUNCH"]
    assert lib.rope_write_kv_packed(A, A, A, ctypes.byref(_dims(batch=1, seqLen=1)),
                                    NUL) == ERR["LAUNCH"]
    assert _paged(lib) == ERR["LAUNCH"]
    assert lib.dflash_prepare_delta_metadata(A, A, 4, A, A, 4, NUL) == ERR["LAUNCH"]
    assert lib.dflash_gather_delta_rope(NUL, A, A, A, NUL, 8, 4, 0, 64, 64, NUL) == ERR["LAUNCH"]
    assert _slotmap(lib) == ERR["LAUNCH"]
    assert _fused(lib, ptrs=[A, A, A, NUL, A, A, A, A, A], rows=0) == ERR["LAUNCH"]
    assert _fused(lib, ptrs=[A, A, A, NUL, A, A, A, A, A], rows=1) == ERR["NULL"]


def test_floor_library_exports_and_checks():
    """libropekv_floor.so (the benchmark's decode-floor copy) exports what
    include/ropekv_floor.h declares and rejects bad arguments on the host."""
    text = open(os.path.join(ROOT, "include", "ropekv_floor.h")).read()
    names = re.findall(r"ROPEKV_FLOOR_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    assert names == ["ropekv_floor_copy"]
    build.build_library()
    fl = rk._binding.load_floor_library()
    for n in names:
        assert hasattr(fl, n)
    f = fl.ropekv_floor_copy
    per = 16 * 4 * 192
    assert f(NUL, A, per, 192, 1, NUL) == -1
    assert f(MIS, A, per, 192, 1, NUL) == -2
    assert f(A, A, per, 100, 1, NUL) == -6          # not a multiple of 32
    assert f(A, A, per + 16, 192, 1, NUL) == -6     # not whole CTAs
    assert f(A, A, 0, 192, 1, NUL) == -6
