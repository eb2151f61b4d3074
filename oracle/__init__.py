"""CPU oracle for the fused RoPE + KV-cache write -- TEST INFRASTRUCTURE.

The oracle is a plain double-precision C implementation (``ropekv_oracle.c``)
of what the fused RoPE + KV-cache write computes, written from the pages:

* TensorRT-Edge-LLM 0.4.0 C++ API, "Apply Rope Write KV" (packed, continuous
  and tree entry points: layouts and in/out roles);
* sglang ``rope_cache.py`` (``_get_neox_rotated_x``, ``_get_gptj_rotated_x``,
  ``_unit_rope``, ``_load_cos_sin``, kernel Stage 2.1);
* TensorRT-Edge-LLM C++ API, "Dflash Runtime Kernels"
  (``launchDFlashTargetKVCacheUpdate``, ``checkDFlashRopeCapacity``).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it and the
two share no code. This module is argument marshalling around the C functions
(numpy arrays in, numpy arrays out); all arithmetic lives in the C file.

Parity status: every function is pinned by the ``-m "not gpu"`` tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ropekv_oracle.c")
_HDR = os.path.join(_HERE, "ropekv_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libropekv_oracle.so")

NEOX = 0
GPTJ = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler into ``oracle/_build``.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded in
    double, so x86_64 and aarch64 builds give the same bits.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (
        not os.path.exists(_LIB_PATH)
        or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    )
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = [
            os.environ.get("CC", "gcc"), "-O2", "-std=c11", "-fPIC", "-shared",
            "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
            "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # ROPEKV_ORACLE_LIB points the loader at another build of this same C file;
    # the mutation tests use it to check that the pins catch planted mistakes.
    path = os.environ.get("ROPEKV_ORACLE_LIB") or build()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.ropekv_oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.ropekv_oracle_f16_to_f64.restype = ctypes.c_double
    lib.ropekv_oracle_f64_to_f16.argtypes = [ctypes.c_double]
    lib.ropekv_oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.ropekv_oracle_rotate_half.argtypes = [P, I, I, P]
    lib.ropekv_oracle_rotate_half.restype = None
    lib.ropekv_oracle_freq_index.argtypes = [I, I, I]
    lib.ropekv_oracle_freq_index.restype = I
    lib.ropekv_oracle_rope_head_f64.argtypes = [P, P, I, I, I, P]
    lib.ropekv_oracle_rope_head_f64.restype = None
    lib.ropekv_oracle_packed.argtypes = [P, P, P] + [I] * 10
    lib.ropekv_oracle_packed.restype = I
    lib.ropekv_oracle_continuous.argtypes = [P, P, P, P, P] + [I] * 10
    lib.ropekv_oracle_continuous.restype = I
    lib.ropekv_oracle_tree.argtypes = [P, P, P, P, P, P] + [I] * 10
    lib.ropekv_oracle_tree.restype = I
    lib.ropekv_oracle_paged_rows.argtypes = [P] * 6 + [I] * 9 + [P] * 4
    lib.ropekv_oracle_paged_rows.restype = I
    lib.ropekv_oracle_paged.argtypes = [P] * 7 + [I] * 9
    lib.ropekv_oracle_paged.restype = I
    lib.ropekv_oracle_delta_metadata.argtypes = [P, P, I, P, P, I]
    lib.ropekv_oracle_delta_metadata.restype = I
    lib.ropekv_oracle_gather_delta_rope.argtypes = [P, P, P, P, P, I, I, I, I, I]
    lib.ropekv_oracle_gather_delta_rope.restype = I
    lib.ropekv_oracle_paged_fused.argtypes = [P] * 9 + [I] * 10
    lib.ropekv_oracle_paged_fused.restype = I
    lib.ropekv_oracle_continuous_qknorm.argtypes = [P] * 7 + [ctypes.c_float] + [I] * 10
    lib.ropekv_oracle_continuous_qknorm.restype = I
    lib.ropekv_oracle_rms_norm_f64.argtypes = [P, P, ctypes.c_double, I, P]
    lib.ropekv_oracle_rms_norm_f64.restype = None
    lib.ropekv_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.ropekv_oracle_e4m3_to_f64.restype = ctypes.c_double
    lib.ropekv_oracle_f64_to_e4m3.argtypes = [ctypes.c_double]
    lib.ropekv_oracle_f64_to_e4m3.restype = ctypes.c_uint8
    lib.ropekv_oracle_continuous_fp8.argtypes = [P] * 5 + [ctypes.c_float] * 2 + [I] * 10
    lib.ropekv_oracle_continuous_fp8.restype = I
    L = ctypes.c_int64
    lib.ropekv_oracle_slot_mapping.argtypes = [P, P, P, L, P, L, P, L, P, P, P, P, P,
                                               I, I, I, I, I, I, L, I, I]
    lib.ropekv_oracle_slot_mapping.restype = I
    lib.ropekv_oracle_capacity_rejected.argtypes = [ctypes.c_int32, ctypes.c_int32]
    lib.ropekv_oracle_capacity_rejected.restype = I
    _lib = lib
    return lib


def _ptr(a: np.ndarray, dtype) -> ctypes.c_void_p:
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("array must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: inconsistent sizes (rc={rc})")


# ----------------------------------------------------------------- scalars --

def f16_to_f64(bits: int) -> float:
    return _load().ropekv_oracle_f16_to_f64(int(bits) & 0xFFFF)


def f64_to_f16(x: float) -> int:
    return int(_load().ropekv_oracle_f64_to_f16(float(x)))


def f16_to_f64_array(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.ropekv_oracle_f16_to_f64(int(b)) for b in flat],
                    dtype=np.float64).reshape(bits.shape)


def f64_to_f16_array(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float64).ravel()
    return np.array([lib.ropekv_oracle_f64_to_f16(float(v)) for v in flat],
                    dtype=np.uint16).reshape(np.shape(x))


def freq_index(d: int, r: int, style: int) -> int:
    return int(_load().ropekv_oracle_freq_index(d, r, style))


def rotate_half(x: np.ndarray, r: int, style: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(r, dtype=np.float64)
    _load().ropekv_oracle_rotate_half(_ptr(x, np.float64), r, style, _ptr(out, np.float64))
    return out


def rope_head_f64(x: np.ndarray, cs_row: np.ndarray, r: int, style: int) -> np.ndarray:
    """One head in double before rounding: x (D,) float64, cs_row (r,) float32."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    cs_row = np.ascontiguousarray(cs_row, dtype=np.float32)
    if cs_row.shape[-1] != r:
        raise ValueError("cos/sin row must hold rotaryDim floats")
    y = np.zeros_like(x)
    _load().ropekv_oracle_rope_head_f64(_ptr(x, np.float64), _ptr(cs_row, np.float32),
                                        x.shape[0], r, style, _ptr(y, np.float64))
    return y


# ------------------------------------------------------------ entry points --

def packed(cos_sin, qkv, kv_cache, Hq, Hkv, style):
    """Packed in-place path. Mutates ``qkv`` and ``kv_cache`` (numpy uint16)."""
    csB, csS, r = cos_sin.shape
    B, S, H, D = qkv.shape
    cap = kv_cache.shape[3]
    assert H == Hq + 2 * Hkv and kv_cache.shape == (B, 2, Hkv, cap, D)
    rc = _load().ropekv_oracle_packed(_ptr(cos_sin, np.float32), _ptr(qkv, np.uint16),
                                      _ptr(kv_cache, np.uint16),
                                      B, S, Hq, Hkv, D, r, cap, csB, csS, style)
    _check(rc, "packed")


def continuous(cos_sin, end_lens, qkv, kv_cache, q_out, Hq, Hkv, style):
    """Continuous path. Mutates ``kv_cache`` and ``q_out``."""
    csB, csS, r = cos_sin.shape
    B, S, H, D = qkv.shape
    cap = kv_cache.shape[3]
    assert H == Hq + 2 * Hkv and kv_cache.shape == (B, 2, Hkv, cap, D)
    assert q_out.shape == (B, S, Hq, D) and end_lens.shape == (B,)
    rc = _load().ropekv_oracle_continuous(_ptr(cos_sin, np.float32), _ptr(end_lens, np.int32),
                                          _ptr(qkv, np.uint16), _ptr(kv_cache, np.uint16),
                                          _ptr(q_out, np.uint16),
                                          B, S, Hq, Hkv, D, r, cap, csB, csS, style)
    _check(rc, "continuous")


def continuous_qknorm(cos_sin, end_lens, qkv, kv_cache, q_out, q_weight, k_weight, eps, Hq, Hkv,
                      style):
    """Continuous path with pre-RoPE RMS normalization of Q and K heads
    (weights: [D] uint16 FP16 bits). Mutates ``kv_cache`` and ``q_out``."""
    csB, csS, r = cos_sin.shape
    B, S, H, D = qkv.shape
    cap = kv_cache.shape[3]
    assert H == Hq + 2 * Hkv and kv_cache.shape == (B, 2, Hkv, cap, D)
    assert q_weight.shape == (D,) and k_weight.shape == (D,)
    rc = _load().ropekv_oracle_continuous_qknorm(
        _ptr(cos_sin, np.float32), _ptr(end_lens, np.int32), _ptr(qkv, np.uint16),
        _ptr(kv_cache, np.uint16), _ptr(q_out, np.uint16), _ptr(q_weight, np.uint16),
        _ptr(k_weight, np.uint16), float(eps), B, S, Hq, Hkv, D, r, cap, csB, csS, style)
    _check(rc, "continuous_qknorm")


def e4m3_to_f64(bits: int) -> float:
    return _load().ropekv_oracle_e4m3_to_f64(int(bits) & 0xFF)


def f64_to_e4m3(x: float) -> int:
    return int(_load().ropekv_oracle_f64_to_e4m3(float(x)))


def continuous_fp8(cos_sin, end_lens, qkv, kv_cache8, q_out, k_scale, v_scale, Hq, Hkv, style):
    """Continuous call with an E4M3 cache (uint8 [B, 2, Hkv, cap, D]). Mutates
    ``kv_cache8`` and ``q_out``."""
    csB, csS, r = cos_sin.shape
    B, S, H, D = qkv.shape
    cap = kv_cache8.shape[3]
    assert H == Hq + 2 * Hkv and kv_cache8.shape == (B, 2, Hkv, cap, D)
    rc = _load().ropekv_oracle_continuous_fp8(
        _ptr(cos_sin, np.float32), _ptr(end_lens, np.int32), _ptr(qkv, np.uint16),
        _ptr(kv_cache8, np.uint8), _ptr(q_out, np.uint16), float(k_scale), float(v_scale),
        B, S, Hq, Hkv, D, r, cap, csB, csS, style)
    _check(rc, "continuous_fp8")


def rms_norm_f64(x, weight, eps):
    x = np.ascontiguousarray(x, dtype=np.float64)
    weight = np.ascontiguousarray(weight, dtype=np.uint16)
    y = np.zeros_like(x)
    _load().ropekv_oracle_rms_norm_f64(_ptr(x, np.float64), _ptr(weight, np.uint16), float(eps),
                                       x.shape[0], _ptr(y, np.float64))
    return y


def tree(cos_sin, end_lens, pos_ids, qkv, kv_cache, q_out, Hq, Hkv, style):
    """Tree path. Mutates ``kv_cache`` and ``q_out``."""
    csB, csS, r = cos_sin.shape
    B, S, H, D = qkv.shape
    cap = kv_cache.shape[3]
    assert H == Hq + 2 * Hkv and kv_cache.shape == (B, 2, Hkv, cap, D)
    assert q_out.shape == (B, S, Hq, D) and end_lens.shape == (B,) and pos_ids.shape == (B, S)
    rc = _load().ropekv_oracle_tree(_ptr(cos_sin, np.float32), _ptr(end_lens, np.int32),
                                    _ptr(pos_ids, np.int32), _ptr(qkv, np.uint16),
                                    _ptr(kv_cache, np.uint16), _ptr(q_out, np.uint16),
                                    B, S, Hq, Hkv, D, r, cap, csB, csS, style)
    _check(rc, "tree")


def paged_rows(k_delta, v_delta, cos_sin_rows, delta_positions, delta_to_seq, page_table,
               num_pages, tokens_per_page, style):
    """Per-row destinations and values of the paged delta update.

    Returns (k_dest, v_dest, k_out, v_out): int64 element offsets into a pool
    [2, num_pages, tokens_per_page, Hkv, D] (-1 = plane skipped) and the
    [N, Hkv, D] uint16 values stored there.
    """
    N, Hkv, D = k_delta.shape
    r = cos_sin_rows.shape[1]
    B, two, mpps = page_table.shape
    assert two == 2 and v_delta.shape == k_delta.shape and cos_sin_rows.shape[0] == N
    k_dest = np.empty(N, dtype=np.int64)
    v_dest = np.empty(N, dtype=np.int64)
    k_out = np.zeros_like(k_delta)
    v_out = np.zeros_like(v_delta)
    rc = _load().ropekv_oracle_paged_rows(
        _ptr(k_delta, np.uint16), _ptr(v_delta, np.uint16), _ptr(cos_sin_rows, np.float32),
        _ptr(delta_positions, np.int32), _ptr(delta_to_seq, np.int32),
        _ptr(page_table, np.int32), N, B, Hkv, D, r, num_pages, mpps, tokens_per_page, style,
        _ptr(k_dest, np.int64), _ptr(v_dest, np.int64), _ptr(k_out, np.uint16),
        _ptr(v_out, np.uint16))
    _check(rc, "paged_rows")
    return k_dest, v_dest, k_out, v_out


def paged(k_delta, v_delta, kv_pool, cos_sin_rows, delta_positions, delta_to_seq, page_table,
          style):
    """Paged delta update into a host pool [2, numPages, TPP, Hkv, D] (mutated)."""
    N, Hkv, D = k_delta.shape
    r = cos_sin_rows.shape[1]
    B, two, mpps = page_table.shape
    _, num_pages, tpp, hk2, d2 = kv_pool.shape
    assert two == 2 and hk2 == Hkv and d2 == D
    rc = _load().ropekv_oracle_paged(
        _ptr(k_delta, np.uint16), _ptr(v_delta, np.uint16), _ptr(kv_pool, np.uint16),
        _ptr(cos_sin_rows, np.float32), _ptr(delta_positions, np.int32),
        _ptr(delta_to_seq, np.int32), _ptr(page_table, np.int32),
        N, B, Hkv, D, r, num_pages, mpps, tpp, style)
    _check(rc, "paged")


def delta_metadata(old_lengths, delta_lengths, delta_width):
    """Returns (delta_positions, delta_token_to_sequence), each [B * delta_width] int32."""
    old_lengths = np.ascontiguousarray(old_lengths, dtype=np.int32)
    delta_lengths = np.ascontiguousarray(delta_lengths, dtype=np.int32)
    B = old_lengths.shape[0]
    pos = np.empty(B * delta_width, dtype=np.int32)
    seq = np.empty(B * delta_width, dtype=np.int32)
    rc = _load().ropekv_oracle_delta_metadata(_ptr(old_lengths, np.int32), _ptr(delta_lengths, np.int32),
                                              delta_width, _ptr(pos, np.int32), _ptr(seq, np.int32), B)
    _check(rc, "delta_metadata")
    return pos, seq


def gather_delta_rope(source, delta_positions, delta_to_seq, state_indices, batch_size):
    """source [sourceRows, cacheCapacity, r] float32 -> [N, r] float32."""
    source = np.ascontiguousarray(source, dtype=np.float32)
    rows, cap, r = source.shape
    N = delta_positions.shape[0]
    out = np.full((N, r), np.nan, dtype=np.float32)
    st = ctypes.c_void_p(0) if state_indices is None else _ptr(state_indices, np.int32)
    rc = _load().ropekv_oracle_gather_delta_rope(_ptr(source, np.float32), _ptr(out, np.float32),
                                                 _ptr(delta_positions, np.int32),
                                                 _ptr(delta_to_seq, np.int32), st, N, batch_size,
                                                 rows, cap, r)
    _check(rc, "gather_delta_rope")
    return out


def paged_fused(k_delta, v_delta, kv_pool, source, old_lengths, delta_lengths, delta_width,
                state_indices, page_table, style):
    """The metadata + gather + paged update composition into a host pool (mutated)."""
    N, Hkv, D = k_delta.shape
    rows, cap, r = source.shape
    B, two, mpps = page_table.shape
    _, num_pages, tpp, hk2, d2 = kv_pool.shape
    assert N == B * delta_width and two == 2 and hk2 == Hkv and d2 == D
    st = ctypes.c_void_p(0) if state_indices is None else _ptr(state_indices, np.int32)
    rc = _load().ropekv_oracle_paged_fused(
        _ptr(k_delta, np.uint16), _ptr(v_delta, np.uint16), _ptr(kv_pool, np.uint16),
        _ptr(source, np.float32), _ptr(np.ascontiguousarray(old_lengths, dtype=np.int32), np.int32),
        _ptr(np.ascontiguousarray(delta_lengths, dtype=np.int32), np.int32), delta_width, st,
        _ptr(page_table, np.int32), B, Hkv, D, r, num_pages, mpps, tpp, rows, cap, style)
    _check(rc, "paged_fused")


def slot_mapping(cos_sin, positions, q, k, v, slots, key_cache, value_cache, q_out, k_out,
                 style):
    """sglang-style call on host arrays. q [T, Hq, D], k / v [T, Hkv, D] may be
    token-strided views (their last two dims contiguous); caches [blocks,
    blockSize, Hkv, D]; q_out [T, Hq, D]; k_out [T, Hkv, D] or None. Mutates the
    caches, q_out and k_out."""
    rows, r = cos_sin.shape
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    blocks, bsz = key_cache.shape[:2]

    def strided(a):
        assert a.dtype == np.uint16 and a.strides[2] == 2 and a.strides[1] == a.shape[2] * 2
        return ctypes.c_void_p(a.ctypes.data), a.strides[0] // 2

    qp, qs = strided(q)
    kp, ks = strided(k)
    vp, vs = strided(v)
    kop = ctypes.c_void_p(0) if k_out is None else _ptr(k_out, np.uint16)
    rc = _load().ropekv_oracle_slot_mapping(
        _ptr(cos_sin, np.float32), _ptr(positions, np.int64), qp, qs, kp, ks, vp, vs,
        _ptr(slots, np.int64), _ptr(key_cache, np.uint16), _ptr(value_cache, np.uint16),
        _ptr(q_out, np.uint16), kop, T, Hq, Hkv, D, r, rows, blocks, bsz, style)
    _check(rc, "slot_mapping")


def capacity_rejected(cos_sin_seq_len: int, kv_capacity: int) -> bool:
    return bool(_load().ropekv_oracle_capacity_rejected(cos_sin_seq_len, kv_capacity))
