"""ctypes binding of libropekv.so.

Each function has the name of the C entry point it calls (include/ropekv.h),
takes torch CUDA tensors in the layouts the header states, checks dtype,
device, contiguity and shape agreement, and passes raw device pointers, the
sizes read from the shapes and the current (or given) stream. It does no
computation: every step runs in the library's kernels. A non-zero status
raises RopeKVError. There is no fallback: without the built library the import
of the functions fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

NEOX = 0
GPTJ = 1

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libropekv.so")

FLOOR_LIB_PATH = os.path.join(_PKG, "lib", "libropekv_floor.so")

_lib = None
_floor_lib = None


class RopeKVError(RuntimeError):
    """A non-zero status from libropekv.so."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status} ({ropekv_status_string(status)})")


class ropekv_dims(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "batch", "seqLen", "numQHeads", "numKVHeads", "headDim", "rotaryDim",
        "kvCapacity", "cosSinBatch", "cosSinSeqLen", "style")]


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load libropekv.so once. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(needs nvcc) -- there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    I32 = ctypes.c_int32
    D = ctypes.POINTER(ropekv_dims)
    lib.rope_write_kv_packed.argtypes = [P, P, P, D, P]
    lib.rope_write_kv_continuous.argtypes = [P, P, P, P, P, D, P]
    lib.rope_write_kv_tree.argtypes = [P, P, P, P, P, P, D, P]
    lib.rope_write_kv_continuous_qknorm.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, D, P]
    lib.rope_write_kv_continuous_fp8.argtypes = [P, P, P, P, P, P, P, D, P]
    lib.paged_kv_delta_update.argtypes = [P] * 7 + [I32] * 9 + [P]
    lib.paged_kv_delta_update_fused.argtypes = [P] * 6 + [I32] + [P] * 2 + [I32] * 10 + [P]
    lib.dflash_prepare_delta_metadata.argtypes = [P, P, I32, P, P, I32, P]
    lib.dflash_gather_delta_rope.argtypes = [P] * 5 + [I32] * 5 + [P]
    I64 = ctypes.c_int64
    lib.rope_write_kv_slot_mapping.argtypes = [P, P, P, I64, P, I64, P, I64, P, P, P, P, P,
                                               I32, I32, I32, I32, I32, I32, I64, I32, I32, P]
    lib.rope_check_capacity.argtypes = [I32, I32]
    lib.ropekv_set_residency_cap.argtypes = [ctypes.c_int]
    lib.ropekv_set_residency_cap.restype = ctypes.c_int
    lib.ropekv_status_string.argtypes = [ctypes.c_int]
    lib.ropekv_status_string.restype = ctypes.c_char_p
    for fn in ("rope_write_kv_packed", "rope_write_kv_continuous", "rope_write_kv_tree",
               "rope_write_kv_continuous_qknorm", "rope_write_kv_continuous_fp8",
               "paged_kv_delta_update", "paged_kv_delta_update_fused",
               "dflash_prepare_delta_metadata", "dflash_gather_delta_rope",
               "rope_write_kv_slot_mapping", "rope_check_capacity"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


class _OnDevice:
    """The library's entry points, each called with ``device`` made the
    calling thread's current CUDA device for the duration of the call: a
    launch, and the residency cap of small launches, act on the current
    device, which need not be the one holding the tensors."""

    def __init__(self, device):
        self._device = device

    def __getattr__(self, name):
        fn = getattr(load_library(), name)

        def call(*args):
            with torch.cuda.device(self._device):
                return fn(*args)
        return call


def ropekv_set_residency_cap(enable: bool) -> bool:
    """Switch the residency cap of decode-sized launches on (default) or off,
    process-wide; returns the previous setting. Results are identical either
    way; see include/ropekv.h for what the cap costs concurrent kernels."""
    return bool(load_library().ropekv_set_residency_cap(1 if enable else 0))


def load_floor_library():
    """Load libropekv_floor.so (the benchmark's decode-floor copy) once."""
    global _floor_lib
    if _floor_lib is None:
        if not os.path.exists(FLOOR_LIB_PATH):
            raise RuntimeError(f"{FLOOR_LIB_PATH} is not built")
        lib = ctypes.CDLL(FLOOR_LIB_PATH)
        lib.ropekv_floor_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
        lib.ropekv_floor_copy.restype = ctypes.c_int
        _floor_lib = lib
    return _floor_lib


def ropekv_floor_copy(src: torch.Tensor, dst: torch.Tensor, threads_per_cta: int = 96,
                      cap: bool = True, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy src to dst (same size, contiguous, on one device) with the launch
    shape and policy of the library's decode-sized launches
    (include/ropekv_floor.h). A measurement reference, not part of the path."""
    if src.numel() * src.element_size() != dst.numel() * dst.element_size():
        raise ValueError("src and dst must have the same size in bytes")
    dev = src.device
    for name, t in (("src", src), ("dst", dst)):
        if t.device != dev or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous on {dev}")
    with torch.cuda.device(dev):
        rc = load_floor_library().ropekv_floor_copy(
            ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()),
            src.numel() * src.element_size(), int(threads_per_cta), 1 if cap else 0,
            _stream_handle(stream, dev))
    if rc != 0:
        raise RuntimeError(f"ropekv_floor_copy: status {rc}")


def ropekv_status_string(status: int) -> str:
    return load_library().ropekv_status_string(int(status)).decode()


def rope_check_capacity(cos_sin_seq_len: int, kv_capacity: int) -> None:
    """Raise RopeKVError when the cos/sin table is longer than the capacity."""
    rc = load_library().rope_check_capacity(int(cos_sin_seq_len), int(kv_capacity))
    if rc != 0:
        raise RopeKVError("rope_check_capacity", rc)


# ------------------------------------------------------------- marshalling --

def _dev_ptr(t: Optional[torch.Tensor], name: str, dtypes, device) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev_rows(t: torch.Tensor, name: str, device):
    """Pointer and token stride of a [T, H, D] FP16 tensor whose last two dims
    are dense (a token-strided view, e.g. a slice of a packed QKV buffer)."""
    if not isinstance(t, torch.Tensor) or t.dim() != 3:
        raise ValueError(f"{name} must be a [T, H, D] tensor")
    if t.dtype not in _F16:
        raise TypeError(f"{name}: dtype {t.dtype} not in {_F16}")
    if t.device.type != "cuda" or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name}: heads and dims must be dense (strides (*, D, 1))")
    return ctypes.c_void_p(t.data_ptr()), int(t.stride(0))


_F16 = (torch.float16, torch.int16)
_I64 = (torch.int64,)
_F32 = (torch.float32,)
_I32 = (torch.int32,)


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_rc(fn: str, rc: int) -> None:
    if rc != 0:
        raise RopeKVError(fn, rc)


def _contiguous_dims(cos_sin, qkv, kv_cache, num_q_heads, num_kv_heads, style) -> ropekv_dims:
    if cos_sin.dim() != 3 or qkv.dim() != 4 or kv_cache.dim() != 5:
        raise ValueError("cos_sin [csB,csS,r], qkv [B,S,H,D], kv_cache [B,2,Hkv,cap,D] expected")
    B, S, H, D = qkv.shape
    if H != num_q_heads + 2 * num_kv_heads:
        raise ValueError(f"qkv has {H} heads, expected Hq + 2*Hkv = {num_q_heads + 2 * num_kv_heads}")
    if kv_cache.shape[0] != B or kv_cache.shape[1] != 2 or kv_cache.shape[2] != num_kv_heads \
            or kv_cache.shape[4] != D:
        raise ValueError(f"kv_cache shape {tuple(kv_cache.shape)} does not match qkv {tuple(qkv.shape)}")
    return ropekv_dims(B, S, num_q_heads, num_kv_heads, D, cos_sin.shape[2], kv_cache.shape[3],
                       cos_sin.shape[0], cos_sin.shape[1], style)


# ------------------------------------------------------------ entry points --

def rope_write_kv_packed(cos_sin: torch.Tensor, qkv: torch.Tensor, kv_cache: torch.Tensor,
                         num_q_heads: int, num_kv_heads: int, style: int = NEOX,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Empty cache: rotate Q and K of ``qkv`` in place and write K, V to slots 0..S-1.

    cos_sin [csB, csS, r] float32; qkv [B, S, Hq+2Hkv, D] float16 (in/out);
    kv_cache [B, 2, Hkv, cap, D] float16 (out).
    """
    dims = _contiguous_dims(cos_sin, qkv, kv_cache, num_q_heads, num_kv_heads, style)
    dev = qkv.device
    rc = _OnDevice(dev).rope_write_kv_packed(
        _dev_ptr(cos_sin, "cos_sin", _F32, dev), _dev_ptr(qkv, "qkv", _F16, dev),
        _dev_ptr(kv_cache, "kv_cache", _F16, dev), ctypes.byref(dims), _stream_handle(stream, dev))
    _check_rc("rope_write_kv_packed", rc)


def rope_write_kv_continuous(cos_sin: torch.Tensor, kv_cache_end_lens: torch.Tensor,
                             qkv: torch.Tensor, kv_cache: torch.Tensor, q_out: torch.Tensor,
                             num_q_heads: int, num_kv_heads: int, style: int = NEOX,
                             stream: Optional[torch.cuda.Stream] = None) -> None:
    """Non-empty cache: token s of sequence b takes slot = position
    kv_cache_end_lens[b] - S + s; rotated Q goes to ``q_out`` [B, S, Hq, D]."""
    dims = _contiguous_dims(cos_sin, qkv, kv_cache, num_q_heads, num_kv_heads, style)
    B, S, _, D = qkv.shape
    if tuple(kv_cache_end_lens.shape) != (B,) or tuple(q_out.shape) != (B, S, num_q_heads, D):
        raise ValueError("kv_cache_end_lens [B] and q_out [B,S,Hq,D] expected")
    dev = qkv.device
    rc = _OnDevice(dev).rope_write_kv_continuous(
        _dev_ptr(cos_sin, "cos_sin", _F32, dev),
        _dev_ptr(kv_cache_end_lens, "kv_cache_end_lens", _I32, dev),
        _dev_ptr(qkv, "qkv", _F16, dev), _dev_ptr(kv_cache, "kv_cache", _F16, dev),
        _dev_ptr(q_out, "q_out", _F16, dev), ctypes.byref(dims), _stream_handle(stream, dev))
    _check_rc("rope_write_kv_continuous", rc)


def rope_write_kv_continuous_qknorm(cos_sin: torch.Tensor, kv_cache_end_lens: torch.Tensor,
                                    qkv: torch.Tensor, kv_cache: torch.Tensor, q_out: torch.Tensor,
                                    q_norm_weight: torch.Tensor, k_norm_weight: torch.Tensor,
                                    eps: float, num_q_heads: int, num_kv_heads: int,
                                    style: int = NEOX,
                                    stream: Optional[torch.cuda.Stream] = None) -> None:
    """rope_write_kv_continuous with per-head RMS normalization of Q and K
    (weights [D] float16) before the rotation."""
    dims = _contiguous_dims(cos_sin, qkv, kv_cache, num_q_heads, num_kv_heads, style)
    B, S, _, D = qkv.shape
    if tuple(kv_cache_end_lens.shape) != (B,) or tuple(q_out.shape) != (B, S, num_q_heads, D) \
            or tuple(q_norm_weight.shape) != (D,) or tuple(k_norm_weight.shape) != (D,):
        raise ValueError("kv_cache_end_lens [B], q_out [B,S,Hq,D], norm weights [D] expected")
    dev = qkv.device
    rc = _OnDevice(dev).rope_write_kv_continuous_qknorm(
        _dev_ptr(cos_sin, "cos_sin", _F32, dev),
        _dev_ptr(kv_cache_end_lens, "kv_cache_end_lens", _I32, dev),
        _dev_ptr(qkv, "qkv", _F16, dev), _dev_ptr(kv_cache, "kv_cache", _F16, dev),
        _dev_ptr(q_out, "q_out", _F16, dev), _dev_ptr(q_norm_weight, "q_norm_weight", _F16, dev),
        _dev_ptr(k_norm_weight, "k_norm_weight", _F16, dev), float(eps), ctypes.byref(dims),
        _stream_handle(stream, dev))
    _check_rc("rope_write_kv_continuous_qknorm", rc)


_U8 = (torch.uint8, torch.float8_e4m3fn) if hasattr(torch, "float8_e4m3fn") else (torch.uint8,)


def rope_write_kv_continuous_fp8(cos_sin: torch.Tensor, kv_cache_end_lens: torch.Tensor,
                                 qkv: torch.Tensor, kv_cache: torch.Tensor, q_out: torch.Tensor,
                                 k_scale: torch.Tensor, v_scale: torch.Tensor,
                                 num_q_heads: int, num_kv_heads: int, style: int = NEOX,
                                 stream: Optional[torch.cuda.Stream] = None) -> None:
    """rope_write_kv_continuous with an E4M3 cache [B, 2, Hkv, cap, D] (uint8 or
    float8_e4m3fn) and per-tensor scales (one-element float32 device tensors)."""
    dims = _contiguous_dims(cos_sin, qkv, kv_cache, num_q_heads, num_kv_heads, style)
    B, S, _, D = qkv.shape
    if tuple(kv_cache_end_lens.shape) != (B,) or tuple(q_out.shape) != (B, S, num_q_heads, D) \
            or k_scale.numel() != 1 or v_scale.numel() != 1:
        raise ValueError("kv_cache_end_lens [B], q_out [B,S,Hq,D], one-element scales expected")
    dev = qkv.device
    rc = _OnDevice(dev).rope_write_kv_continuous_fp8(
        _dev_ptr(cos_sin, "cos_sin", _F32, dev),
        _dev_ptr(kv_cache_end_lens, "kv_cache_end_lens", _I32, dev),
        _dev_ptr(qkv, "qkv", _F16, dev), _dev_ptr(kv_cache, "kv_cache", _U8, dev),
        _dev_ptr(q_out, "q_out", _F16, dev), _dev_ptr(k_scale, "k_scale", _F32, dev),
        _dev_ptr(v_scale, "v_scale", _F32, dev), ctypes.byref(dims), _stream_handle(stream, dev))
    _check_rc("rope_write_kv_continuous_fp8", rc)


def rope_write_kv_tree(cos_sin: torch.Tensor, kv_cache_end_lens: torch.Tensor,
                       token_pos_ids: torch.Tensor, qkv: torch.Tensor, kv_cache: torch.Tensor,
                       q_out: torch.Tensor, num_q_heads: int, num_kv_heads: int,
                       style: int = NEOX, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Tree speculative decoding: RoPE position token_pos_ids[b, s], cache slot
    kv_cache_end_lens[b] - S + s."""
    dims = _contiguous_dims(cos_sin, qkv, kv_cache, num_q_heads, num_kv_heads, style)
    B, S, _, D = qkv.shape
    if tuple(kv_cache_end_lens.shape) != (B,) or tuple(token_pos_ids.shape) != (B, S) \
            or tuple(q_out.shape) != (B, S, num_q_heads, D):
        raise ValueError("kv_cache_end_lens [B], token_pos_ids [B,S], q_out [B,S,Hq,D] expected")
    dev = qkv.device
    rc = _OnDevice(dev).rope_write_kv_tree(
        _dev_ptr(cos_sin, "cos_sin", _F32, dev),
        _dev_ptr(kv_cache_end_lens, "kv_cache_end_lens", _I32, dev),
        _dev_ptr(token_pos_ids, "token_pos_ids", _I32, dev),
        _dev_ptr(qkv, "qkv", _F16, dev), _dev_ptr(kv_cache, "kv_cache", _F16, dev),
        _dev_ptr(q_out, "q_out", _F16, dev), ctypes.byref(dims), _stream_handle(stream, dev))
    _check_rc("rope_write_kv_tree", rc)


def paged_kv_delta_update(k_delta: torch.Tensor, v_delta: torch.Tensor, kv_cache: torch.Tensor,
                          token_aligned_cos_sin: torch.Tensor, delta_positions: torch.Tensor,
                          delta_token_to_sequence: torch.Tensor, page_table: torch.Tensor,
                          batch_size: Optional[int] = None, style: int = NEOX,
                          stream: Optional[torch.cuda.Stream] = None) -> None:
    """Paged delta update. k_delta, v_delta [N, Hkv, D] float16;
    kv_cache [2, numPages, tokensPerPage, Hkv, D] float16; token_aligned_cos_sin
    [N, r] float32; delta_positions, delta_token_to_sequence [N] int32;
    page_table [B, 2, maxPagesPerSeq] int32. batch_size defaults to B."""
    if k_delta.dim() != 3 or kv_cache.dim() != 5 or page_table.dim() != 3 \
            or token_aligned_cos_sin.dim() != 2:
        raise ValueError("k_delta [N,Hkv,D], kv_cache [2,P,TPP,Hkv,D], page_table [B,2,M], "
                         "token_aligned_cos_sin [N,r] expected")
    N, Hkv, D = k_delta.shape
    two, num_pages, tpp, hk2, d2 = kv_cache.shape
    B, two_b, mpps = page_table.shape
    if tuple(v_delta.shape) != (N, Hkv, D) or two != 2 or hk2 != Hkv or d2 != D or two_b != 2 \
            or token_aligned_cos_sin.shape[0] != N or tuple(delta_positions.shape) != (N,) \
            or tuple(delta_token_to_sequence.shape) != (N,):
        raise ValueError("inconsistent shapes for paged_kv_delta_update")
    if batch_size is None:
        batch_size = B
    if batch_size > B:
        raise ValueError("batch_size exceeds the page table's rows")
    dev = k_delta.device
    rc = _OnDevice(dev).paged_kv_delta_update(
        _dev_ptr(k_delta, "k_delta", _F16, dev), _dev_ptr(v_delta, "v_delta", _F16, dev),
        _dev_ptr(kv_cache, "kv_cache", _F16, dev),
        _dev_ptr(token_aligned_cos_sin, "token_aligned_cos_sin", _F32, dev),
        _dev_ptr(delta_positions, "delta_positions", _I32, dev),
        _dev_ptr(delta_token_to_sequence, "delta_token_to_sequence", _I32, dev),
        _dev_ptr(page_table, "page_table", _I32, dev),
        N, batch_size, Hkv, D, token_aligned_cos_sin.shape[1], num_pages, mpps, tpp, style,
        _stream_handle(stream, dev))
    _check_rc("paged_kv_delta_update", rc)


def paged_kv_delta_update_fused(k_delta: torch.Tensor, v_delta: torch.Tensor,
                                kv_cache: torch.Tensor, cos_sin_source: torch.Tensor,
                                old_draft_cache_lengths: torch.Tensor,
                                delta_lengths: torch.Tensor, page_table: torch.Tensor,
                                state_indices: Optional[torch.Tensor] = None, style: int = NEOX,
                                stream: Optional[torch.cuda.Stream] = None) -> None:
    """DFlash metadata + cos/sin gather + paged update in one launch.

    k_delta, v_delta [B * W, Hkv, D] float16 (row b*W + j = sequence b's token j);
    kv_cache [2, numPages, tokensPerPage, Hkv, D] float16; cos_sin_source
    [sourceRows, cacheCapacity, r] float32; old_draft_cache_lengths, delta_lengths
    [B] int32; page_table [B, 2, maxPagesPerSeq] int32; state_indices [B] int32 or None.
    """
    if k_delta.dim() != 3 or kv_cache.dim() != 5 or page_table.dim() != 3 \
            or cos_sin_source.dim() != 3:
        raise ValueError("k_delta [B*W,Hkv,D], kv_cache [2,P,TPP,Hkv,D], page_table [B,2,M], "
                         "cos_sin_source [rows,cap,r] expected")
    N, Hkv, D = k_delta.shape
    two, num_pages, tpp, hk2, d2 = kv_cache.shape
    B, two_b, mpps = page_table.shape
    rows, cap, r = cos_sin_source.shape
    if B == 0 or N % B != 0:
        raise ValueError("k_delta rows must be batch * deltaWidth")
    width = N // B
    if tuple(v_delta.shape) != (N, Hkv, D) or two != 2 or hk2 != Hkv or d2 != D or two_b != 2 \
            or tuple(old_draft_cache_lengths.shape) != (B,) or tuple(delta_lengths.shape) != (B,) \
            or (state_indices is not None and tuple(state_indices.shape) != (B,)):
        raise ValueError("inconsistent shapes for paged_kv_delta_update_fused")
    dev = k_delta.device
    rc = _OnDevice(dev).paged_kv_delta_update_fused(
        _dev_ptr(k_delta, "k_delta", _F16, dev), _dev_ptr(v_delta, "v_delta", _F16, dev),
        _dev_ptr(kv_cache, "kv_cache", _F16, dev),
        _dev_ptr(cos_sin_source, "cos_sin_source", _F32, dev),
        _dev_ptr(old_draft_cache_lengths, "old_draft_cache_lengths", _I32, dev),
        _dev_ptr(delta_lengths, "delta_lengths", _I32, dev), width,
        _dev_ptr(state_indices, "state_indices", _I32, dev),
        _dev_ptr(page_table, "page_table", _I32, dev),
        B, Hkv, D, r, num_pages, mpps, tpp, rows, cap, style, _stream_handle(stream, dev))
    _check_rc("paged_kv_delta_update_fused", rc)


def dflash_prepare_delta_metadata(old_draft_cache_lengths: torch.Tensor,
                                  delta_lengths: torch.Tensor, delta_width: int,
                                  delta_positions: torch.Tensor,
                                  delta_token_to_sequence: torch.Tensor,
                                  stream: Optional[torch.cuda.Stream] = None) -> None:
    """Rows [B, delta_width]: position old[b] + j and sequence b when j < delta_lengths[b],
    else -1 / -1. Outputs are int32 tensors of B * delta_width elements."""
    B = old_draft_cache_lengths.shape[0]
    if tuple(delta_lengths.shape) != (B,) or delta_positions.numel() != B * delta_width \
            or delta_token_to_sequence.numel() != B * delta_width:
        raise ValueError("inconsistent shapes for dflash_prepare_delta_metadata")
    dev = old_draft_cache_lengths.device
    rc = _OnDevice(dev).dflash_prepare_delta_metadata(
        _dev_ptr(old_draft_cache_lengths, "old_draft_cache_lengths", _I32, dev),
        _dev_ptr(delta_lengths, "delta_lengths", _I32, dev), int(delta_width),
        _dev_ptr(delta_positions, "delta_positions", _I32, dev),
        _dev_ptr(delta_token_to_sequence, "delta_token_to_sequence", _I32, dev), B,
        _stream_handle(stream, dev))
    _check_rc("dflash_prepare_delta_metadata", rc)


def dflash_gather_delta_rope(source: torch.Tensor, output: torch.Tensor,
                             delta_positions: torch.Tensor, delta_token_to_sequence: torch.Tensor,
                             state_indices: Optional[torch.Tensor] = None,
                             batch_size: Optional[int] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> None:
    """output[t] = source[state(seq_t), pos_t] (zero rows where out of range).
    source [sourceRows, cacheCapacity, r] float32; output [N, r] float32;
    batch_size defaults to len(state_indices) when given, else to N."""
    if source.dim() != 3 or output.dim() != 2:
        raise ValueError("source [rows,cap,r] and output [N,r] expected")
    rows, cap, r = source.shape
    N = output.shape[0]
    if output.shape[1] != r or delta_positions.numel() != N or delta_token_to_sequence.numel() != N:
        raise ValueError("inconsistent shapes for dflash_gather_delta_rope")
    if batch_size is None:
        batch_size = state_indices.shape[0] if state_indices is not None else N
    dev = output.device
    rc = _OnDevice(dev).dflash_gather_delta_rope(
        _dev_ptr(source, "source", _F32, dev), _dev_ptr(output, "output", _F32, dev),
        _dev_ptr(delta_positions, "delta_positions", _I32, dev),
        _dev_ptr(delta_token_to_sequence, "delta_token_to_sequence", _I32, dev),
        _dev_ptr(state_indices, "state_indices", _I32, dev), N, int(batch_size), rows, cap, r,
        _stream_handle(stream, dev))
    _check_rc("dflash_gather_delta_rope", rc)


def rope_write_kv_slot_mapping(cos_sin: torch.Tensor, positions: torch.Tensor, q: torch.Tensor,
                               k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                               key_cache: torch.Tensor, value_cache: torch.Tensor,
                               q_out: torch.Tensor, k_out: Optional[torch.Tensor] = None,
                               style: int = NEOX,
                               stream: Optional[torch.cuda.Stream] = None) -> None:
    """sglang-style interface: cos_sin [rows, r] float32; positions, slot_mapping
    [T] int64; q [T, Hq, D], k, v [T, Hkv, D] float16 (token-strided views allowed);
    key_cache, value_cache [blocks, block_size, Hkv, D] float16; q_out [T, Hq, D];
    k_out [T, Hkv, D] or None. A negative slot skips that token's cache writes."""
    dev = q.device
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if cos_sin.dim() != 2 or tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D) \
            or tuple(positions.shape) != (T,) or tuple(slot_mapping.shape) != (T,) \
            or key_cache.dim() != 4 or tuple(key_cache.shape[2:]) != (Hkv, D) \
            or tuple(value_cache.shape) != tuple(key_cache.shape) \
            or tuple(q_out.shape) != (T, Hq, D) \
            or (k_out is not None and tuple(k_out.shape) != (T, Hkv, D)):
        raise ValueError("inconsistent shapes for rope_write_kv_slot_mapping")
    qp, qs = _dev_rows(q, "q", dev)
    kp, ks = _dev_rows(k, "k", dev)
    vp, vs = _dev_rows(v, "v", dev)
    rc = _OnDevice(dev).rope_write_kv_slot_mapping(
        _dev_ptr(cos_sin, "cos_sin", _F32, dev), _dev_ptr(positions, "positions", _I64, dev),
        qp, qs, kp, ks, vp, vs, _dev_ptr(slot_mapping, "slot_mapping", _I64, dev),
        _dev_ptr(key_cache, "key_cache", _F16, dev), _dev_ptr(value_cache, "value_cache", _F16, dev),
        _dev_ptr(q_out, "q_out", _F16, dev), _dev_ptr(k_out, "k_out", _F16, dev),
        T, Hq, Hkv, D, cos_sin.shape[1], cos_sin.shape[0], key_cache.shape[0], key_cache.shape[1],
        style, _stream_handle(stream, dev))
    _check_rc("rope_write_kv_slot_mapping", rc)
