"""Fused RoPE + KV-cache write for GB300 (sm_103a).

The compute lives in ``lib/libropekv.so`` (C ABI: ``include/ropekv.h``; kernels:
``csrc/``). This package is its Python binding: functions with the entry
points' names that take torch CUDA tensors and launch on the current stream.
"""
from ._binding import (  # noqa: F401
    GPTJ,
    NEOX,
    LIB_PATH,
    RopeKVError,
    dflash_gather_delta_rope,
    dflash_prepare_delta_metadata,
    library_path,
    load_library,
    paged_kv_delta_update,
    paged_kv_delta_update_fused,
    rope_check_capacity,
    ropekv_floor_copy,
    ropekv_set_residency_cap,
    rope_write_kv_continuous,
    rope_write_kv_continuous_fp8,
    rope_write_kv_continuous_qknorm,
    rope_write_kv_packed,
    rope_write_kv_slot_mapping,
    rope_write_kv_tree,
    ropekv_status_string,
)

__all__ = [
    "NEOX", "GPTJ", "RopeKVError", "load_library", "library_path",
    "rope_write_kv_packed", "rope_write_kv_continuous", "rope_write_kv_continuous_qknorm",
    "rope_write_kv_continuous_fp8",
    "rope_write_kv_tree",
    "paged_kv_delta_update", "paged_kv_delta_update_fused", "dflash_prepare_delta_metadata",
    "dflash_gather_delta_rope", "rope_write_kv_slot_mapping", "rope_check_capacity",
    "ropekv_set_residency_cap", "ropekv_floor_copy", "ropekv_status_string",
]
