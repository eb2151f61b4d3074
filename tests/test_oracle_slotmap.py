"""Pins for the oracle's sglang-style call (separate Q/K/V, flat slot mapping).

sglang rope_cache.py, fused_qk_rope_reshape_and_cache with the flash layout:
slot s goes to block s // block_size, offset s % block_size (Stage 3.1 and 3.4);
a negative slot skips the K/V cache writes and k_out but not Q (Stage 3.2);
k_out holds the rotated K (Stage 3.2). Written out by hand below with integer
codes and "scale" cos/sin rows (cos 0, sin 2^p in row p) that reveal the row
each output used.
"""
import numpy as np
import pytest

import oracle
import workloads
from test_oracle_entries import coded_qkv, identity_table, rotated_scaled, scale_table, val

SENT = workloads.SENTINEL


def _views(T, Hq, Hkv, D):
    qkv = coded_qkv(1, T, Hq + 2 * Hkv, D)[0]          # [T, H, D]
    return qkv, qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_slot_mapping_placement_by_hand(style):
    T, Hq, Hkv, D, r, bsz, blocks = 5, 2, 1, 16, 16, 4, 3
    qkv, q, k, v = _views(T, Hq, Hkv, D)
    assert q.strides[0] == 4 * D * 2      # token-strided views into the packed row
    cs = scale_table(4, r)[0]             # rows 0..3
    positions = np.array([3, 0, 1, 2, 1], dtype=np.int64)
    slots = np.array([5, -1, 0, 11, 12], dtype=np.int64)   # 12 == blocks*bsz: skipped
    kc = workloads.sentinel_fill((blocks, bsz, Hkv, D))
    vc = workloads.sentinel_fill((blocks, bsz, Hkv, D))
    qo = workloads.sentinel_fill((T, Hq, D))
    ko = workloads.sentinel_fill((T, Hkv, D))
    oracle.slot_mapping(cs, positions, q, k, v, slots, kc, vc, qo, ko, style)
    for t in range(T):
        for h in range(Hq):
            want = rotated_scaled(val(q[t, h]), r, style, positions[t])
            assert np.array_equal(val(qo[t, h]), want)
    # hand-written destinations: token -> (block, offset)
    dest = {0: (1, 1), 2: (0, 0), 3: (2, 3)}
    written = np.zeros((blocks, bsz), dtype=bool)
    for t, (blk, off) in dest.items():
        written[blk, off] = True
        want = rotated_scaled(val(k[t, 0]), r, style, positions[t])
        assert np.array_equal(val(kc[blk, off, 0]), want)
        assert np.array_equal(vc[blk, off, 0], v[t, 0])
        assert np.array_equal(ko[t], kc[blk, off])
    assert np.all(kc[~written] == SENT) and np.all(vc[~written] == SENT)
    assert np.all(ko[1] == SENT) and np.all(ko[4] == SENT)


def test_slot_mapping_position_out_of_table_skips_token():
    T, Hq, Hkv, D, r = 3, 2, 1, 16, 16
    qkv, q, k, v = _views(T, Hq, Hkv, D)
    cs = identity_table(4, r)[0]
    positions = np.array([4, -1, 2], dtype=np.int64)
    slots = np.array([0, 1, 2], dtype=np.int64)
    kc = workloads.sentinel_fill((1, 4, Hkv, D))
    vc = workloads.sentinel_fill((1, 4, Hkv, D))
    qo = workloads.sentinel_fill((T, Hq, D))
    oracle.slot_mapping(cs, positions, q, k, v, slots, kc, vc, qo, None, oracle.NEOX)
    assert np.all(qo[:2] == SENT) and np.all(kc[0, :2] == SENT) and np.all(vc[0, :2] == SENT)
    assert np.array_equal(qo[2], q[2]) and np.array_equal(kc[0, 2], k[2])
    assert np.array_equal(vc[0, 2], v[2]) and np.all(kc[0, 3] == SENT)


def test_slot_mapping_gqa_heads():
    T, Hq, Hkv, D, r = 2, 4, 2, 16, 16
    qkv = coded_qkv(1, T, 8, D, tok_stride=128)[0]
    q, k, v = qkv[:, :4], qkv[:, 4:6], qkv[:, 6:8]
    cs = identity_table(2, r)[0]
    kc = workloads.sentinel_fill((2, 2, Hkv, D))
    vc = workloads.sentinel_fill((2, 2, Hkv, D))
    qo = workloads.sentinel_fill((T, Hq, D))
    oracle.slot_mapping(cs, np.array([0, 1], dtype=np.int64), q, k, v,
                        np.array([3, 0], dtype=np.int64), kc, vc, qo, None, oracle.GPTJ)
    assert np.array_equal(kc[1, 1], k[0]) and np.array_equal(vc[1, 1], v[0])
    assert np.array_equal(kc[0, 0], k[1]) and np.array_equal(vc[0, 0], v[1])
    assert np.array_equal(qo, q)


def test_slot_mapping_separate_strides():
    """q, k and v each carry their own token stride (sglang rope_cache.py passes
    q_stride_t, k_stride_t and v_stride_t separately). Here q and v are views
    into two differently padded buffers and k is a plain array; every output
    must still come from its own token's row."""
    T, Hq, Hkv, D, r = 3, 2, 1, 16, 16
    qbuf = coded_qkv(1, T, 5, D, tok_stride=1000)[0]          # stride 5 heads
    vbuf = coded_qkv(1, T, 3, D, tok_stride=1000)[0] + 7      # stride 3 heads
    q, v = qbuf[:, 1:1 + Hq], vbuf[:, 2:2 + Hkv]
    k = np.ascontiguousarray(coded_qkv(1, T, Hkv, D, tok_stride=1000)[0] + 3)
    assert len({q.strides[0], k.strides[0], v.strides[0]}) == 3
    cs = identity_table(2, r)[0]
    kc = workloads.sentinel_fill((1, 4, Hkv, D))
    vc = workloads.sentinel_fill((1, 4, Hkv, D))
    qo = workloads.sentinel_fill((T, Hq, D))
    oracle.slot_mapping(cs, np.array([0, 0, 0], dtype=np.int64), q, k, v,
                        np.array([2, 0, 3], dtype=np.int64), kc, vc, qo, None, oracle.NEOX)
    assert np.array_equal(qo, q)
    for t, slot in enumerate((2, 0, 3)):
        assert np.array_equal(kc[0, slot], k[t]) and np.array_equal(vc[0, slot], v[t])
    assert np.all(kc[0, 1] == SENT) and np.all(vc[0, 1] == SENT)


@pytest.mark.parametrize("Hq,Hkv,r", [(3, 2, 16), (2, 1, 15)])
def test_slot_mapping_rejects_invalid_dims(Hq, Hkv, r):
    """Q heads in whole groups per KV head (QH_PER_KH = qh // kh) and an even
    rotary width: anything else is an error that writes nothing."""
    T, D = 2, 16
    qkv = coded_qkv(1, T, Hq + 2 * Hkv, D)[0]
    q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    cs = np.zeros((2, r), dtype=np.float32)
    kc = workloads.sentinel_fill((1, 4, Hkv, D))
    vc = workloads.sentinel_fill((1, 4, Hkv, D))
    qo = workloads.sentinel_fill((T, Hq, D))
    with pytest.raises(ValueError):
        oracle.slot_mapping(cs, np.zeros(T, dtype=np.int64), q, k, v,
                            np.arange(T, dtype=np.int64), kc, vc, qo, None, oracle.NEOX)
    assert np.all(kc == SENT) and np.all(vc == SENT) and np.all(qo == SENT)
