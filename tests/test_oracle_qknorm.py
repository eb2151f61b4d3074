"""Pins for the oracle's pre-RoPE QK RMS normalization.

Reading of libmir-cuda execution.rs (qkv_postprocess: query_norm / key_norm
weights, epsilon, then RoPE, then the KV store) and of "Dflash Runtime
Kernels" (K deltas arrive "k_normed"): x_hat = x / sqrt(mean(x^2) + eps) * w
per head, before the rotation. Pinned by closed forms (constant heads, unit
RMS, scale invariance, a single weighted dim) and by reduction to the plain
continuous call on inputs whose RMS is exactly 1.
"""
import math

import numpy as np
import pytest

import oracle
import workloads


def _w(values):
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_constant_head_normalizes_to_weight():
    D = 64
    for c in (3.0, -0.25, 1e-3):
        y = oracle.rms_norm_f64(np.full(D, c), _w(np.ones(D)), 0.0)
        assert np.allclose(y, np.sign(c), rtol=0, atol=1e-15)
    # with eps: c / sqrt(c^2 + eps)
    y = oracle.rms_norm_f64(np.full(D, 2.0), _w(np.ones(D)), 0.5)
    assert np.allclose(y, 2.0 / math.sqrt(4.5), rtol=1e-15)


def test_unit_rms_and_scale_invariance():
    rng = np.random.Generator(np.random.PCG64(3))
    for D in (64, 128, 256):
        x = rng.standard_normal(D)
        y = oracle.rms_norm_f64(x, _w(np.ones(D)), 0.0)
        assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-14
        y2 = oracle.rms_norm_f64(37.5 * x, _w(np.ones(D)), 0.0)
        assert np.allclose(y, y2, rtol=1e-14, atol=0)


def test_weight_scales_its_own_dim_only():
    D = 128
    x = np.linspace(-2, 2, D)
    w = np.ones(D)
    w[5] = 2.0
    base = oracle.rms_norm_f64(x, _w(np.ones(D)), 1e-6)
    y = oracle.rms_norm_f64(x, _w(w), 1e-6)
    assert y[5] == 2 * base[5]
    assert np.array_equal(np.delete(y, 5), np.delete(base, 5))


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_unit_rms_inputs_reduce_to_the_plain_call(style):
    """Heads of +-1 have RMS exactly 1: with unit weights and eps 0 the
    normalized call must give the plain continuous call's bytes."""
    rng = workloads.rng_for(8)
    B, S, Hq, Hkv, D, r, cap = 2, 5, 4, 2, 64, 32, 16
    signs = np.where(rng.random((B, S, Hq + 2 * Hkv, D)) < 0.5, -1.0, 1.0)
    qkv = signs.astype(np.float16).view(np.uint16)
    cs = workloads.cos_sin_table(1e4, cap, r)
    end = np.array([7, 16], dtype=np.int32)
    ones = _w(np.ones(D))
    c1, q1 = workloads.sentinel_fill((B, 2, Hkv, cap, D)), workloads.sentinel_fill((B, S, Hq, D))
    c2, q2 = workloads.sentinel_fill((B, 2, Hkv, cap, D)), workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(cs, end, qkv, c1, q1, Hq, Hkv, style)
    oracle.continuous_qknorm(cs, end, qkv, c2, q2, ones, ones, 0.0, Hq, Hkv, style)
    assert np.array_equal(c1, c2) and np.array_equal(q1, q2)


def test_q_and_k_use_their_own_weights_and_v_is_copied():
    B, S, Hq, Hkv, D, r, cap = 1, 1, 2, 1, 64, 64, 4
    qkv = np.full((B, S, 4, D), 1.0).astype(np.float16).view(np.uint16)
    cs = workloads.cos_sin_table(1e4, cap, r)     # position 0 is the identity row
    end = np.array([1], dtype=np.int32)
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qo = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous_qknorm(cs, end, qkv, cache, qo, _w(np.full(D, 0.5)), _w(np.full(D, 4.0)),
                             0.0, Hq, Hkv, oracle.NEOX)
    assert np.all(qo.view(np.float16) == 0.5)
    assert np.all(cache[0, 0, 0, 0].view(np.float16) == 4.0)
    assert np.array_equal(cache[0, 1, 0, 0], qkv[0, 0, 3])


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_partial_rotary_tail_is_normalized_with_weights(style):
    """Constant heads c with eps 0 normalize to sign(c) * w exactly. With
    r < D and weights that differ per dim, dims past rotaryDim must hold
    fp16(sign(c) * w[d]) -- normalized, not the input bits -- and rotated dims
    must be rotate(sign(c) * w) * 2^p for a "scale" row p (cos 0, sin 2^p):
    the weight is applied before the rotation, on the head's own dims."""
    B, S, Hq, Hkv, D, r, cap = 1, 2, 2, 1, 64, 32, 4
    consts = {(0, 0): 3.0, (0, 1): -0.25, (0, 2): 0.5, (1, 0): -2.0, (1, 1): 1.0, (1, 2): 4.0}
    qkv = np.zeros((B, S, Hq + 2 * Hkv, D), dtype=np.float64)
    for (s, h), c in consts.items():
        qkv[0, s, h] = c
    qkv[0, :, 3] = np.arange(D) / 8.0                     # V heads: copied as bits
    qkv = qkv.astype(np.float16).view(np.uint16)
    wq = 1.0 + np.arange(D) / 64.0                        # exact in FP16
    wk = 2.0 - np.arange(D) / 128.0
    cs = np.zeros((1, cap, r), dtype=np.float32)
    for p in range(cap):
        cs[0, p, r // 2:] = 2.0 ** p
    end = np.array([3], dtype=np.int32)                   # positions 1, 2
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qo = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous_qknorm(cs, end, qkv, cache, qo, _w(wq), _w(wk), 0.0, Hq, Hkv, style)
    h = r // 2
    for s in range(S):
        p = s + 1
        for head in range(3):
            w = wq if head < Hq else wk
            n = np.sign(consts[(s, head)]) * w
            want = n.copy()
            for d in range(r):
                if style == oracle.NEOX:
                    want[d] = (-n[d + h] if d < h else n[d - h]) * 2.0 ** p
                else:
                    want[d] = (-n[d + 1] if d % 2 == 0 else n[d - 1]) * 2.0 ** p
            got = qo[0, s, head] if head < Hq else cache[0, 0, 0, p]
            assert np.array_equal(got.view(np.float16).astype(np.float64), want), (s, head)
        assert np.array_equal(cache[0, 1, 0, p], qkv[0, s, 3])


def test_qknorm_position_past_table_is_skipped():
    # as the continuous call: a slot/position >= cosSinSeqLen writes nothing
    B, S, Hq, Hkv, D, r, cap = 1, 3, 2, 1, 64, 64, 8
    qkv = np.ones((B, S, 4, D)).astype(np.float16).view(np.uint16)
    big = np.zeros((1, 6, r), dtype=np.float32)
    big[0, :, : r // 2] = 1.0
    big[0, 5] = 2.0 ** 10                                 # one row past the table
    cs = big[:, :5]
    end = np.array([6], dtype=np.int32)                   # positions 3, 4, 5
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qo = workloads.sentinel_fill((B, S, Hq, D))
    ones = _w(np.ones(D))
    oracle.continuous_qknorm(cs, end, qkv, cache, qo, ones, ones, 0.0, Hq, Hkv, oracle.NEOX)
    assert np.all(qo[0, 2] == workloads.SENTINEL) and np.all(cache[0, :, 0, 5] == workloads.SENTINEL)
    assert np.all(qo[0, :2].view(np.float16) == 1.0)
    assert np.all(cache[0, 0, 0, 3:5].view(np.float16) == 1.0)


def test_entry_point_applies_its_eps():
    """The call's eps enters the RMS denominator (libmir-cuda execution.rs,
    qkv_postprocess: x / sqrt(mean(x^2) + eps) * w): a constant head c at
    position 0 becomes c / sqrt(c^2 + eps), rounded once to FP16 (numpy's
    float16 conversion, an independent library routine, rounds it here)."""
    B, S, Hq, Hkv, D, r, cap = 1, 1, 1, 1, 64, 64, 2
    qkv = np.zeros((B, S, 3, D))
    qkv[0, 0, 0], qkv[0, 0, 1], qkv[0, 0, 2] = 2.0, -1.0, 0.75
    qkv = qkv.astype(np.float16).view(np.uint16)
    cs = workloads.cos_sin_table(1e4, cap, r)      # row 0: the identity
    ones = _w(np.ones(D))
    for eps in (0.5, 3.0):
        cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
        qo = workloads.sentinel_fill((B, S, Hq, D))
        oracle.continuous_qknorm(cs, np.array([1], dtype=np.int32), qkv, cache, qo, ones, ones,
                                 eps, Hq, Hkv, oracle.NEOX)
        want_q = np.float16(2.0 / math.sqrt(4.0 + eps))
        want_k = np.float16(-1.0 / math.sqrt(1.0 + eps))
        assert np.all(qo.view(np.float16) == want_q), eps
        assert np.all(cache[0, 0, 0, 0].view(np.float16) == want_k), eps
        assert np.array_equal(cache[0, 1, 0, 0], qkv[0, 0, 2])
