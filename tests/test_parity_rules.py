"""The GPU parity tests' comparison rules, checked on the CPU.

Every parity claim rests on parity.compare (FP16 outputs), the rotated-region
masks that say which elements may differ at all, and the E4M3 comparison of
the FP8 cache. Planted differences here must pass or fail exactly as the rule
states: bit-exact outside the rotated region, and inside it at most one FP16
ulp (for |oracle| >= 2^-6) within |gpu - oracle| <= 2^-10 |oracle| + 1e-6.
"""
import numpy as np
import pytest

import workloads
from parity import (TOL_ABS, TOL_REL, ULP_RULE_MIN, cache_rotated, compare, pool_rotated,
                    qkv_rotated, qout_rotated)
from test_gpu_fp8 import compare_e4m3


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def step(bits, k):
    """k FP16 steps away from zero (positive and negative values alike)."""
    return (bits.astype(np.int32) + k).astype(np.uint16)


ROT = (np.arange(16) < 8)[None, :]          # dims 0..7 rotated, 8..15 copied


def _head(seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return f16(rng.uniform(0.1, 4.0, (3, 16)) * rng.choice([-1, 1], (3, 16)))


def test_bound_is_the_stated_one():
    assert TOL_REL == 2.0 ** -10 and TOL_ABS == 1e-6 and ULP_RULE_MIN == 2.0 ** -6


def test_identical_results_pass():
    a = _head()
    assert compare(a, a.copy(), ROT)["n_diff"] == 0


def test_any_difference_outside_the_rotated_region_fails():
    a = _head()
    for flip in (1, 0x0400, 0x8000):         # last bit, exponent bit, sign bit
        b = a.copy()
        b[1, 12] ^= flip
        with pytest.raises(AssertionError, match="outside the rotated region"):
            compare(b, a, ROT)


def test_one_ulp_in_the_rotated_region_passes_two_fail():
    a = _head()
    b = a.copy()
    b[:, :8] = step(a[:, :8], 1)
    assert compare(b, a, ROT)["max_ulp"] == 1
    b[2, 3] = step(a[2:3, 3], 2)[0]
    with pytest.raises(AssertionError, match="off by 2 ulp"):
        compare(b, a, ROT)


def test_signed_zeros_are_equal_only_where_rotated():
    want = f16(np.zeros((1, 16)))
    got = want.copy()
    got[0, 2] = 0x8000                       # -0 in a rotated dim
    compare(got, want, ROT)
    got[0, 10] = 0x8000                      # -0 in a copied dim
    with pytest.raises(AssertionError):
        compare(got, want, ROT)


def test_non_finite_mismatches_fail():
    want = f16(np.ones((1, 16)))
    for bad in (0x7E00, 0x7C00):             # NaN, +inf
        got = want.copy()
        got[0, 1] = bad
        with pytest.raises(AssertionError, match="non-finite"):
            compare(got, want, ROT)


def test_small_magnitudes_follow_the_absolute_term():
    want = f16(np.full((1, 16), 1e-4))       # below 2^-6: the ulp rule does not apply
    got = want.copy()
    got[0, 0] = step(want[:, 0], 3)[0]       # 3 ulp of 6e-8: inside 1e-6 + 2^-10 * 1e-4
    compare(got, want, ROT)
    got[0, 0] = f16([1e-4 + 3e-6])[0]        # 3e-6 off: outside the bound
    with pytest.raises(AssertionError):
        compare(got, want, ROT)


def test_shape_mismatch_fails():
    with pytest.raises(AssertionError):
        compare(_head()[:2], _head(), ROT)


def test_rotated_masks_cover_exactly_the_rotated_dims():
    B, S, Hq, Hkv, D, r, cap = 2, 3, 4, 2, 16, 8, 5
    q = np.broadcast_to(qout_rotated((B, S, Hq, D), r), (B, S, Hq, D))
    assert np.array_equal(q[0, 0, 0], np.arange(D) < r) and q.all(axis=(0, 1, 2)).sum() == r
    c = np.broadcast_to(cache_rotated((B, 2, Hkv, cap, D), r), (B, 2, Hkv, cap, D))
    assert c[:, 0, ..., :r].all() and not c[:, 0, ..., r:].any() and not c[:, 1].any()
    k = np.broadcast_to(qkv_rotated(Hq, Hkv, D, r), (B, S, Hq + 2 * Hkv, D))
    assert k[..., :Hq + Hkv, :r].all() and not k[..., :Hq + Hkv, r:].any()
    assert not k[..., Hq + Hkv:, :].any()    # V heads are copies
    p = np.broadcast_to(pool_rotated((2, 3, 4, Hkv, D), r), (2, 3, 4, Hkv, D))
    assert p[0, ..., :r].all() and not p[0, ..., r:].any() and not p[1].any()


def test_e4m3_rule():
    want = np.array([0x38, 0x40, 0xB8, 0x01, workloads.SENTINEL8], dtype=np.uint8)
    got = want.copy()
    got[:4] = [0x39, 0x3F, 0xB9, 0x02]       # one E4M3 step each (both signs)
    assert compare_e4m3(got, want, "one step")["n_diff"] == 4
    got[0] = 0x3A                            # two steps
    with pytest.raises(AssertionError, match="more than one ulp"):
        compare_e4m3(got, want, "two steps")
    got = want.copy()
    got[4] = 0x38                            # a sentinel byte written
    with pytest.raises(AssertionError, match="untouched"):
        compare_e4m3(got, want, "sentinel")
    got = want.copy()
    got[1] = 0x7F                            # NaN written
    with pytest.raises(AssertionError, match="NaN"):
        compare_e4m3(got, want, "nan")
