"""Pins for the oracle's IEEE 754 binary16 encode/decode.

The oracle writes its own FP16 conversions from the binary16 definition. They
are pinned here against numpy's float16 (an independent library routine) and
against the exact round trip over every bit pattern.
"""
import math

import numpy as np
import pytest

import oracle


def _np_f16_bits(x: np.ndarray) -> np.ndarray:
    # overflow to infinity is one of the cases under test
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_decode_all_bit_patterns_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64_array(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle.f16_to_f64(0x8000)) == -1.0


def test_round_trip_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = oracle.f16_to_f64_array(bits)
    enc = oracle.f64_to_f16_array(dec)
    nan = np.isnan(dec)
    assert np.array_equal(enc[~nan], bits[~nan])
    # NaN inputs stay NaN (exponent all ones, fraction non-zero)
    assert np.all((enc[nan] & 0x7C00) == 0x7C00) and np.all((enc[nan] & 0x03FF) != 0)


def _hard_doubles(rng, n):
    """Random doubles biased towards the cases that break a hand-written RNE:
    exact ties between neighbours, values just off a tie, subnormals, the
    normal/subnormal boundary, overflow and binade edges."""
    finite = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    vals = finite.view(np.float16).astype(np.float64)
    lo = vals[:-1]
    hi = vals[1:]
    pick = rng.integers(0, len(lo), size=n // 4)
    mid = (lo[pick] + hi[pick]) / 2.0                      # exact ties
    eps = np.abs(hi[pick] - lo[pick]) * 1e-6
    near = mid + np.where(rng.random(n // 4) < 0.5, -eps, eps)  # just off a tie
    wide = np.ldexp(rng.random(n // 4) + 0.5, rng.integers(-30, 18, size=n // 4))
    sub = rng.random(n // 8) * 2.0 ** -14                   # subnormal range
    specials = np.array([0.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14,
                         2.0 ** -14 - 2.0 ** -25, 65504.0, 65519.999, 65520.0, 65536.0,
                         1e300, 2.0 ** -1074, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                         2048.0 + 1.0, 2048.0 + 3.0])
    allv = np.concatenate([mid, near, wide, sub, specials])
    signs = np.where(rng.random(len(allv)) < 0.5, -1.0, 1.0)
    out = allv * signs
    return out[: n] if len(out) > n else out


def test_rne_matches_numpy_on_hard_doubles():
    rng = np.random.Generator(np.random.PCG64(1234))
    x = _hard_doubles(rng, 1_000_000)
    ours = oracle.f64_to_f16_array(x)
    ref = _np_f16_bits(x)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"first mismatch x={x[bad[0]]!r}: {ours[bad[0]]:#06x} vs {ref[bad[0]]:#06x}"


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3C00), (-2.0, 0xC000), (65504.0, 0x7BFF), (65520.0, 0x7C00),
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (3 * 2.0 ** -25, 0x0002),
    (1.0 + 2.0 ** -11, 0x3C00),            # tie, rounds to the even significand
    (1.0 + 3 * 2.0 ** -11, 0x3C02),        # tie, rounds up to even
    (float("inf"), 0x7C00), (-0.0, 0x8000),
])
def test_rne_closed_forms(x, bits):
    assert oracle.f64_to_f16(x) == bits


def test_nan_encodes_as_a_quiet_nan_like_numpy():
    # IEEE 754 arithmetic delivers quiet NaNs (top fraction bit set); the sign
    # is kept. numpy's conversion gives the same patterns.
    for x in (float("nan"), -float("nan")):
        bits = oracle.f64_to_f16(x)
        assert bits == int(_np_f16_bits(np.array([x]))[0])
        assert bits & 0x7E00 == 0x7E00 and (bits >> 15) == int(math.copysign(1, x) < 0)
