"""Pins for the oracle's FP8 (OCP E4M3, "e4m3fn") conversions and the
FP8-cache variant of the continuous call (sglang rope_cache.py, Stage 3.3:
K and V scaled by 1/k_scale, 1/v_scale before the FP8 cache store).

Decoding is checked against the closed form and against torch's float8_e4m3fn
(an independent library routine); encoding against torch on in-range values
and by hand on saturation (the FP8 store saturates to the largest finite
value, 448, rather than producing NaN).
"""
import math

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")


def _closed_form(b):
    s = -1.0 if b & 0x80 else 1.0
    e = (b >> 3) & 0xF
    f = b & 7
    if e == 15 and f == 7:
        return math.nan
    return s * (f * 2.0 ** -9 if e == 0 else (8 + f) * 2.0 ** (e - 10))


def test_decode_all_patterns():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        ours = oracle.e4m3_to_f64(b)
        want = _closed_form(b)
        if math.isnan(want):
            assert math.isnan(ours) and math.isnan(t[b])
        else:
            assert ours == want == t[b]


def test_round_trip_all_finite_patterns():
    for b in range(256):
        v = oracle.e4m3_to_f64(b)
        if not math.isnan(v):
            assert oracle.f64_to_e4m3(v) == b


def test_rne_matches_torch_in_range():
    rng = np.random.Generator(np.random.PCG64(5))
    finite = np.array([oracle.e4m3_to_f64(b) for b in range(0x7F)])
    mids = (finite[:-1] + finite[1:]) / 2                      # exact ties
    x = np.concatenate([mids, mids * (1 + 1e-6), mids * (1 - 1e-6),
                        rng.uniform(-447.9, 447.9, 20000),
                        np.ldexp(rng.random(5000), rng.integers(-12, 8, 5000))])
    x = np.concatenate([x, -x])
    # float32-representable inputs: torch converts a double to FP8 through
    # float32, so only those see one rounding on both sides
    x = x.astype(np.float32).astype(np.float64)
    x = x[np.abs(x) < 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.f64_to_e4m3(v) for v in x], dtype=np.uint8)
    bad = np.nonzero(ours != want)[0]
    assert bad.size == 0, (x[bad[0]], ours[bad[0]], want[bad[0]])


@pytest.mark.parametrize("x,bits", [
    (448.0, 0x7E), (449.0, 0x7E), (463.99, 0x7E), (464.0, 0x7E), (1e6, 0x7E),
    (float("inf"), 0x7E), (-500.0, 0xFE), (float("-inf"), 0xFE),
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (2.0 ** -6, 0x08),
    (1.0, 0x38), (1.0625, 0x38), (1.1875, 0x3A), (-0.0, 0x80),
])
def test_encode_closed_forms(x, bits):
    assert oracle.f64_to_e4m3(x) == bits
    assert oracle.f64_to_e4m3(float("nan")) == 0x7F


def _e4m3_of_f16(bits16, scale=1.0):
    v = bits16.view(np.float16).astype(np.float64) / scale
    return np.array([oracle.f64_to_e4m3(x) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_fp8_cache_is_the_fp16_result_converted(style):
    """With identity cos/sin rows and inputs that E4M3 holds exactly, the FP8
    cache must be the FP16 call's cache converted element by element; a
    power-of-two scale divides exactly."""
    rng = workloads.rng_for(6)
    B, S, Hq, Hkv, D, r, cap = 2, 4, 4, 2, 64, 64, 8
    vals = rng.integers(-15, 16, size=(B, S, Hq + 2 * Hkv, D)).astype(np.float64) / 4
    qkv = vals.astype(np.float16).view(np.uint16)
    cs = np.zeros((1, cap, r), dtype=np.float32)
    cs[..., : r // 2] = 1.0
    end = np.array([4, 8], dtype=np.int32)
    c16 = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    q16 = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(cs, end, qkv, c16, q16, Hq, Hkv, style)
    for ks, vs in ((1.0, 1.0), (2.0, 0.5)):
        c8 = np.full((B, 2, Hkv, cap, D), 0x7F, dtype=np.uint8)
        q8 = workloads.sentinel_fill((B, S, Hq, D))
        oracle.continuous_fp8(cs, end, qkv, c8, q8, ks, vs, Hq, Hkv, style)
        assert np.array_equal(q8, q16)
        written = c16[:, 0, 0, :, 0] != workloads.SENTINEL            # [B, cap]
        for b in range(B):
            for slot in np.nonzero(written[b])[0]:
                assert np.array_equal(c8[b, 0, :, slot], _e4m3_of_f16(c16[b, 0, :, slot], ks))
                assert np.array_equal(c8[b, 1, :, slot], _e4m3_of_f16(c16[b, 1, :, slot], vs))
        assert np.all(c8[~np.broadcast_to(written[:, None, None, :], (B, 2, Hkv, cap))] == 0x7F)


def test_fp8_cache_scaled_rotation_closed_form():
    # D = r = 16, one K head, position 1 of theta 1e4: K = (1, 0, ...) rotates
    # to (cos 1, 0.., sin 1, 0..) (NeoX); scaled by 1/0.25 then rounded to E4M3.
    D = r = 16
    qkv = np.zeros((1, 1, 3, D), dtype=np.float16)
    qkv[0, 0, 1, 0] = 1.0
    cs = workloads.cos_sin_table(1e4, 2, r)
    c8 = np.zeros((1, 2, 1, 2, D), dtype=np.uint8)
    q8 = workloads.sentinel_fill((1, 1, 1, D))
    oracle.continuous_fp8(cs, np.array([2], dtype=np.int32), qkv.view(np.uint16), c8, q8, 0.25,
                          1.0, 1, 1, oracle.NEOX)
    c1, s1 = float(cs[0, 1, 0]), float(cs[0, 1, r // 2])
    assert c8[0, 0, 0, 1, 0] == oracle.f64_to_e4m3(c1 / 0.25)
    assert c8[0, 0, 0, 1, r // 2] == oracle.f64_to_e4m3(s1 / 0.25)
    assert abs(oracle.e4m3_to_f64(c8[0, 0, 0, 1, 0]) - math.cos(1.0) * 4) <= 0.0625 * 2


def test_fp8_position_past_table_is_skipped():
    # slots and positions as the continuous call: position 5 of a 5-row table
    # has no cos/sin row, so that token writes neither qOut nor the FP8 cache
    B, S, Hq, Hkv, D, r, cap = 1, 3, 2, 1, 16, 16, 8
    qkv = np.full((B, S, 4, D), 0.5).astype(np.float16).view(np.uint16)
    big = np.zeros((1, 6, r), dtype=np.float32)
    big[0, :, : r // 2] = 1.0
    big[0, 5] = 2.0 ** 10                                 # one row past the table
    cs = big[:, :5]
    end = np.array([6], dtype=np.int32)                   # positions 3, 4, 5
    c8 = np.full((B, 2, Hkv, cap, D), 0x7F, dtype=np.uint8)
    q8 = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous_fp8(cs, end, qkv, c8, q8, 1.0, 1.0, Hq, Hkv, oracle.NEOX)
    assert np.all(q8[0, 2] == workloads.SENTINEL) and np.all(c8[0, :, 0, 5] == 0x7F)
    assert np.all(c8[0, :, 0, 3:5] == oracle.f64_to_e4m3(0.5))
    assert np.all(c8[0, :, 0, :3] == 0x7F) and np.all(c8[0, :, 0, 6:] == 0x7F)


def test_fp8_k_rounds_once_from_the_rotation():
    """sglang rope_cache.py Stage 3.2-3.4: the rotated K stays in the RoPE's
    working precision, is multiplied by 1 / k_scale and is rounded once, to the
    cache type; the FP16 rounding belongs only to the k_out/qOut copy. A row
    with cos = 1 + 2^-12 and sin = 0 turns 1.0625 (an E4M3 tie between 1.0 and
    1.125) into 1.0625 + 2^-12 * 1.0625: rounded directly that is 1.125
    (0x39); through FP16 it would first fall back to the tie 1.0625 and then to
    the even 1.0 (0x38)."""
    D = r = 16
    qkv = np.zeros((1, 1, 3, D), dtype=np.float16)
    qkv[0, 0, :2, 0] = 1.0625                              # the Q head and the K head
    cs = np.zeros((1, 1, r), dtype=np.float32)
    cs[0, 0, : r // 2] = np.float32(1.0 + 2.0 ** -12)
    c8 = np.zeros((1, 2, 1, 1, D), dtype=np.uint8)
    q8 = workloads.sentinel_fill((1, 1, 1, D))
    oracle.continuous_fp8(cs, np.array([1], dtype=np.int32), qkv.view(np.uint16), c8, q8, 1.0,
                          1.0, 1, 1, oracle.NEOX)
    assert c8[0, 0, 0, 0, 0] == 0x39
    assert q8[0, 0, 0, 0] == 0x3C40                        # FP16 1.0625
    assert oracle.f64_to_e4m3(1.0625) == 0x38              # the tie alone goes to even


def test_fp8_scale_covers_the_whole_k_head():
    """Stage 3.3 scales the whole K head vector (the kernel's head block is the
    full head width) by 1 / k_scale, so with rotaryDim < headDim the dims past
    rotaryDim are scaled too. Position 0 (identity row), k_scale 0.5: every K
    element e becomes E4M3(2e); V scales by 1 / v_scale = 4."""
    D, r = 32, 16
    qkv = np.zeros((1, 1, 3, D))
    qkv[0, 0, 1] = 1.0 + np.arange(D) / 16.0          # K head, exact in FP16
    qkv[0, 0, 2] = 0.25
    qkv = qkv.astype(np.float16).view(np.uint16)
    cs = np.zeros((1, 1, r), dtype=np.float32)
    cs[0, 0, : r // 2] = 1.0
    c8 = np.zeros((1, 2, 1, 1, D), dtype=np.uint8)
    q8 = workloads.sentinel_fill((1, 1, 1, D))
    oracle.continuous_fp8(cs, np.array([1], dtype=np.int32), qkv, c8, q8, 0.5, 0.25, 1, 1,
                          oracle.NEOX)
    k = 1.0 + np.arange(D) / 16.0
    assert [int(b) for b in c8[0, 0, 0, 0]] == [oracle.f64_to_e4m3(2 * e) for e in k]
    assert np.all(c8[0, 1, 0, 0] == 0x38)              # 0.25 * 4 = 1.0
