"""GPU parity of the continuous call with an E4M3 (FP8) cache against the
oracle. Q (FP16) follows the usual rule; every cache byte is either the
untouched 0x7F sentinel (bit-exact) or within one E4M3 ulp of the oracle's byte
(the GPU rounds its FP32 value, the oracle its double), never NaN."""
import numpy as np
import pytest

import workloads
from parity import compare, qout_rotated, to_dev, to_host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
NEOX, GPTJ = workloads.NEOX, workloads.GPTJ


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rope_kv_cache_gb300 import build
    build.build_library()


def _ordered8(b):
    b = b.astype(np.int32)
    mag = b & 0x7F
    return np.where(b & 0x80, -mag, mag)


def compare_e4m3(got, want, what):
    untouched = want == workloads.SENTINEL8
    assert np.array_equal(got[untouched], want[untouched]), f"{what}: untouched bytes changed"
    g, w = got[~untouched], want[~untouched]
    assert not np.any((g & 0x7F) == 0x7F), f"{what}: NaN written"
    d = np.abs(_ordered8(g) - _ordered8(w))
    assert d.max(initial=0) <= 1, f"{what}: {int((d > 1).sum())} bytes more than one ulp off"
    return {"n": int(g.size), "n_diff": int((d > 0).sum())}


def _run(case):
    import rope_kv_cache_gb300 as rk
    ks, vs = case.fp8_scales
    cache = torch.full(case.new_cache8().shape, workloads.SENTINEL8, dtype=torch.uint8,
                       device="cuda:0")
    qout = to_dev(case.new_qout())
    rk.rope_write_kv_continuous_fp8(to_dev(case.cos_sin), to_dev(case.end_lens), to_dev(case.qkv),
                                    cache, qout,
                                    torch.tensor([ks], dtype=torch.float32, device="cuda:0"),
                                    torch.tensor([vs], dtype=torch.float32, device="cuda:0"),
                                    case.Hq, case.Hkv, case.style)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), to_host_bits(qout)


def _oracle(case):
    import oracle
    cache = case.new_cache8()
    qout = case.new_qout()
    oracle.continuous_fp8(case.cos_sin, case.end_lens, case.qkv, cache, qout, *case.fp8_scales,
                          case.Hq, case.Hkv, case.style)
    return cache, qout


CASES = [
    # B, S, Hq, Hkv, D, r, cap, style, k_scale, v_scale
    (3, 37, 8, 2, 128, 128, 128, NEOX, 1.0, 1.0),
    (2, 19, 4, 4, 128, 64, 64, GPTJ, 0.05, 0.04),
    (2, 50, 6, 3, 64, 32, 96, NEOX, 0.005, 2.0),      # K x 200: saturates at +-448
    (2, 9, 8, 1, 256, 256, 40, NEOX, 0.5, 0.25),
    (2, 700, 4, 1, 64, 64, 1024, GPTJ, 0.1, 0.1),     # two items per thread
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_small_cases(idx):
    B, S, Hq, Hkv, D, r, cap, style, ks, vs = CASES[idx]
    case = workloads.make_continuous(B, S, Hq, Hkv, D, r, cap, style, 1e4, seed=700 + idx,
                                     name=f"fp8_{idx}")
    case.fp8_scales = (ks, vs)
    g_cache, g_q = _run(case)
    o_cache, o_q = _oracle(case)
    compare(g_q, o_q, qout_rotated(o_q.shape, r), f"{case.name} qOut")
    compare_e4m3(g_cache, o_cache, f"{case.name} cache")
    if ks == 0.005:
        assert np.isin(o_cache[:, 0], [0x7E, 0xFE]).any()   # the case does saturate


@pytest.mark.parametrize("tokens", [1, 153, 700, 1023, 1024, 1025])
def test_small_launch_residency_caps(tokens):
    """Decode-sized FP8 launches (two CTAs per token): 1 and 3 CTAs per SM,
    700 tokens, 1400 CTAs, past the 8-per-SM limit above which no shared
    memory is reserved, and both sides of the 1024-token switch to the larger
    launch's shape and policy."""
    case = workloads.make_continuous(tokens, 1, 8, 2, 128, 128, 16, NEOX, 5e5, seed=800 + tokens,
                                     name=f"fp8_caps{tokens}")
    case.fp8_scales = (0.05, 0.04)
    g_cache, g_q = _run(case)
    o_cache, o_q = _oracle(case)
    compare(g_q, o_q, qout_rotated(o_q.shape, 128), f"{case.name} qOut")
    compare_e4m3(g_cache, o_cache, f"{case.name} cache")


def test_skips_and_saturation():
    case = workloads.make_continuous(4, 6, 4, 2, 128, 128, 32, NEOX, 5e5, seed=21,
                                     end_lens=[3, 35, 32, 20], cs_seq=30, name="fp8_skips")
    case.fp8_scales = (0.002, 0.003)      # |x| > ~0.9 saturates to 448
    g_cache, g_q = _run(case)
    o_cache, o_q = _oracle(case)
    assert np.any((o_cache & 0x7F) == 0x7E)
    compare(g_q, o_q, qout_rotated(o_q.shape, 128), "fp8_skips qOut")
    compare_e4m3(g_cache, o_cache, "fp8_skips cache")


@pytest.mark.parametrize("name", ["prefill_fp8", "decode_fp8"])
def test_configs_full(name):
    case = workloads.config(name)
    if name == "decode_fp8":
        case.cap = 1024
        case.end_lens = (case.end_lens % 1024 + 1).astype(np.int32)
        case.cos_sin = np.ascontiguousarray(case.cos_sin[:, :1024])
    g_cache, g_q = _run(case)
    o_cache, o_q = _oracle(case)
    compare(g_q, o_q, qout_rotated(o_q.shape, case.r), f"{name} qOut")
    stats = compare_e4m3(g_cache, o_cache, f"{name} cache")
    assert stats["n_diff"] <= stats["n"] // 100


def test_large_launch_of_one_token_sequences():
    """1536 one-token sequences: an FP8 decode batch large enough for the
    large-launch path."""
    case = workloads.make_continuous(1536, 1, 8, 2, 128, 128, 16, NEOX, 5e5, seed=810,
                                     name="fp8_one_token_large")
    case.fp8_scales = (0.05, 0.04)
    g_cache, g_q = _run(case)
    o_cache, o_q = _oracle(case)
    compare(g_q, o_q, qout_rotated(o_q.shape, 128), f"{case.name} qOut")
    compare_e4m3(g_cache, o_cache, f"{case.name} cache")
