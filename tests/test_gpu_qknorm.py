"""GPU parity of the continuous call with pre-RoPE QK RMS normalization,
against the oracle: every head dim, both pairings, partial rotary, several eps,
skipped tokens, and the prefill and decode workloads at full size."""
import numpy as np
import pytest

import workloads
from parity import check_contiguous

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
NEOX, GPTJ = workloads.NEOX, workloads.GPTJ


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rope_kv_cache_gb300 import build
    build.build_library()


CASES = [
    # B, S, Hq, Hkv, D, r, cap, style, eps
    (3, 37, 8, 2, 128, 128, 128, NEOX, 1e-6),
    (2, 19, 4, 4, 128, 64, 64, GPTJ, 1e-5),
    (2, 50, 6, 3, 64, 32, 96, NEOX, 0.0),
    (2, 9, 8, 1, 256, 256, 40, NEOX, 1e-6),
    (1, 33, 16, 8, 256, 128, 64, GPTJ, 0.1),
    (2, 700, 4, 1, 64, 64, 1024, NEOX, 1e-6),     # >= 1024 tokens: two items per thread
    (1, 3, 64, 64, 128, 128, 8, GPTJ, 1e-6),      # several CTAs per token
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_small_cases(idx):
    B, S, Hq, Hkv, D, r, cap, style, eps = CASES[idx]
    case = workloads.make_continuous(B, S, Hq, Hkv, D, r, cap, style, 1e4, seed=500 + idx,
                                     name=f"qknorm{idx}")
    qw, kw, _ = workloads.norm_weights(600 + idx, D)
    case.norm = (qw, kw, eps)
    check_contiguous(case)


def test_scaled_inputs_and_skips():
    case = workloads.make_continuous(4, 6, 4, 2, 128, 128, 32, NEOX, 5e5, seed=21,
                                     end_lens=[3, 35, 32, 20], cs_seq=30, name="qknorm_skips")
    # very small and very large heads: the normalization brings both back
    q = case.qkv.view(np.float16).astype(np.float32)
    q[0] *= 1e-3
    q[1] *= 50.0
    case.qkv = np.ascontiguousarray(q.astype(np.float16).view(np.uint16))
    case.norm = workloads.norm_weights(9, 128)
    check_contiguous(case)


@pytest.mark.parametrize("name", ["prefill_qknorm", "decode_qknorm"])
def test_configs_full(name):
    case = workloads.config(name)
    if name == "decode_qknorm":
        # the decode cache is 8.6 GB: check the same tokens on a 1024-slot cache
        case.cap = 1024
        case.end_lens = (case.end_lens % 1024 + 1).astype(np.int32)
        case.cos_sin = np.ascontiguousarray(case.cos_sin[:, :1024])
    stats = check_contiguous(case)
    assert stats["qout"]["max_ulp"] <= 1 and stats["cache"]["max_ulp"] <= 1
