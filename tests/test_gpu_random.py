"""Seeded random sweep of GPU parity against the oracle: for each seed a random
entry point, pairing, head dim, rotary dim, GQA ratio, batch, sequence length
(ragged tails, several CTAs, one or two items per thread) and cache capacity,
including tokens whose slots or positions fall outside the cache or table."""
import numpy as np
import pytest

import workloads
from parity import check_contiguous

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rope_kv_cache_gb300 import build
    build.build_library()


def _random_case(seed):
    rng = np.random.Generator(np.random.PCG64(10_000 + seed))
    mode = ["continuous", "tree", "packed", "qknorm"][seed % 4]
    style = int(rng.integers(0, 2))
    D = int(rng.choice([64, 128, 256]))
    r = int(rng.choice([x for x in (16, 32, 48, 64, 96, 128, 256) if x <= D]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    Hq = Hkv * int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 5))
    S = int(rng.choice([1, 2, 7, 33, 129, int(rng.integers(1, 700))]))
    cap = S + int(rng.integers(0, 200))
    theta = float(rng.choice([1e4, 5e5]))
    cs_batch = int(rng.choice([1, B]))
    name = f"rand{seed}_{mode}"
    if mode == "packed":
        return workloads.make_packed(B, S, Hq, Hkv, D, r, cap, style, theta, seed, cs_batch=cs_batch,
                                     cache_init="sentinel", name=name)
    if mode == "tree":
        return workloads.make_tree(B, S, Hq, Hkv, D, r, cap, style, theta, seed,
                                   base_range=(0, cap - S), cs_batch=cs_batch, name=name)
    # continuous (and normalized): end lengths may push a few slots out of range
    end = rng.integers(S - 3, cap + 4, size=B).astype(np.int32)
    case = workloads.make_continuous(B, S, Hq, Hkv, D, r, cap, style, theta, seed, end_lens=end,
                                     cs_batch=cs_batch, name=name)
    if mode == "qknorm":
        case.norm = workloads.norm_weights(seed, D, eps=float(rng.choice([0.0, 1e-6, 1e-3])))
    return case


@pytest.mark.parametrize("seed", range(40))
def test_random_contiguous(seed):
    check_contiguous(_random_case(seed))
