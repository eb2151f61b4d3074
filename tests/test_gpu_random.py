"""Seeded random sweeps of GPU parity against the oracle.

Contiguous layouts (40 seeds): a random entry point, pairing, head dim, rotary
dim, GQA ratio, batch, sequence length (ragged tails, small and large launch
paths) and cache capacity, including tokens whose slots or positions fall
outside the cache or table. Paged updates (20 seeds) and fused DFlash updates
(20 seeds): random heads, dims, page size, pages per sequence, pool size,
padding and unmapped pages, cos/sin source rows and state indices. Slot
mapping (20 seeds): random sequence mixes, block sizes, strided or separate
Q/K/V, optional kOut, skipped slots and positions past the table. FP8 cache
(12 seeds): random shapes and K/V scales, some small enough to saturate."""
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


def _random_paged(seed):
    rng = np.random.Generator(np.random.PCG64(20_000 + seed))
    style = int(rng.integers(0, 2))
    D = int(rng.choice([64, 128, 256]))
    r = int(rng.choice([x for x in (16, 32, 64, 96, 128, 256) if x <= D]))
    Hkv = int(rng.choice([1, 2, 4, 8, 16]))
    B = int(rng.integers(1, 17))
    tpp = int(rng.choice([1, 4, 16, 64]))
    mpps = int(rng.integers(1, 65))
    max_len = min(256, tpp * mpps)
    N = int(rng.integers(1, max(2, int(B * max_len / 0.9))))
    N = min(N, 2500)
    valid = max(B, int(0.9 * N)) if N >= B else N
    valid = min(valid, B * max_len)
    N = max(N, valid)
    P = int(rng.integers(B * mpps, B * mpps + 64))  # no two logical pages share a page
    return workloads.make_paged(N, B, Hkv, D, r, tpp, mpps, P, style, 1e4, seed=20_000 + seed,
                                valid_rows=valid, len_range=(1, max_len),
                                unmapped_frac=float(rng.choice([0.0, 0.05, 0.3])),
                                name=f"rpaged{seed}")


@pytest.mark.parametrize("seed", range(20))
def test_random_paged(seed):
    import oracle
    import rope_kv_cache_gb300 as rk
    from parity import compare, dev_sentinel, pool_rotated, to_dev, to_host_bits
    pc = _random_paged(seed)
    pool = dev_sentinel(pc.pool_shape())
    rk.paged_kv_delta_update(to_dev(pc.k_delta), to_dev(pc.v_delta), pool,
                             to_dev(pc.cos_sin_rows), to_dev(pc.positions), to_dev(pc.seq_ids),
                             to_dev(pc.page_table), style=pc.style)
    torch.cuda.synchronize()
    want = pc.new_pool()
    oracle.paged(pc.k_delta, pc.v_delta, want, pc.cos_sin_rows, pc.positions, pc.seq_ids,
                 pc.page_table, pc.style)
    compare(to_host_bits(pool), want, pool_rotated(want.shape, pc.r), pc.name)


@pytest.mark.parametrize("seed", range(20))
def test_random_paged_fused(seed):
    import oracle
    import rope_kv_cache_gb300 as rk
    from parity import compare, dev_sentinel, pool_rotated, to_dev, to_host_bits
    rng = np.random.Generator(np.random.PCG64(30_000 + seed))
    style = int(rng.integers(0, 2))
    D = int(rng.choice([64, 128, 256]))
    r = int(rng.choice([x for x in (16, 32, 64, 128, 256) if x <= D]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 24))
    W = int(rng.integers(1, 80))
    tpp = int(rng.choice([4, 16, 64]))
    lo = max(1, -(-W // tpp))
    mpps = int(rng.integers(lo, lo + 12))
    P = int(rng.integers(B * mpps, B * mpps + 64))  # no two logical pages share a page
    rows = int(rng.integers(1, 4))
    st = bool(rng.integers(0, 2))
    cap = None if rng.integers(0, 2) else int(rng.integers(W, tpp * mpps + 1))
    fc = workloads.make_paged_fused(B, W, Hkv, D, r, tpp, mpps, P, style, 1e4, seed=30_000 + seed,
                                    len_range=(0, W + 2), unmapped_frac=0.05, source_rows=rows,
                                    with_state=st, cache_capacity=cap, name=f"rfused{seed}")
    pool = dev_sentinel(fc.pool_shape())
    rk.paged_kv_delta_update_fused(to_dev(fc.k_delta), to_dev(fc.v_delta), pool,
                                   to_dev(fc.source), to_dev(fc.old_lengths),
                                   to_dev(fc.delta_lengths), to_dev(fc.page_table),
                                   to_dev(fc.state) if fc.state is not None else None,
                                   style=fc.style)
    torch.cuda.synchronize()
    want = fc.new_pool()
    oracle.paged_fused(fc.k_delta, fc.v_delta, want, fc.source, fc.old_lengths, fc.delta_lengths,
                       fc.W, fc.state, fc.page_table, fc.style)
    compare(to_host_bits(pool), want, pool_rotated(want.shape, fc.r), fc.name)


@pytest.mark.parametrize("seed", range(20))
def test_random_slot_mapping(seed):
    """Random sglang-style calls: sequence mix, heads, dims, pairing, block size,
    token-strided or separate Q/K/V, with or without kOut, and some tokens with
    a negative slot, a slot past the caches or a position past the table."""
    import oracle
    import rope_kv_cache_gb300 as rk
    from parity import compare, dev_sentinel, to_dev, to_host_bits
    rng = np.random.Generator(np.random.PCG64(40_000 + seed))
    style = int(rng.integers(0, 2))
    D = int(rng.choice([64, 128, 256]))
    r = int(rng.choice([x for x in (16, 32, 64, 128, 256) if x <= D]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    Hq = Hkv * int(rng.choice([1, 2, 4, 8]))
    lens = [int(x) for x in rng.integers(1, int(rng.choice([2, 40, 700])), size=int(rng.integers(1, 6)))]
    bsz = int(rng.choice([1, 4, 16, 64]))
    nb = sum(-(-(n + bsz) // bsz) for n in lens) + int(rng.integers(0, 8))
    case = workloads.make_slotmap(lens, Hq, Hkv, D, r, style, 1e4, seed=40_000 + seed,
                                  block_size=bsz, num_blocks=nb, start_range=(0, 300),
                                  cs_rows=1024, name=f"rslot{seed}")
    T = case.T
    bad = rng.choice(T, size=max(1, T // 10), replace=False)
    case.slots[bad[: len(bad) // 2 + 1]] = -1
    case.slots[bad[len(bad) // 2 + 1:]] = nb * bsz + int(rng.integers(0, 5))
    if T > 2:
        case.positions[int(rng.integers(0, T))] = 1024 + int(rng.integers(0, 3))
    separate, with_kout = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    qkv = to_dev(case.qkv)
    q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    if separate:
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    kc, vc = dev_sentinel(case.cache_shape()), dev_sentinel(case.cache_shape())
    qo = dev_sentinel((T, Hq, D))
    ko = dev_sentinel((T, Hkv, D)) if with_kout else None
    rk.rope_write_kv_slot_mapping(to_dev(case.cos_sin), to_dev(case.positions), q, k, v,
                                  to_dev(case.slots), kc, vc, qo, ko, style=case.style)
    torch.cuda.synchronize()
    w = [workloads.sentinel_fill(case.cache_shape()), workloads.sentinel_fill(case.cache_shape()),
         workloads.sentinel_fill((T, Hq, D)),
         workloads.sentinel_fill((T, Hkv, D)) if with_kout else None]
    oracle.slot_mapping(case.cos_sin, case.positions, case.q, case.k, case.v, case.slots,
                        w[0], w[1], w[2], w[3], case.style)
    rot = (np.arange(D) < r)
    compare(to_host_bits(kc), w[0], rot[None, None, None, :], f"{case.name} keyCache")
    compare(to_host_bits(vc), w[1], np.zeros((1, 1, 1, D), bool), f"{case.name} valueCache")
    compare(to_host_bits(qo), w[2], rot[None, None, :], f"{case.name} qOut")
    if with_kout:
        compare(to_host_bits(ko), w[3], rot[None, None, :], f"{case.name} kOut")


@pytest.mark.parametrize("seed", range(12))
def test_random_fp8(seed):
    """Random continuous calls into an E4M3 cache: dims, pairing, heads,
    ragged lengths, out-of-cache slots and K/V scales from 1/64 to 4 (small
    scales saturate)."""
    import oracle
    import rope_kv_cache_gb300 as rk
    from parity import compare, qout_rotated, to_dev, to_host_bits
    from test_gpu_fp8 import compare_e4m3
    rng = np.random.Generator(np.random.PCG64(50_000 + seed))
    style = int(rng.integers(0, 2))
    D = int(rng.choice([64, 128, 256]))
    r = int(rng.choice([x for x in (16, 32, 64, 128, 256) if x <= D]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 5))
    S = int(rng.choice([1, 3, 37, int(rng.integers(1, 600))]))
    cap = S + int(rng.integers(0, 100))
    end = rng.integers(S - 2, cap + 3, size=B).astype(np.int32)
    case = workloads.make_continuous(B, S, Hq, Hkv, D, r, cap, style, 1e4, seed=50_000 + seed,
                                     end_lens=end, name=f"rfp8_{seed}")
    case.fp8_scales = (float(2.0 ** rng.integers(-6, 3)) * float(rng.choice([1.0, 0.7])),
                       float(2.0 ** rng.integers(-6, 3)))
    cache = torch.full(case.new_cache8().shape, workloads.SENTINEL8, dtype=torch.uint8,
                       device="cuda:0")
    qout = to_dev(case.new_qout())
    ks, vs = case.fp8_scales
    rk.rope_write_kv_continuous_fp8(to_dev(case.cos_sin), to_dev(case.end_lens),
                                    to_dev(case.qkv), cache, qout,
                                    torch.tensor([ks], dtype=torch.float32, device="cuda:0"),
                                    torch.tensor([vs], dtype=torch.float32, device="cuda:0"),
                                    Hq, Hkv, style)
    torch.cuda.synchronize()
    w_cache = case.new_cache8()
    w_q = case.new_qout()
    oracle.continuous_fp8(case.cos_sin, case.end_lens, case.qkv, w_cache, w_q, ks, vs, Hq, Hkv,
                          style)
    compare(to_host_bits(qout), w_q, qout_rotated(w_q.shape, r), f"{case.name} qOut")
    compare_e4m3(cache.cpu().numpy(), w_cache, f"{case.name} cache")
