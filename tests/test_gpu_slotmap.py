"""GPU parity of the sglang-style slot-mapping call against the oracle: Q, K, V
as token-strided views of one packed buffer (and as separate tensors), every
head dim, both pairings, negative / out-of-range slots, positions outside the
table, with and without kOut; the two benchmark workloads at full size."""
import numpy as np
import pytest

import workloads
from parity import compare, dev_sentinel, to_dev, to_host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
NEOX, GPTJ = workloads.NEOX, workloads.GPTJ


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rope_kv_cache_gb300 import build
    build.build_library()


def _rot_mask(D, r, plane_k):
    return (np.arange(D) < r)[None, None, None, :] if plane_k else np.zeros((1, 1, 1, D), bool)


def _run(case, with_kout, separate=False):
    import rope_kv_cache_gb300 as rk
    qkv = to_dev(case.qkv)
    Hq, Hkv = case.Hq, case.Hkv
    if separate:
        q = qkv[:, :Hq].contiguous()
        k = qkv[:, Hq:Hq + Hkv].contiguous()
        v = qkv[:, Hq + Hkv:].contiguous()
    else:
        q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    kc = dev_sentinel(case.cache_shape())
    vc = dev_sentinel(case.cache_shape())
    qo = dev_sentinel((case.T, Hq, case.D))
    ko = dev_sentinel((case.T, Hkv, case.D)) if with_kout else None
    rk.rope_write_kv_slot_mapping(to_dev(case.cos_sin), to_dev(case.positions), q, k, v,
                                  to_dev(case.slots), kc, vc, qo, ko, style=case.style)
    torch.cuda.synchronize()
    return kc, vc, qo, ko


def _oracle(case, with_kout):
    import oracle
    kc = workloads.sentinel_fill(case.cache_shape())
    vc = workloads.sentinel_fill(case.cache_shape())
    qo = workloads.sentinel_fill((case.T, case.Hq, case.D))
    ko = workloads.sentinel_fill((case.T, case.Hkv, case.D)) if with_kout else None
    oracle.slot_mapping(case.cos_sin, case.positions, case.q, case.k, case.v, case.slots, kc, vc,
                        qo, ko, case.style)
    return kc, vc, qo, ko


SMALL = [
    # seq_lens, Hq, Hkv, D, r, style, block_size, num_blocks, with_kout, separate
    ([5, 17, 1, 40], 8, 2, 128, 128, NEOX, 16, 12, True, False),
    ([33, 9], 4, 4, 64, 32, GPTJ, 8, 12, False, False),
    ([7, 7, 7], 16, 1, 256, 128, NEOX, 4, 20, True, True),
    ([600, 500], 4, 2, 128, 64, GPTJ, 64, 24, True, False),   # >= 1024 tokens
    ([3], 64, 64, 128, 128, NEOX, 2, 4, True, False),         # 192 heads
    ([1] * 153, 8, 2, 128, 128, NEOX, 4, 160, False, False),  # 153 one-token CTAs: 2 per SM
    ([1] * 700, 8, 2, 128, 128, GPTJ, 4, 704, True, False),   # 700: 5 per SM
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_small_cases(idx):
    lens, Hq, Hkv, D, r, style, bsz, nb, with_kout, separate = SMALL[idx]
    case = workloads.make_slotmap(lens, Hq, Hkv, D, r, style, 1e4, seed=400 + idx, block_size=bsz,
                                  num_blocks=nb, start_range=(0, 100), cs_rows=1024,
                                  name=f"slotmap{idx}")
    rng = workloads.rng_for(idx)
    T = case.T
    bad = rng.choice(T, size=max(1, T // 8), replace=False)
    case.slots[bad[: len(bad) // 2 + 1]] = -1                       # skipped KV writes
    case.slots[bad[len(bad) // 2 + 1:]] = nb * bsz + 3               # past the caches
    if T > 3:
        case.positions[rng.integers(0, T)] = 1024                    # past the table
        case.positions[rng.integers(0, T)] = -2
    g = [to_host_bits(x) if x is not None else None for x in _run(case, with_kout, separate)]
    o = _oracle(case, with_kout)
    compare(g[0], o[0], _rot_mask(D, r, True), "keyCache")
    compare(g[1], o[1], _rot_mask(D, r, False), "valueCache")
    compare(g[2], o[2], (np.arange(D) < r)[None, None, :], "qOut")
    if with_kout:
        compare(g[3], o[3], (np.arange(D) < r)[None, None, :], "kOut")


@pytest.mark.parametrize("name", ["slotmap_decode", "slotmap_prefill"])
def test_configs_full(name):
    case = workloads.config(name)
    kc, vc, qo, _ = _run(case, False)
    o_kc, o_vc, o_qo, _ = _oracle(case, False)
    D, r = case.D, case.r
    compare(to_host_bits(qo), o_qo, (np.arange(D) < r)[None, None, :], f"{name} qOut")
    slots = torch.as_tensor(case.slots, device=kc.device)
    gk = to_host_bits(kc.view(-1, case.Hkv, D)[slots])
    gv = to_host_bits(vc.view(-1, case.Hkv, D)[slots])
    ok = o_kc.reshape(-1, case.Hkv, D)[case.slots]
    ov = o_vc.reshape(-1, case.Hkv, D)[case.slots]
    compare(gk, ok, (np.arange(D) < r)[None, None, :], f"{name} keyCache rows")
    compare(gv, ov, np.zeros((1, 1, D), bool), f"{name} valueCache rows")
    sent = np.uint16(workloads.SENTINEL).view(np.int16).item()
    for cache in (kc, vc):
        n = int((cache.view(torch.int16) != sent).sum().item())
        assert n == case.T * case.Hkv * D


@pytest.mark.parametrize("idx", [5, 6])
def test_small_launches_with_residency_cap_off(idx):
    """The decode-sized slot-mapping launches give the same result with the
    residency cap switched off by the caller."""
    import rope_kv_cache_gb300 as rk
    prev = rk.ropekv_set_residency_cap(False)
    try:
        test_small_cases(idx)
    finally:
        rk.ropekv_set_residency_cap(prev)


@pytest.mark.parametrize("T", [37, 1500])
def test_three_different_token_strides(T):
    """q, k and v each with a token stride of its own: q a view of a row padded
    by three heads, k a plain tensor, v a view of a row padded by one head (and
    starting one head in), against the oracle on the same views."""
    import oracle
    import rope_kv_cache_gb300 as rk
    Hq, Hkv, D, r, bsz, nb = 8, 2, 128, 64, 16, (T + 15) // 16 + 2
    rng = workloads.rng_for(4242 + T)
    qbuf = workloads.fp16_normal(rng, (T, Hq + 3, D))
    kbuf = workloads.fp16_normal(rng, (T, Hkv, D))
    vbuf = workloads.fp16_normal(rng, (T, Hkv + 1, D))
    q, k, v = qbuf[:, :Hq], kbuf, vbuf[:, 1:]
    positions = rng.integers(0, 1024, size=T).astype(np.int64)
    slots = rng.permutation(nb * bsz)[:T].astype(np.int64)
    slots[::9] = -1
    cs = workloads.cos_sin_table(1e4, 1024, r)[0]
    dq, dk, dv = to_dev(qbuf), to_dev(kbuf), to_dev(vbuf)
    gq, gk, gv = dq[:, :Hq], dk, dv[:, 1:]
    assert len({gq.stride(0), gk.stride(0), gv.stride(0)}) == 3
    kc, vc = dev_sentinel((nb, bsz, Hkv, D)), dev_sentinel((nb, bsz, Hkv, D))
    qo, ko = dev_sentinel((T, Hq, D)), dev_sentinel((T, Hkv, D))
    rk.rope_write_kv_slot_mapping(to_dev(cs), to_dev(positions), gq, gk, gv, to_dev(slots), kc,
                                  vc, qo, ko, style=GPTJ)
    torch.cuda.synchronize()
    o_kc, o_vc = workloads.sentinel_fill((nb, bsz, Hkv, D)), workloads.sentinel_fill((nb, bsz, Hkv, D))
    o_qo, o_ko = workloads.sentinel_fill((T, Hq, D)), workloads.sentinel_fill((T, Hkv, D))
    oracle.slot_mapping(cs, positions, q, k, v, slots, o_kc, o_vc, o_qo, o_ko, GPTJ)
    compare(to_host_bits(kc), o_kc, _rot_mask(D, r, True), "keyCache")
    compare(to_host_bits(vc), o_vc, _rot_mask(D, r, False), "valueCache")
    compare(to_host_bits(qo), o_qo, (np.arange(D) < r)[None, None, :], "qOut")
    compare(to_host_bits(ko), o_ko, (np.arange(D) < r)[None, None, :], "kOut")


@pytest.mark.parametrize("tokens", [1023, 1024, 1025])
def test_launch_policy_boundary(tokens):
    """One-token sequences on both sides of the 1024-token switch from the
    decode-sized launch (prologue and residency cap) to the larger one
    (prologue, no cap), with skipped slots and positions on each side."""
    case = workloads.make_slotmap([1] * tokens, 8, 2, 128, 128, NEOX, 5e5, seed=600 + tokens,
                                  block_size=4, num_blocks=tokens + 8,
                                  start_range=(0, 1023), cs_rows=1024, name=f"smedge{tokens}")
    rng = workloads.rng_for(tokens)
    case.slots[rng.choice(tokens, size=9, replace=False)] = -1
    case.positions[rng.choice(tokens, size=5, replace=False)] = 1024
    g = [to_host_bits(x) if x is not None else None for x in _run(case, True)]
    o = _oracle(case, True)
    D, r = case.D, case.r
    compare(g[0], o[0], _rot_mask(D, r, True), "keyCache")
    compare(g[1], o[1], _rot_mask(D, r, False), "valueCache")
    compare(g[2], o[2], (np.arange(D) < r)[None, None, :], "qOut")
    compare(g[3], o[3], (np.arange(D) < r)[None, None, :], "kOut")
