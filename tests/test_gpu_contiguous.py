"""GPU parity of the contiguous-cache entry points against the oracle.

Small seeded cases (several tiles, ragged tails, every head dim, partial
rotary, MHA/GQA/MQA, skipped tokens, per-sequence tables) are compared on every
output element. The benchmark workloads run at full size in the launch shape
the benchmark times: packed_tiny and prefill on every element; decode and tree
on every written slot plus a device-side count proving nothing else changed.
"""
import numpy as np
import pytest

import workloads
from parity import (cache_rotated, check_contiguous, compare, dev_sentinel, qout_rotated,
                    to_dev, to_host_bits)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
NEOX, GPTJ = workloads.NEOX, workloads.GPTJ


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rope_kv_cache_gb300 import build
    build.build_library()


SMALL = [
    # mode, style, D, r, Hq, Hkv, B, S, cap
    ("continuous", NEOX, 128, 128, 8, 2, 3, 37, 128),
    ("continuous", GPTJ, 128, 64, 4, 4, 2, 19, 64),
    ("continuous", NEOX, 64, 32, 6, 3, 2, 50, 96),
    ("continuous", NEOX, 256, 256, 8, 1, 2, 9, 40),
    ("continuous", GPTJ, 256, 128, 16, 8, 1, 33, 64),
    ("continuous", NEOX, 128, 16, 4, 2, 2, 5, 8),
    ("continuous", NEOX, 64, 64, 4, 1, 2, 700, 1024),   # >= 1024 tokens: two items per thread
    ("continuous", GPTJ, 128, 128, 64, 64, 1, 3, 8),    # 192 heads: several CTAs per token
    ("tree", NEOX, 128, 128, 32, 8, 3, 20, 64),
    ("tree", GPTJ, 64, 64, 4, 2, 4, 11, 32),
    ("tree", GPTJ, 128, 64, 32, 8, 2, 64, 256),
    ("packed", NEOX, 128, 128, 8, 2, 2, 40, 64),
    ("packed", GPTJ, 64, 48, 4, 1, 1, 7, 8),
    ("packed", NEOX, 256, 96, 4, 2, 3, 13, 13),
    ("packed", GPTJ, 128, 128, 32, 8, 1, 1100, 1100),
]


def _small_case(mode, style, D, r, Hq, Hkv, B, S, cap, seed, cs_batch=1):
    theta = 1e4 if style == GPTJ else 5e5
    if mode == "continuous":
        return workloads.make_continuous(B, S, Hq, Hkv, D, r, cap, style, theta, seed,
                                         cs_batch=cs_batch, name=f"cont{seed}")
    if mode == "tree":
        return workloads.make_tree(B, S, Hq, Hkv, D, r, cap, style, theta, seed,
                                   base_range=(0, cap - S), cs_batch=cs_batch, name=f"tree{seed}")
    return workloads.make_packed(B, S, Hq, Hkv, D, r, cap, style, theta, seed, cs_batch=cs_batch,
                                 cache_init="sentinel", name=f"packed{seed}")


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_small_cases(idx):
    case = _small_case(*SMALL[idx], seed=100 + idx)
    check_contiguous(case)


@pytest.mark.parametrize("mode", ["continuous", "tree", "packed"])
def test_per_sequence_tables(mode):
    case = _small_case(mode, NEOX, 128, 128, 8, 2, 3, 17, 64, seed=7, cs_batch=3)
    check_contiguous(case)


def test_skipped_tokens_continuous():
    # slots below 0, at/after the capacity, and past a short table are skipped
    B, S, Hq, Hkv, D, r, cap = 4, 6, 4, 2, 128, 128, 32
    case = workloads.make_continuous(B, S, Hq, Hkv, D, r, cap, NEOX, 5e5, seed=21,
                                     end_lens=[3, 35, 32, 20], cs_seq=30, name="skips")
    check_contiguous(case)


def test_skipped_tokens_tree():
    case = workloads.make_tree(3, 16, 8, 2, 128, 64, 64, GPTJ, 1e4, seed=22, base_range=(0, 40),
                               cs_seq=44, name="tree_skips")
    case.pos_ids[0, 3] = -1
    case.pos_ids[1, 5] = -7
    case.pos_ids[2, 0] = 44          # == cosSinSeqLen: skipped
    case.end_lens[2] = 70            # last slots past the capacity
    check_contiguous(case)


def test_empty_inputs_are_no_ops():
    import rope_kv_cache_gb300 as rk
    for B, S in ((0, 5), (3, 0)):
        case = workloads.make_continuous(B, S, 4, 2, 64, 64, 16, NEOX, 1e4, seed=3,
                                         end_lens=np.full(B, S, dtype=np.int32))
        cache = to_dev(case.new_cache())
        qout = to_dev(case.new_qout())
        rk.rope_write_kv_continuous(to_dev(case.cos_sin), to_dev(case.end_lens), to_dev(case.qkv),
                                    cache, qout, 4, 2, NEOX)
        torch.cuda.synchronize()
        assert np.all(to_host_bits(cache) == workloads.SENTINEL)


def test_non_default_stream_and_repeat():
    case = _small_case("continuous", NEOX, 128, 128, 8, 2, 2, 33, 64, seed=5)
    s = torch.cuda.Stream()
    first = check_contiguous(case, stream=s)
    second = check_contiguous(case, stream=s)
    assert first == second


# ---------------------------------------------------------- full configs --

def test_config_packed_tiny():
    case = workloads.config("packed_tiny")
    check_contiguous(case)


def test_config_prefill_full():
    case = workloads.config("prefill")
    stats = check_contiguous(case)
    assert stats["qout"]["max_ulp"] <= 1 and stats["cache"]["max_ulp"] <= 1


def _count_not_sentinel(cache_t) -> int:
    n = 0
    v = cache_t.view(torch.int16)
    sent = np.uint16(workloads.SENTINEL).view(np.int16).item()
    for b in range(v.shape[0]):
        n += int((v[b] != sent).sum().item())
    return n


def _per_sequence_oracle(case, b):
    """Oracle for sequence b alone (sequences are independent)."""
    import oracle
    sub_qkv = np.ascontiguousarray(case.qkv[b:b + 1])
    cs = case.cos_sin if case.cos_sin.shape[0] == 1 else np.ascontiguousarray(case.cos_sin[b:b + 1])
    cache = workloads.sentinel_fill((1, 2, case.Hkv, case.cap, case.D))
    qout = workloads.sentinel_fill((1, case.S, case.Hq, case.D))
    end = np.ascontiguousarray(case.end_lens[b:b + 1])
    if case.mode == "tree":
        oracle.tree(cs, end, np.ascontiguousarray(case.pos_ids[b:b + 1]), sub_qkv, cache, qout,
                    case.Hq, case.Hkv, case.style)
    else:
        oracle.continuous(cs, end, sub_qkv, cache, qout, case.Hq, case.Hkv, case.style)
    return cache[0], qout[0]


@pytest.mark.parametrize("name", ["decode", "tree"])
def test_config_written_slots_and_untouched(name):
    import rope_kv_cache_gb300 as rk
    case = workloads.config(name)
    cs = to_dev(case.cos_sin)
    qkv = to_dev(case.qkv)
    end = to_dev(case.end_lens)
    cache = dev_sentinel((case.B, 2, case.Hkv, case.cap, case.D))
    qout = dev_sentinel((case.B, case.S, case.Hq, case.D))
    if case.mode == "tree":
        rk.rope_write_kv_tree(cs, end, to_dev(case.pos_ids), qkv, cache, qout, case.Hq, case.Hkv,
                              case.style)
    else:
        rk.rope_write_kv_continuous(cs, end, qkv, cache, qout, case.Hq, case.Hkv, case.style)
    torch.cuda.synchronize()
    g_qout = to_host_bits(qout)
    written = 0
    for b in range(case.B):
        o_cache, o_qout = _per_sequence_oracle(case, b)
        compare(g_qout[b], o_qout, qout_rotated((1,) + o_qout.shape, case.r)[0], f"{name} qOut b={b}")
        slots = np.arange(case.S) + int(case.end_lens[b]) - case.S
        slots = slots[(slots >= 0) & (slots < case.cap)]
        g_rows = to_host_bits(cache[b][:, :, torch.as_tensor(slots, device=cache.device), :])
        o_rows = np.ascontiguousarray(o_cache[:, :, slots, :])
        compare(g_rows, o_rows, cache_rotated((1,) + o_rows.shape, case.r)[0], f"{name} cache b={b}")
        written += len(slots) * 2 * case.Hkv * case.D
    assert _count_not_sentinel(cache) == written


@pytest.mark.parametrize("B,S", [(2, 7), (3, 600)])
def test_dependent_back_to_back_calls(B, S):
    """Each call consumes the previous call's in-place output. Small launches
    are dependent launches that prefetch before waiting on the previous grid,
    large ones are plain launches; either way every call must see the previous
    result. Three calls issued back to back, and replayed from a CUDA graph,
    must give the bytes of three calls separated by host synchronisation."""
    import rope_kv_cache_gb300 as rk
    case = workloads.make_packed(B, S, 8, 2, 128, 128, 1024, NEOX, 1e4, seed=33,
                                 cache_init="sentinel")
    cs = to_dev(case.cos_sin)

    def run(mode):
        qkv = to_dev(case.qkv)
        cache = to_dev(case.new_cache())
        if mode == "graph":
            s = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(3):
                    rk.rope_write_kv_packed(cs, qkv, cache, case.Hq, case.Hkv, case.style,
                                            stream=torch.cuda.current_stream())
            qkv.copy_(to_dev(case.qkv))
            cache.copy_(to_dev(case.new_cache()))
            torch.cuda.synchronize()
            g.replay()
        else:
            for _ in range(3):
                rk.rope_write_kv_packed(cs, qkv, cache, case.Hq, case.Hkv, case.style)
                if mode == "synced":
                    torch.cuda.synchronize()
        torch.cuda.synchronize()
        return to_host_bits(qkv), to_host_bits(cache)

    ref_qkv, ref_cache = run("synced")
    assert not np.array_equal(ref_qkv, case.qkv)
    for mode in ("back_to_back", "graph"):
        q, c = run(mode)
        assert np.array_equal(q, ref_qkv), mode
        assert np.array_equal(c, ref_cache), mode


@pytest.mark.parametrize("tokens", [1, 152, 153, 450, 608, 609, 1000, 1023])
@pytest.mark.parametrize("norm", [False, True])
@pytest.mark.parametrize("cap_on", [True, False])
def test_small_launch_residency_caps(tokens, norm, cap_on):
    """Decode-sized launches (fewer than 1024 tokens; two CTAs per token of
    8 + 2 x 2 heads here) reserve dynamic shared memory so that at most
    ceil(CTAs / SMs) CTAs share an SM: 1, 2, 3, 6 and 8 CTAs per SM here, and
    609 tokens and more cross the 8-per-SM limit above which no memory is
    reserved. Every cap, and the cap switched off by the caller, gives the
    oracle's result."""
    import rope_kv_cache_gb300 as rk
    case = workloads.make_continuous(tokens, 1, 8, 2, 128, 128, 16, NEOX, 5e5, seed=4000 + tokens,
                                     name=f"caps{tokens}")
    if norm:
        case.norm = workloads.norm_weights(4000 + tokens, 128)
    prev = rk.ropekv_set_residency_cap(cap_on)
    try:
        check_contiguous(case)
    finally:
        rk.ropekv_set_residency_cap(prev)


def test_tensors_on_a_non_current_device():
    """The binding makes the tensors' device current for the call: a call
    whose tensors live on cuda:1 while cuda:0 is current gives the oracle's
    result (and sets up the residency cap on cuda:1)."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two CUDA devices")
    case = workloads.make_continuous(64, 1, 8, 2, 128, 128, 16, NEOX, 5e5, seed=77,
                                     name="device1")
    from parity import on_device
    with on_device(torch.device("cuda:1")), torch.cuda.device(0):
        check_contiguous(case)


@pytest.mark.parametrize("B,S", [(4, 1), (2, 600)])
def test_mixed_dependent_chain(B, S):
    """Four different entry points, each reading or overwriting what the one
    before it wrote, issued back to back and replayed from a CUDA graph, give
    the bytes of the same calls separated by host synchronisation: the packed
    call rotates qkv in place and fills cache slots 0..S-1; the continuous call
    reads that qkv, writes qOut and rewrites slots 5..S+4; the normalized call
    reads qkv again and rewrites those slots; the slot-mapping call takes the
    first qOut as its Q and the K/V heads of qkv as token-strided views.
    (4, 1) runs every call as a small dependent launch with the prefetch
    prologue and residency cap, (2, 600) as large ones."""
    import rope_kv_cache_gb300 as rk
    Hq, Hkv, D = 8, 2, 128
    H, T = Hq + 2 * Hkv, B * S
    case = workloads.make_packed(B, S, Hq, Hkv, D, 128, 1024, NEOX, 1e4, seed=77,
                                 cache_init="sentinel")
    cs = to_dev(case.cos_sin)
    end = torch.full((B,), S + 5, dtype=torch.int32, device="cuda:0")
    qw, kw, eps = workloads.norm_weights(77, D)
    qw, kw = to_dev(qw), to_dev(kw)
    positions = (torch.arange(T, device="cuda:0", dtype=torch.int64) * 7) % 1000
    slots = torch.arange(T, device="cuda:0", dtype=torch.int64).flip(0)
    sent = np.uint16(workloads.SENTINEL).view(np.int16).item()

    def run(mode):
        qkv = to_dev(case.qkv)
        cache = to_dev(case.new_cache())
        qout = torch.zeros((B, S, Hq, D), dtype=torch.float16, device="cuda:0")
        qout2 = torch.zeros_like(qout)
        kc = torch.full((T, 1, Hkv, D), sent, dtype=torch.int16, device="cuda:0").view(torch.float16)
        vc = kc.clone()
        qo3 = torch.zeros((T, Hq, D), dtype=torch.float16, device="cuda:0")

        def chain(stream):
            rk.rope_write_kv_packed(cs, qkv, cache, Hq, Hkv, NEOX, stream=stream)
            rk.rope_write_kv_continuous(cs, end, qkv, cache, qout, Hq, Hkv, NEOX, stream=stream)
            rk.rope_write_kv_continuous_qknorm(cs, end, qkv, cache, qout2, qw, kw, eps, Hq, Hkv,
                                               NEOX, stream=stream)
            flat = qkv.view(T, H, D)
            rk.rope_write_kv_slot_mapping(cs[0], positions, qout.view(T, Hq, D),
                                          flat[:, Hq:Hq + Hkv], flat[:, Hq + Hkv:], slots, kc, vc,
                                          qo3, style=NEOX, stream=stream)

        if mode == "graph":
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=torch.cuda.Stream()):
                chain(torch.cuda.current_stream())
            qkv.copy_(to_dev(case.qkv))
            cache.copy_(to_dev(case.new_cache()))
            for t in (qout, qout2, qo3):
                t.zero_()
            kc.view(torch.int16).fill_(sent)
            vc.view(torch.int16).fill_(sent)
            torch.cuda.synchronize()
            g.replay()
        elif mode == "synced":
            for step in range(4):
                # the same calls one at a time, each completed before the next
                calls = [
                    lambda: rk.rope_write_kv_packed(cs, qkv, cache, Hq, Hkv, NEOX),
                    lambda: rk.rope_write_kv_continuous(cs, end, qkv, cache, qout, Hq, Hkv, NEOX),
                    lambda: rk.rope_write_kv_continuous_qknorm(cs, end, qkv, cache, qout2, qw, kw,
                                                               eps, Hq, Hkv, NEOX),
                    lambda: rk.rope_write_kv_slot_mapping(
                        cs[0], positions, qout.view(T, Hq, D), qkv.view(T, H, D)[:, Hq:Hq + Hkv],
                        qkv.view(T, H, D)[:, Hq + Hkv:], slots, kc, vc, qo3, style=NEOX),
                ]
                calls[step]()
                torch.cuda.synchronize()
        else:
            chain(None)
        torch.cuda.synchronize()
        return [to_host_bits(t) for t in (qkv, cache, qout, qout2, kc, vc, qo3)]

    ref = run("synced")
    # every output was written (position 0 of the packed call is the identity,
    # so qkv itself only changes when S > 1)
    assert all(np.any(x != 0) for x in ref[2:4] + ref[6:])
    assert not np.array_equal(ref[1], case.new_cache()) and np.all(ref[4] != workloads.SENTINEL)
    for mode in ("back_to_back", "graph"):
        got = run(mode)
        for name, g_, r_ in zip(("qkv", "cache", "qout", "qout2", "kc", "vc", "qo3"), got, ref):
            assert np.array_equal(g_, r_), f"{mode}: {name}"


def test_first_call_inside_graph_capture():
    """A decode-sized call made for the first time in a process while a CUDA
    graph is being captured (the library then raises the kernel's shared
    memory limit during the capture) is captured and replays correctly. Runs
    in a fresh interpreter so that no earlier call has raised the limit."""
    import os
    import subprocess
    import sys
    code = r'''
import sys
sys.path.insert(0, "tests")
import numpy as np, torch
import workloads
from parity import check_contiguous, run_oracle_contiguous, to_dev, to_host_bits
import rope_kv_cache_gb300 as rk
case = workloads.make_continuous(256, 1, 32, 8, 128, 128, 64, workloads.NEOX, 5e5, seed=91)
cs, end, qkv = to_dev(case.cos_sin), to_dev(case.end_lens), to_dev(case.qkv)
cache, qout = to_dev(case.new_cache()), to_dev(case.new_qout())
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=torch.cuda.Stream()):
    rk.rope_write_kv_continuous(cs, end, qkv, cache, qout, case.Hq, case.Hkv, case.style,
                                stream=torch.cuda.current_stream())
g.replay()
torch.cuda.synchronize()
o_qkv, o_cache, o_qout = run_oracle_contiguous(case)
from parity import compare, cache_rotated, qout_rotated
compare(to_host_bits(qout), o_qout, qout_rotated(o_qout.shape, 128), "qOut")
compare(to_host_bits(cache), o_cache, cache_rotated(o_cache.shape, 128), "cache")
print("ok")
'''
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


@pytest.mark.parametrize("layout", ["one_token_sequences", "short_tree_sequences",
                                    "qknorm_one_token"])
def test_large_launches_of_short_sequences(layout):
    """Launches of 1024 tokens and more take the large-launch path whatever
    the sequences look like: 1536 one-token sequences (a large decode batch)
    and 96 tree sequences of 16 tokens, on every element against the oracle
    (small caches keep the oracle quick)."""
    if layout == "short_tree_sequences":
        case = workloads.make_tree(96, 16, 8, 2, 128, 64, 64, GPTJ, 1e4, seed=71,
                                   base_range=(0, 40), name=layout)
    else:
        case = workloads.make_continuous(1536, 1, 8, 2, 128, 128, 16, NEOX, 5e5, seed=72,
                                         name=layout)
        if layout == "qknorm_one_token":
            case.norm = workloads.norm_weights(72, 128)
    check_contiguous(case)


@pytest.mark.parametrize("mode,variant", [("continuous", "plain"), ("continuous", "norm"),
                                          ("packed", "plain"), ("tree", "plain")])
@pytest.mark.parametrize("tokens", [1023, 1024, 1025])
def test_launch_policy_boundary(mode, variant, tokens):
    """1023 tokens launch as decode-sized (prefetch prologue and residency
    cap); 1024 and more switch to the larger launch's shape and policy, which
    keeps the prologue for the plain continuous and packed calls only. Each
    side of the switch gives the oracle's result (the FP8-cache call's
    boundary is in test_gpu_fp8.py, the slot-mapping call's in
    test_gpu_slotmap.py)."""
    if mode == "continuous":
        case = workloads.make_continuous(tokens, 1, 8, 2, 128, 128, 16, GPTJ, 5e5,
                                         seed=5000 + tokens, name=f"edge{tokens}")
        if variant == "norm":
            case.norm = workloads.norm_weights(5000 + tokens, 128)
    elif mode == "packed":
        case = workloads.make_packed(1, tokens, 8, 2, 128, 64, tokens + 3, NEOX, 1e4,
                                     seed=5100 + tokens, cs_seq=tokens, cache_init="sentinel",
                                     name=f"edgep{tokens}")
    else:
        case = workloads.make_tree(tokens, 1, 8, 2, 128, 64, 64, GPTJ, 1e4, seed=5200 + tokens,
                                   base_range=(0, 60), cs_seq=64, name=f"edget{tokens}")
    check_contiguous(case)
