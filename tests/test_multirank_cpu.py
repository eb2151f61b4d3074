"""The multi-rank path on the CPU with gloo (world size 2).

The fused RoPE + KV-cache write has no exchange step: sequences are
independent, so ranks run replicas (or disjoint batch shards) and share only
the barrier and the max-over-ranks timing reduction. These tests run that host
logic as two gloo processes on 127.0.0.1.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, out):
    import bench
    _init(rank, world, port)
    try:
        mine = [0.25, 0.75][rank]
        m = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        dist.barrier()
        out[rank] = (m, bench.whole_job_rate(world, 8192, 100, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_timing_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    assert out[0][0] == 0.75
    assert out[0][1] == pytest.approx(2 * 8192 * 100 / 0.75)


def _shard_worker(rank, world, port, out):
    import oracle
    import workloads
    _init(rank, world, port)
    try:
        case = workloads.make_continuous(4, 9, 4, 2, 64, 64, 32, workloads.NEOX, 1e4, seed=42)
        lo, hi = rank * case.B // world, (rank + 1) * case.B // world
        cache = workloads.sentinel_fill((hi - lo, 2, case.Hkv, case.cap, case.D))
        qout = workloads.sentinel_fill((hi - lo, case.S, case.Hq, case.D))
        oracle.continuous(case.cos_sin, np.ascontiguousarray(case.end_lens[lo:hi]),
                          np.ascontiguousarray(case.qkv[lo:hi]), cache, qout, case.Hq, case.Hkv,
                          case.style)
        parts = [None] * world
        dist.all_gather_object(parts, (lo, cache, qout))
        if rank == 0:
            out["parts"] = parts
    finally:
        dist.destroy_process_group()


def test_batch_shards_recompose_the_whole_batch():
    """Two ranks each handle half of the sequences; their results, put side by
    side, equal the single-process result: nothing crosses a shard."""
    import oracle
    import workloads
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_shard_worker, args=(world, port, out), nprocs=world, join=True)
    parts = sorted(out["parts"], key=lambda p: p[0])
    case = workloads.make_continuous(4, 9, 4, 2, 64, 64, 32, workloads.NEOX, 1e4, seed=42)
    cache = case.new_cache()
    qout = case.new_qout()
    oracle.continuous(case.cos_sin, case.end_lens, case.qkv, cache, qout, case.Hq, case.Hkv,
                      case.style)
    assert np.array_equal(np.concatenate([p[1] for p in parts]), cache)
    assert np.array_equal(np.concatenate([p[2] for p in parts]), qout)
