"""The benchmark's CPU baseline cuts each workload into small oracle calls
(bench.OracleUnits) so that no multi-GB cache or pool is allocated on the
host. These tests check, on small cases of every workload kind, that the
units compute exactly what the oracle's call on the whole case computes:
every output of every unit is compared bit for bit with the corresponding
part of the whole call's output. CPU only."""
import numpy as np
import pytest

import bench
import oracle
import workloads

NEOX, GPTJ = workloads.NEOX, workloads.GPTJ


def _contiguous(mode, style, norm=False, fp8=False):
    if mode == "tree":
        c = workloads.make_tree(3, 37, 4, 2, 64, 32, 96, style, 1e4, seed=61, base_range=(0, 40),
                                name="units_tree")
    elif mode == "packed":
        c = workloads.make_packed(2, 21, 4, 2, 64, 64, 32, style, 1e4, seed=62, name="units_packed")
    else:
        c = workloads.make_continuous(3, 37, 4, 2, 64, 64, 96, style, 1e4, seed=63,
                                      start_range=(0, 50), name="units_cont")
    if norm:
        c.norm = workloads.norm_weights(64, 64)
    if fp8:
        c.fp8_scales = (0.05, 0.04)
    return c


def _whole(c):
    qkv = c.qkv.copy()
    qout = c.new_qout()
    if c.fp8_scales is not None:
        cache = c.new_cache8()
        oracle.continuous_fp8(c.cos_sin, c.end_lens, qkv, cache, qout, *c.fp8_scales, c.Hq,
                              c.Hkv, c.style)
    else:
        cache = c.new_cache()
        if c.mode == "packed":
            oracle.packed(c.cos_sin, qkv, cache, c.Hq, c.Hkv, c.style)
        elif c.mode == "tree":
            oracle.tree(c.cos_sin, c.end_lens, c.pos_ids, qkv, cache, qout, c.Hq, c.Hkv, c.style)
        elif c.norm is not None:
            oracle.continuous_qknorm(c.cos_sin, c.end_lens, qkv, cache, qout, *c.norm, c.Hq,
                                     c.Hkv, c.style)
        else:
            oracle.continuous(c.cos_sin, c.end_lens, qkv, cache, qout, c.Hq, c.Hkv, c.style)
    return qkv, cache, qout


@pytest.mark.parametrize("mode,style,norm,fp8", [
    ("continuous", NEOX, False, False), ("continuous", GPTJ, True, False),
    ("continuous", NEOX, False, True), ("tree", GPTJ, False, False), ("packed", NEOX, False, False)])
def test_contiguous_units(mode, style, norm, fp8):
    c = _contiguous(mode, style, norm, fp8)
    w_qkv, w_cache, w_qout = _whole(c)
    u = bench.OracleUnits("units", chunk=16, case=c)
    assert sum(t for _, t in u.calls) == c.tokens
    for (fn, _), meta in zip(u.calls, u.meta):
        if meta[0] == "all":
            qkv, cache = fn()
            assert np.array_equal(qkv, w_qkv) and np.array_equal(cache, w_cache)
            continue
        _, b, s0, m = meta
        qout, cache = fn()
        assert np.array_equal(qout[0, :m], w_qout[b, s0:s0 + m]), meta
        slots = int(c.end_lens[b]) - c.S + s0 + np.arange(m)
        ok = (slots >= 0) & (slots < c.cap)
        assert np.array_equal(cache[0][:, :, slots[ok]], w_cache[b][:, :, slots[ok]]), meta


def test_paged_units():
    c = workloads.make_paged(300, 4, 2, 64, 64, 16, 32, 128, GPTJ, 1e4, seed=64,
                             len_range=(1, 100))
    whole = oracle.paged_rows(c.k_delta, c.v_delta, c.cos_sin_rows, c.positions, c.seq_ids,
                              c.page_table, c.num_pages, c.tokens_per_page, c.style)
    u = bench.OracleUnits("units", chunk=64, case=c)
    for (fn, _), (_, t0, n) in zip(u.calls, u.meta):
        for got, want in zip(fn(), whole):
            assert np.array_equal(got, want[t0:t0 + n])


def test_fused_units():
    c = workloads.make_paged_fused(5, 21, 2, 64, 64, 8, 6, 40, NEOX, 1e4, seed=65,
                                   len_range=(0, 21), source_rows=2, with_state=True)
    pos, seq = oracle.delta_metadata(c.old_lengths, c.delta_lengths, c.W)
    cs = oracle.gather_delta_rope(c.source, pos, seq, c.state, c.B)
    whole = oracle.paged_rows(c.k_delta, c.v_delta, cs, pos, seq, c.page_table, c.num_pages,
                              c.tokens_per_page, c.style)
    u = bench.OracleUnits("units", case=c)
    for (fn, _), (_, b) in zip(u.calls, u.meta):
        for got, want in zip(fn(), whole):
            assert np.array_equal(got, want[b * c.W:(b + 1) * c.W]), b


def test_slotmap_units():
    c = workloads.make_slotmap([5, 40, 1, 23], 4, 2, 64, 64, NEOX, 1e4, seed=66, block_size=8,
                               num_blocks=20, start_range=(0, 50), cs_rows=128)
    c.slots[3] = -1
    kc = workloads.sentinel_fill(c.cache_shape())
    vc = workloads.sentinel_fill(c.cache_shape())
    qo = workloads.sentinel_fill((c.T, c.Hq, c.D))
    oracle.slot_mapping(c.cos_sin, c.positions, c.q, c.k, c.v, c.slots, kc, vc, qo, None, c.style)
    u = bench.OracleUnits("units", chunk=16, case=c)
    for (fn, _), (_, t0, n) in zip(u.calls, u.meta):
        qout, ukc, uvc, uslots = fn()
        assert np.array_equal(qout, qo[t0:t0 + n])
        for j in range(n):
            if uslots[j] >= 0:
                s = c.slots[t0 + j]
                assert np.array_equal(ukc.reshape(-1, c.Hkv, c.D)[uslots[j]],
                                      kc.reshape(-1, c.Hkv, c.D)[s])
                assert np.array_equal(uvc.reshape(-1, c.Hkv, c.D)[uslots[j]],
                                      vc.reshape(-1, c.Hkv, c.D)[s])
