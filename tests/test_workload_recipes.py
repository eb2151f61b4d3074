"""The seeded inputs follow the stated recipes.

Both sides of every parity test, and the benchmark, draw their inputs from
workloads.py; these checks hold the generated configurations to the shapes and
distributions the recipes state (the TensorRT-Edge-LLM "Apply Rope Write KV"
and "Dflash Runtime Kernels" workloads: Llama-style GQA prefill, decode,
tree-speculative decoding and paged delta updates), and to the input
contracts the oracle assumes (no two tokens of a call share a cache slot).
CPU only.
"""
import numpy as np
import pytest

import workloads


def test_prefill_recipe():
    c = workloads.config("prefill")
    assert (c.mode, c.B, c.S, c.Hq, c.Hkv, c.D, c.r, c.cap) == ("continuous", 4, 2048, 32, 8,
                                                                128, 128, 8192)
    assert c.style == workloads.NEOX and c.cos_sin.shape == (1, 8192, 128)
    start = c.end_lens.astype(np.int64) - c.S
    assert np.all((start >= 0) & (start <= 4096))
    assert c.qkv.shape == (4, 2048, 48, 128) and c.qkv.dtype == np.uint16


def test_decode_recipe():
    c = workloads.config("decode")
    assert (c.B, c.S, c.cap) == (256, 1, 8192)
    assert np.all((c.end_lens >= 1) & (c.end_lens <= 8192))
    assert len(np.unique(c.end_lens)) > 200            # spread over the cache


def test_tree_recipe():
    c = workloads.config("tree")
    assert (c.mode, c.B, c.S, c.D, c.r, c.cap) == ("tree", 64, 64, 128, 64, 4096)
    assert c.style == workloads.GPTJ
    for b in range(c.B):
        base = int(c.end_lens[b]) - c.S
        assert 128 <= base <= 4000
        depth = c.pos_ids[b].astype(np.int64) - base
        assert depth[0] == 0 and np.all((depth >= 0) & (depth <= 6))
        # node i > 0 hangs under an earlier node of depth <= 5: depth d > 0
        # appears only after some node of depth d - 1
        for i in range(1, c.S):
            assert depth[i] >= 1 and (depth[:i] == depth[i] - 1).any()
    rows = sum(len(np.unique(c.pos_ids[b])) for b in range(c.B))
    assert rows == 7 * c.B                             # seven tree levels per sequence


def test_paged_recipe():
    c = workloads.config("paged")
    assert (c.N, c.B, c.Hkv, c.D, c.r, c.tokens_per_page, c.max_pages_per_seq) == \
        (16384, 128, 8, 128, 128, 64, 512)
    pad = c.positions < 0
    assert pad.sum() == 819 and np.all(c.seq_ids[pad] == -1)
    valid = ~pad
    assert valid.sum() == 15565
    seq, pos = c.seq_ids[valid], c.positions[valid].astype(np.int64)
    assert np.all(np.diff(seq) >= 0)                   # grouped by sequence, in order
    for b in np.unique(seq):
        p = pos[seq == b]
        assert np.array_equal(p, p[0] + np.arange(len(p)))   # consecutive positions
        assert 1 <= len(p) <= 256 and p[-1] < 512 * 64
    k, v = c.page_table[:, 0], c.page_table[:, 1]
    num = c.num_pages
    km, vm = k[k >= 0], v[v >= 0]
    assert len(np.unique(km)) == km.size and np.all(km < num)
    assert len(np.unique(vm)) == vm.size and np.all((vm >= num) & (vm < 2 * num))
    unmapped = (c.page_table < 0).mean()
    assert 0.015 < unmapped < 0.025
    # token-aligned cos/sin: row t is the table row of row t's position
    table = workloads.cos_sin_table(c.theta, int(pos.max()) + 1, c.r)[0]
    assert np.array_equal(c.cos_sin_rows[valid], table[pos])
    assert np.all(c.cos_sin_rows[pad] == 0)


@pytest.mark.parametrize("name", ["slotmap_prefill", "slotmap_decode"])
def test_slot_mapping_slots_unique_in_every_ring_step(name):
    c = workloads.config(name)
    n_slots = c.num_blocks * c.block_size
    for k in range(4):
        pos, slots = workloads.step_variant(c, k)
        assert len(np.unique(slots)) == slots.size and slots.min() >= 0 and slots.max() < n_slots
        start = 0
        for n in c.seq_lens:                            # a sequence's positions run on
            p = pos[start:start + n]
            assert np.array_equal(p, p[0] + np.arange(n))
            start += n


@pytest.mark.parametrize("name", ["prefill", "decode", "tree"])
def test_contiguous_ring_steps_stay_in_the_cache(name):
    c = workloads.config(name)
    ends = []
    for k in range(4):
        end, pos = workloads.step_variant(c, k)
        assert np.all((end - c.S >= 0) & (end <= c.cap))
        if c.mode == "tree":
            assert np.all((pos >= 0) & (pos < c.cos_sin.shape[1]))
        ends.append(end)
    assert not np.array_equal(ends[0], ends[1])         # steps write different slots


def test_packed_tiny_recipe():
    c = workloads.config("packed_tiny")
    assert (c.mode, c.B, c.S, c.Hq, c.Hkv, c.D, c.r, c.cap) == ("packed", 1, 16, 4, 2, 64, 64, 64)
    assert c.cache_init == "zero" and np.all(c.new_cache() == 0)
