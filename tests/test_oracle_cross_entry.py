"""Cross-checks between the oracle's entry points, over random shapes.

The entry points come from different passages of the pages: the packed call
fills an empty cache from slot 0 (TensorRT-Edge-LLM "Apply Rope Write KV",
packed QKV), the continuous call takes kvCacheEndLens as where each sequence
ends once the call's tokens are written, the tree call takes the RoPE position from tokenPosIds, the
sglang-style call (rope_cache.py, fused_qk_rope_reshape_and_cache) takes a
position and a flat slot per token, and the paged update ("Dflash Runtime
Kernels") places rows through a page table. Where two of them must describe
the same write, their results must agree bit for bit:

* continuous with kvCacheEndLens = S is the packed call (cache from slot 0,
  positions s; the packed call's in-place Q equals the continuous qOut);
* tree with tokenPosIds = the linear positions end - S + s is the continuous
  call;
* the slot-mapping call, fed the continuous call's positions and the flat
  index of each token's slot in a one-block-per-sequence cache, is the
  continuous call;
* the paged update with one page per (sequence, slot range), the rows'
  positions and cos/sin rows taken from the contiguous layout, writes the
  rows the continuous call writes to the cache.

A wrong slot, position, block/offset split, head order or plane in any one
entry point breaks at least one of these. CPU only.
"""
import numpy as np
import pytest

import oracle
import workloads

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

NEOX, GPTJ = workloads.NEOX, workloads.GPTJ
SETTINGS = settings(max_examples=40, deadline=None, derandomize=True)


@st.composite
def shapes(draw):
    D = draw(st.sampled_from([16, 32, 64]))
    r = draw(st.sampled_from([x for x in (16, 32, 64) if x <= D]))
    Hkv = draw(st.integers(1, 3))
    Hq = Hkv * draw(st.integers(1, 3))
    B = draw(st.integers(1, 3))
    S = draw(st.integers(1, 9))
    style = draw(st.sampled_from([NEOX, GPTJ]))
    seed = draw(st.integers(0, 10 ** 6))
    return D, r, Hq, Hkv, B, S, style, seed


def _inputs(D, r, Hq, Hkv, B, S, seed, cap, cs_seq):
    rng = workloads.rng_for(seed)
    qkv = workloads.fp16_normal(rng, (B, S, Hq + 2 * Hkv, D))
    cs = workloads.cos_sin_table(1e4, cs_seq, r)
    return rng, qkv, cs


@SETTINGS
@given(shapes(), st.integers(0, 5))
def test_continuous_from_the_start_is_packed(sh, extra):
    D, r, Hq, Hkv, B, S, style, seed = sh
    cap = S + extra
    _, qkv, cs = _inputs(D, r, Hq, Hkv, B, S, seed, cap, cap)
    c_cache, c_q = workloads.sentinel_fill((B, 2, Hkv, cap, D)), workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(cs, np.full(B, S, np.int32), qkv, c_cache, c_q, Hq, Hkv, style)
    p_qkv, p_cache = qkv.copy(), workloads.sentinel_fill((B, 2, Hkv, cap, D))
    oracle.packed(cs, p_qkv, p_cache, Hq, Hkv, style)
    assert np.array_equal(c_cache, p_cache)
    assert np.array_equal(c_q, p_qkv[:, :, :Hq])
    for hk in range(Hkv):                       # the packed call's in-place K is the cache's K
        assert np.array_equal(p_qkv[:, :, Hq + hk], c_cache[:, 0, hk, :S])
    assert np.array_equal(p_qkv[:, :, Hq + Hkv:], qkv[:, :, Hq + Hkv:])


@SETTINGS
@given(shapes(), st.integers(0, 6), st.integers(0, 3))
def test_tree_with_linear_positions_is_continuous(sh, extra, short_table):
    D, r, Hq, Hkv, B, S, style, seed = sh
    cap = S + extra
    cs_seq = max(1, cap - short_table)         # a short table skips the tail
    rng, qkv, cs = _inputs(D, r, Hq, Hkv, B, S, seed, cap, cs_seq)
    end = rng.integers(0, cap + 3, size=B).astype(np.int32)   # some slots out of range
    c_cache, c_q = workloads.sentinel_fill((B, 2, Hkv, cap, D)), workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(cs, end, qkv, c_cache, c_q, Hq, Hkv, style)
    pos = (end[:, None] - S + np.arange(S)[None, :]).astype(np.int32)
    t_cache, t_q = workloads.sentinel_fill((B, 2, Hkv, cap, D)), workloads.sentinel_fill((B, S, Hq, D))
    oracle.tree(cs, end, pos, qkv, t_cache, t_q, Hq, Hkv, style)
    assert np.array_equal(c_cache, t_cache) and np.array_equal(c_q, t_q)


@SETTINGS
@given(shapes(), st.integers(0, 6))
def test_slot_mapping_of_a_contiguous_layout_is_continuous(sh, extra):
    """One block of `cap` slots per sequence: sequence b's token s goes to
    block b, offset end_b - S + s. The continuous cache [B, 2, Hkv, cap, D]
    holds the same rows as the [B blocks, cap, Hkv, D] caches, transposed."""
    D, r, Hq, Hkv, B, S, style, seed = sh
    cap = S + extra
    rng, qkv, cs = _inputs(D, r, Hq, Hkv, B, S, seed, cap, cap)
    end = rng.integers(S, cap + 1, size=B).astype(np.int32)   # every slot in range
    c_cache, c_q = workloads.sentinel_fill((B, 2, Hkv, cap, D)), workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(cs, end, qkv, c_cache, c_q, Hq, Hkv, style)
    T = B * S
    flat = qkv.reshape(T, Hq + 2 * Hkv, D)
    slot_in_seq = (end[:, None] - S + np.arange(S)[None, :])
    slots = (np.arange(B)[:, None] * cap + slot_in_seq).reshape(T).astype(np.int64)
    positions = slot_in_seq.reshape(T).astype(np.int64)
    kc = workloads.sentinel_fill((B, cap, Hkv, D))
    vc = workloads.sentinel_fill((B, cap, Hkv, D))
    qo = workloads.sentinel_fill((T, Hq, D))
    oracle.slot_mapping(cs[0], positions, flat[:, :Hq], flat[:, Hq:Hq + Hkv], flat[:, Hq + Hkv:],
                        slots, kc, vc, qo, None, style)
    assert np.array_equal(qo.reshape(B, S, Hq, D), c_q)
    assert np.array_equal(kc.transpose(0, 2, 1, 3), c_cache[:, 0])
    assert np.array_equal(vc.transpose(0, 2, 1, 3), c_cache[:, 1])


@SETTINGS
@given(shapes(), st.integers(1, 4), st.integers(1, 3))
def test_paged_identity_pages_is_continuous(sh, tpp, pages_per_seq):
    """Page table: sequence b's logical page l is K page b * M + l and V page
    numPages + b * M + l, so the pool [2, B * M, tpp, Hkv, D] is the
    continuous cache [B, 2, Hkv, M * tpp, D] with heads and slots swapped.
    Delta rows are the continuous call's K and V heads, each with the cos/sin
    row of its position (token-aligned)."""
    D, r, Hq, Hkv, B, S, style, seed = sh
    M = pages_per_seq
    cap = M * tpp
    S = min(S, cap)
    rng, qkv, cs = _inputs(D, r, Hq, Hkv, B, S, seed, cap, cap)
    qkv = np.ascontiguousarray(qkv[:, :S])
    end = rng.integers(S, cap + 1, size=B).astype(np.int32)
    c_cache, c_q = workloads.sentinel_fill((B, 2, Hkv, cap, D)), workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(cs, end, qkv, c_cache, c_q, Hq, Hkv, style)
    N = B * S
    pos = (end[:, None] - S + np.arange(S)[None, :]).reshape(N).astype(np.int32)
    seq = np.repeat(np.arange(B), S).astype(np.int32)
    k = np.ascontiguousarray(qkv[:, :, Hq:Hq + Hkv].reshape(N, Hkv, D))
    v = np.ascontiguousarray(qkv[:, :, Hq + Hkv:].reshape(N, Hkv, D))
    rows = np.ascontiguousarray(cs[0][pos])
    P = B * M
    table = np.empty((B, 2, M), np.int32)
    table[:, 0, :] = np.arange(B)[:, None] * M + np.arange(M)[None, :]
    table[:, 1, :] = P + table[:, 0, :]
    pool = workloads.sentinel_fill((2, P, tpp, Hkv, D))
    oracle.paged(k, v, pool, rows, pos, seq, table, style)
    as_cache = pool.reshape(2, B, M * tpp, Hkv, D).transpose(1, 0, 3, 2, 4)
    assert np.array_equal(as_cache, c_cache)
