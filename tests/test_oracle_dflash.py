"""Pins for the oracle's DFlash prologue: delta metadata, the cos/sin gather,
and their composition with the paged update.

TensorRT-Edge-LLM "Dflash Runtime Kernels" prints only the signatures of
launchDFlashPrepareDeltaMetadata and launchDFlashGatherDeltaRope; the readings
(rows laid out [batchSize, deltaWidth]; positions oldDraftCacheLengths[b] + j,
the target length after the delta being old + deltaLen as the proposal-inputs
entry states; gather source [sourceRows, cacheCapacity, rotaryDim] indexed by
stateIndices[seq] and position, zero rows when out of range) are pinned here by
hand-written tables.
"""
import numpy as np
import pytest

import oracle
import workloads


def test_delta_metadata_by_hand():
    pos, seq = oracle.delta_metadata([10, 3, 0, 7], [2, 0, 7, -1], 4)
    assert pos.tolist() == [10, 11, -1, -1, -1, -1, -1, -1, 0, 1, 2, 3, -1, -1, -1, -1]
    assert seq.tolist() == [0, 0, -1, -1, -1, -1, -1, -1, 2, 2, 2, 2, -1, -1, -1, -1]


def test_delta_metadata_zero_width():
    pos, seq = oracle.delta_metadata([5, 6], [3, 1], 0)
    assert pos.size == 0 and seq.size == 0


def _source():
    # source[s, p, d] = 100 s + 10 p + d  (2 state rows, capacity 5, r = 4)
    s, p, d = np.meshgrid(np.arange(2), np.arange(5), np.arange(4), indexing="ij")
    return (100 * s + 10 * p + d).astype(np.float32)


ROWS_POS = np.array([1, 4, 5, -1, 2, 0, 3], dtype=np.int32)
ROWS_SEQ = np.array([0, 1, 0, -1, 2, 1, 0], dtype=np.int32)


def test_gather_with_state_indices_by_hand():
    out = oracle.gather_delta_rope(_source(), ROWS_POS, ROWS_SEQ,
                                   np.array([1, 0], dtype=np.int32), batch_size=2)
    want = [[110, 111, 112, 113],   # seq 0 -> state 1, pos 1
            [40, 41, 42, 43],       # seq 1 -> state 0, pos 4
            [0, 0, 0, 0],           # pos 5 == cacheCapacity
            [0, 0, 0, 0],           # padding
            [0, 0, 0, 0],           # seq 2 >= batchSize
            [0, 1, 2, 3],           # seq 1 -> state 0, pos 0
            [130, 131, 132, 133]]   # seq 0 -> state 1, pos 3
    assert out.tolist() == want


def test_gather_without_state_indices_by_hand():
    out = oracle.gather_delta_rope(_source(), ROWS_POS, ROWS_SEQ, None, batch_size=2)
    assert out[0].tolist() == [10, 11, 12, 13]      # seq 0 -> row 0
    assert out[1].tolist() == [140, 141, 142, 143]  # seq 1 -> row 1
    assert out[5].tolist() == [100, 101, 102, 103]
    # a single shared source row serves every sequence
    one = _source()[:1].copy()
    out = oracle.gather_delta_rope(one, ROWS_POS, ROWS_SEQ, None, batch_size=2)
    assert out[1].tolist() == [40, 41, 42, 43] and out[0].tolist() == [10, 11, 12, 13]
    # a state index outside [0, sourceRows) gives a zero row
    out = oracle.gather_delta_rope(one, ROWS_POS, ROWS_SEQ, np.array([0, 1], dtype=np.int32), 2)
    assert out[1].tolist() == [0, 0, 0, 0] and out[0].tolist() == [10, 11, 12, 13]


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_fused_is_the_composition(style):
    rng = workloads.rng_for(77)
    B, W, Hkv, D, r, tpp, mpps, P = 5, 6, 2, 64, 64, 4, 8, 40
    k = workloads.fp16_normal(rng, (B * W, Hkv, D))
    v = workloads.fp16_normal(rng, (B * W, Hkv, D))
    old = rng.integers(0, 20, size=B).astype(np.int32)
    lens = np.array([6, 0, 3, 9, 1], dtype=np.int32)
    src = workloads.cos_sin_table(1e4, 32, r, batch=3, pos_offset=[0, 7, 19])
    state = np.array([2, 0, 1, 1, -1], dtype=np.int32)
    table = np.full((B, 2, mpps), -1, dtype=np.int32)
    table[:, 0, :] = rng.permutation(P)[: B * mpps].reshape(B, mpps)
    table[:, 1, :] = P + rng.permutation(P)[: B * mpps].reshape(B, mpps)
    pool = workloads.sentinel_fill((2, P, tpp, Hkv, D))
    oracle.paged_fused(k, v, pool, src, old, lens, W, state, table, style)
    pos, seq = oracle.delta_metadata(old, lens, W)
    cs = oracle.gather_delta_rope(src, pos, seq, state, B)
    want = workloads.sentinel_fill((2, P, tpp, Hkv, D))
    oracle.paged(k, v, want, cs, pos, seq, table, style)
    assert np.array_equal(pool, want)
    # sequence 4 has no source row: its K is rotated by a zero row (zeros),
    # its V is still written
    assert (seq == 4).sum() == 1


def test_gather_sequence_past_batch_is_zero_even_with_a_valid_state():
    """A row whose sequence is not below batchSize has no state index to read
    (stateIndices has batchSize entries), so its row is zero even where
    stateIndices' memory past the batch would name a valid state row."""
    pos = np.array([1, 2, 3], dtype=np.int32)
    seq = np.array([0, 1, 2], dtype=np.int32)
    states = np.array([1, 0, 1], dtype=np.int32)   # entry 2 lies past batchSize = 2
    out = oracle.gather_delta_rope(_source(), pos, seq, states, batch_size=2)
    assert out.tolist() == [[110, 111, 112, 113], [20, 21, 22, 23], [0, 0, 0, 0]]
    three = np.concatenate([_source(), _source()[:1] + 1000])   # sourceRows 3 > batchSize
    out = oracle.gather_delta_rope(three, pos, seq, None, batch_size=2)
    assert out[2].tolist() == [0, 0, 0, 0] and out[1].tolist() == [120, 121, 122, 123]
