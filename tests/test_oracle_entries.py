"""Brute-force placement pins for the oracle's four entry points.

Inputs are tiny and every element carries a unique integer code that FP16
holds exactly. Two kinds of cos/sin tables make the outputs readable by hand:

* identity rows (cos = 1, sin = 0): rotated heads pass through, so each cache
  slot and qOut row must hold the code of the token/head that the pages send
  there;
* "scale" rows (cos = 0, sin = 2^k in row k): x*cos + rotate(x)*sin becomes
  rotate(x) * 2^k exactly, so each output also tells which table row was used.

The expected slot maps are written out by hand from the pages:
TensorRT-Edge-LLM "Apply Rope Write KV" (packed: an empty cache fills from
slot 0; continuous/tree: kvCacheEndLens is where a sequence ends once the
call's tokens are written) and
"Dflash Runtime Kernels" (launchDFlashTargetKVCacheUpdate skip rules).
Everything not listed must keep the sentinel.
"""
import numpy as np
import pytest

import oracle
import workloads

SENT = workloads.SENTINEL


def f16(v):
    return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def val(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def coded_qkv(B, S, H, D, tok_stride=64):
    """qkv[b, s, head, d] = 1 + tok_stride*(b*S+s) + 16*head + d (exact in FP16)."""
    b, s, h, d = np.meshgrid(np.arange(B), np.arange(S), np.arange(H), np.arange(D),
                             indexing="ij")
    return f16(1 + tok_stride * (b * S + s) + 16 * h + d)


def identity_table(rows, r):
    t = np.zeros((1, rows, r), dtype=np.float32)
    t[:, :, : r // 2] = 1.0
    return t


def scale_table(rows, r):
    t = np.zeros((1, rows, r), dtype=np.float32)
    for k in range(rows):
        t[0, k, r // 2:] = 2.0 ** k
    return t


def rotated_scaled(x, r, style, k):
    """rotate(x) * 2^k on dims < r, x unchanged past r, written from the printed
    layouts: NeoX [x0,x1,x2,x3] -> [-x2,-x3,x0,x1], GPT-J -> [-x1,x0,-x3,x2]."""
    h = r // 2
    y = np.array(x, dtype=np.float64)
    for d in range(r):
        if style == oracle.NEOX:
            y[d] = (-x[d + h] if d < h else x[d - h]) * 2.0 ** k
        else:
            y[d] = (-x[d + 1] if d % 2 == 0 else x[d - 1]) * 2.0 ** k
    return y


# ----------------------------------------------------------- continuous --

# B=2, S=3, Hq=2, Hkv=1 (heads: Q0 Q1 K V), D=16, capacity 8, end = [5, 3]
CONT_MAP = {
    # (b, plane, hk, slot): (b, s, head)
    (0, 0, 0, 2): (0, 0, 2), (0, 0, 0, 3): (0, 1, 2), (0, 0, 0, 4): (0, 2, 2),
    (0, 1, 0, 2): (0, 0, 3), (0, 1, 0, 3): (0, 1, 3), (0, 1, 0, 4): (0, 2, 3),
    (1, 0, 0, 0): (1, 0, 2), (1, 0, 0, 1): (1, 1, 2), (1, 0, 0, 2): (1, 2, 2),
    (1, 1, 0, 0): (1, 0, 3), (1, 1, 0, 1): (1, 1, 3), (1, 1, 0, 2): (1, 2, 3),
}
CONT_POS = {(0, 0): 2, (0, 1): 3, (0, 2): 4, (1, 0): 0, (1, 1): 1, (1, 2): 2}


def _check_cache(cache, qkv, expect_map, pos_of, r, style, scaled):
    written = np.zeros(cache.shape[:4], dtype=bool)
    for (b, plane, hk, slot), (sb, ss, head) in expect_map.items():
        written[b, plane, hk, slot] = True
        x = val(qkv[sb, ss, head])
        if plane == 0 and scaled:
            want = rotated_scaled(x, r, style, pos_of[(sb, ss)])
            assert np.array_equal(val(cache[b, plane, hk, slot]), want), (b, plane, hk, slot)
        else:
            assert np.array_equal(cache[b, plane, hk, slot], qkv[sb, ss, head]), (b, plane, hk, slot)
    assert np.all(cache[~written] == SENT)


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
@pytest.mark.parametrize("scaled", [False, True])
def test_continuous_placement(style, scaled):
    B, S, Hq, Hkv, D, r, cap = 2, 3, 2, 1, 16, 16, 8
    qkv = coded_qkv(B, S, Hq + 2 * Hkv, D)
    cs = scale_table(cap, r) if scaled else identity_table(cap, r)
    end = np.array([5, 3], dtype=np.int32)
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout = workloads.sentinel_fill((B, S, Hq, D))
    qkv_before = qkv.copy()
    oracle.continuous(cs, end, qkv, cache, qout, Hq, Hkv, style)
    assert np.array_equal(qkv, qkv_before)  # qkv is read only here
    _check_cache(cache, qkv, CONT_MAP, CONT_POS, r, style, scaled)
    for (b, s), p in CONT_POS.items():
        for hq in range(Hq):
            x = val(qkv[b, s, hq])
            want = rotated_scaled(x, r, style, p) if scaled else x
            assert np.array_equal(val(qout[b, s, hq]), want)


def test_continuous_skips_out_of_range_slots():
    # end = [2, 9], S = 3, capacity 8: b0 slots -1,0,1 (s=0 skipped),
    # b1 slots 6,7,8 (s=2 skipped); table of 8 rows.
    B, S, Hq, Hkv, D, r, cap = 2, 3, 2, 1, 16, 16, 8
    qkv = coded_qkv(B, S, 4, D)
    end = np.array([2, 9], dtype=np.int32)
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(identity_table(cap, r), end, qkv, cache, qout, Hq, Hkv, oracle.NEOX)
    expect = {
        (0, 0, 0, 0): (0, 1, 2), (0, 0, 0, 1): (0, 2, 2),
        (0, 1, 0, 0): (0, 1, 3), (0, 1, 0, 1): (0, 2, 3),
        (1, 0, 0, 6): (1, 0, 2), (1, 0, 0, 7): (1, 1, 2),
        (1, 1, 0, 6): (1, 0, 3), (1, 1, 0, 7): (1, 1, 3),
    }
    _check_cache(cache, qkv, expect, {}, r, oracle.NEOX, False)
    assert np.all(qout[0, 0] == SENT) and np.all(qout[1, 2] == SENT)
    assert np.array_equal(qout[0, 1], qkv[0, 1, :2]) and np.array_equal(qout[1, 1], qkv[1, 1, :2])
    # a table shorter than the capacity also skips: positions >= 7 are dropped
    cache2 = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout2 = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(identity_table(7, r), end, qkv, cache2, qout2, Hq, Hkv, oracle.NEOX)
    assert np.all(cache2[1, :, :, 7] == SENT) and np.all(qout2[1, 1] == SENT)
    assert np.array_equal(cache2[1, 0, 0, 6], qkv[1, 0, 2])


def test_continuous_head_order_gqa():
    # Hq=4, Hkv=2: qkv heads are Q0..Q3, K0, K1, V0, V1.
    B, S, Hq, Hkv, D, r, cap = 1, 2, 4, 2, 16, 16, 4
    qkv = coded_qkv(B, S, 8, D, tok_stride=128)
    end = np.array([3], dtype=np.int32)  # slots 1, 2
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(identity_table(cap, r), end, qkv, cache, qout, Hq, Hkv, oracle.GPTJ)
    expect = {}
    for s, slot in ((0, 1), (1, 2)):
        expect[(0, 0, 0, slot)] = (0, s, 4)
        expect[(0, 0, 1, slot)] = (0, s, 5)
        expect[(0, 1, 0, slot)] = (0, s, 6)
        expect[(0, 1, 1, slot)] = (0, s, 7)
    _check_cache(cache, qkv, expect, {}, r, oracle.GPTJ, False)
    assert np.array_equal(qout[0], qkv[0, :, :4])


def test_partial_rotary_tail_is_bit_copy():
    B, S, Hq, Hkv, D, r, cap = 1, 2, 2, 1, 32, 16, 4
    rng = np.random.Generator(np.random.PCG64(9))
    qkv = workloads.fp16_normal(rng, (B, S, 4, D))
    cs = workloads.cos_sin_table(1e4, cap, r)
    end = np.array([2], dtype=np.int32)
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout = workloads.sentinel_fill((B, S, Hq, D))
    oracle.continuous(cs, end, qkv, cache, qout, Hq, Hkv, oracle.NEOX)
    assert np.array_equal(qout[0, :, :, r:], qkv[0, :, :2, r:])
    assert np.array_equal(cache[0, 0, 0, :2, r:], qkv[0, :, 2, r:])
    assert np.array_equal(cache[0, 1, 0, :2, :], qkv[0, :, 3, :])


# --------------------------------------------------------------- packed --

@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_packed_in_place_placement(style):
    # B=2, S=3, capacity 4: positions = slots = 0,1,2; slot 3 untouched;
    # Q and K rotated in place, V heads in qkv untouched.
    B, S, Hq, Hkv, D, r, cap = 2, 3, 2, 1, 16, 16, 4
    qkv = coded_qkv(B, S, 4, D)
    orig = qkv.copy()
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    oracle.packed(scale_table(cap, r), qkv, cache, Hq, Hkv, style)
    for b in range(B):
        for s in range(S):
            for head in range(3):  # Q0, Q1, K
                want = rotated_scaled(val(orig[b, s, head]), r, style, s)
                assert np.array_equal(val(qkv[b, s, head]), want)
            assert np.array_equal(qkv[b, s, 3], orig[b, s, 3])
            assert np.array_equal(cache[b, 0, 0, s], qkv[b, s, 2])
            assert np.array_equal(cache[b, 1, 0, s], orig[b, s, 3])
        assert np.all(cache[b, :, :, 3] == SENT)


def test_packed_rejects_sequence_longer_than_capacity():
    qkv = coded_qkv(1, 5, 4, 16)
    cache = workloads.sentinel_fill((1, 2, 1, 4, 16))
    with pytest.raises(ValueError):
        oracle.packed(identity_table(8, 16), qkv, cache, 2, 1, oracle.NEOX)


# ----------------------------------------------------------------- tree --

@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_tree_position_vs_slot(style):
    # end = [6, 3], S = 3: b0 slots 3,4,5; b1 slots 0,1,2. Tree positions
    # b0 [3,4,4] (siblings share a position), b1 [0,1,-1] (last token padding).
    B, S, Hq, Hkv, D, r, cap = 2, 3, 2, 1, 16, 16, 8
    qkv = coded_qkv(B, S, 4, D)
    end = np.array([6, 3], dtype=np.int32)
    pos = np.array([[3, 4, 4], [0, 1, -1]], dtype=np.int32)
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout = workloads.sentinel_fill((B, S, Hq, D))
    oracle.tree(scale_table(cap, r), end, pos, qkv, cache, qout, Hq, Hkv, style)
    expect = {
        (0, 0, 0, 3): (0, 0, 2), (0, 0, 0, 4): (0, 1, 2), (0, 0, 0, 5): (0, 2, 2),
        (0, 1, 0, 3): (0, 0, 3), (0, 1, 0, 4): (0, 1, 3), (0, 1, 0, 5): (0, 2, 3),
        (1, 0, 0, 0): (1, 0, 2), (1, 0, 0, 1): (1, 1, 2),
        (1, 1, 0, 0): (1, 0, 3), (1, 1, 0, 1): (1, 1, 3),
    }
    pos_of = {(0, 0): 3, (0, 1): 4, (0, 2): 4, (1, 0): 0, (1, 1): 1}
    _check_cache(cache, qkv, expect, pos_of, r, style, True)
    for (b, s), p in pos_of.items():
        for hq in range(Hq):
            assert np.array_equal(val(qout[b, s, hq]), rotated_scaled(val(qkv[b, s, hq]), r, style, p))
    assert np.all(qout[1, 2] == SENT)


# ---------------------------------------------------------------- paged --

def _paged_case(Hkv=1, D=16, r=16):
    """3 sequences, 2 logical pages each, 4 tokens per page, 4 pages per plane.

    page table (canonical ids; V ids live in [4, 8)):
      seq 0: K [2, 0]   V [5, 7]
      seq 1: K [-1, 3]  V [6, 2]     (2 is a K-plane id in the V column)
      seq 2: K [5, 1]   V [8, 4]     (5 is a V-plane id in the K column, 8 >= 2*4)
    rows (position, sequence):
      t0 (1, 0)  t1 (-1, -1)  t2 (6, 0)  t3 (2, 1)  t4 (5, 1)
      t5 (9, 0)  t6 (0, 2)    t7 (4, 2)  t8 (0, 3)  t9 (8, 1)
    (t5 and t9 fall one logical page past maxPagesPerSeq; t8 names a sequence
    past batchSize.)
    """
    table = np.array([[[2, 0], [5, 7]], [[-1, 3], [6, 2]], [[5, 1], [8, 4]]], dtype=np.int32)
    positions = np.array([1, -1, 6, 2, 5, 9, 0, 4, 0, 8], dtype=np.int32)
    seqs = np.array([0, -1, 0, 1, 1, 0, 2, 2, 3, 1], dtype=np.int32)
    N = len(positions)
    t, h, d = np.meshgrid(np.arange(N), np.arange(Hkv), np.arange(D), indexing="ij")
    k = f16(1 + d + 16 * h + 17 * Hkv * t) if Hkv > 1 else f16(1 + d + 17 * t)
    v = f16(200 + d + 16 * h + 17 * Hkv * t) if Hkv > 1 else f16(200 + d + 17 * t)
    return table, positions, seqs, k, v


# hand-written destinations: (plane, page within plane, slot in page) <- row
PAGED_K = {(0, 2, 1): 0, (0, 0, 2): 2, (0, 3, 1): 4, (0, 1, 0): 7}
PAGED_V = {(1, 1, 1): 0, (1, 3, 2): 2, (1, 2, 2): 3, (1, 0, 0): 7}


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_paged_placement_and_skips(style):
    table, positions, seqs, k, v = _paged_case()
    N, Hkv, D, r = len(positions), 1, 16, 16
    cs = np.zeros((N, r), dtype=np.float32)
    for t in range(N):
        cs[t, r // 2:] = 2.0 ** t  # row t scales by 2^t: token-aligned, not by position
    pool = workloads.sentinel_fill((2, 4, 4, Hkv, D))
    oracle.paged(k, v, pool, cs, positions, seqs, table, style)
    written = np.zeros(pool.shape[:3], dtype=bool)
    for (plane, page, slot), t in PAGED_K.items():
        written[plane, page, slot] = True
        want = rotated_scaled(val(k[t, 0]), r, style, t)
        assert np.array_equal(val(pool[plane, page, slot, 0]), want), (plane, page, slot)
    for (plane, page, slot), t in PAGED_V.items():
        written[plane, page, slot] = True
        assert np.array_equal(pool[plane, page, slot, 0], v[t, 0])
    assert np.all(pool[~written] == SENT)


def test_paged_heads_are_token_major():
    table, positions, seqs, k, v = _paged_case(Hkv=2)
    N, D, r = len(positions), 16, 16
    cs = np.zeros((N, r), dtype=np.float32)
    cs[:, : r // 2] = 1.0  # identity rows
    pool = workloads.sentinel_fill((2, 4, 4, 2, D))
    oracle.paged(k, v, pool, cs, positions, seqs, table, oracle.NEOX)
    for (plane, page, slot), t in PAGED_K.items():
        assert np.array_equal(pool[plane, page, slot], k[t])
    for (plane, page, slot), t in PAGED_V.items():
        assert np.array_equal(pool[plane, page, slot], v[t])


def test_paged_rows_agree_with_pool():
    table, positions, seqs, k, v = _paged_case()
    N, D, r = len(positions), 16, 16
    cs = workloads.cos_sin_table(5e5, 16, r)[0][np.maximum(positions, 0)]
    kd, vd, ko, vo = oracle.paged_rows(k, v, cs, positions, seqs, table, 4, 4, oracle.NEOX)
    assert list(kd >= 0) == [True, False, True, False, True, False, False, True, False, False]
    assert list(vd >= 0) == [True, False, True, True, False, False, False, True, False, False]
    pool = workloads.sentinel_fill((2, 4, 4, 1, D))
    oracle.paged(k, v, pool, cs, positions, seqs, table, oracle.NEOX)
    flat = pool.reshape(-1)
    for t in range(N):
        if kd[t] >= 0:
            assert np.array_equal(flat[kd[t]: kd[t] + D], ko[t].reshape(-1))
        if vd[t] >= 0:
            assert np.array_equal(flat[vd[t]: vd[t] + D], vo[t].reshape(-1))


def test_capacity_rule():
    # checkDFlashRopeCapacity: reject only a table longer than the capacity
    assert not oracle.capacity_rejected(4096, 4096)
    assert not oracle.capacity_rejected(4000, 4096)
    assert oracle.capacity_rejected(4097, 4096)
    assert not oracle.capacity_rejected(0, 0)


# ----------------------------------------------------- per-sequence tables --

def batched_scale_table(B, rows, r):
    """One table per sequence ("Apply Rope Write KV", cosSinCacheBatchSize = B):
    sequence b's row k has cos 0 and sin 2^(k + 4b), so every rotated output
    names both the row and the table it was read from."""
    t = np.zeros((B, rows, r), dtype=np.float32)
    for b in range(B):
        for k in range(rows):
            t[b, k, r // 2:] = 2.0 ** (k + 4 * b)
    return t


@pytest.mark.parametrize("mode", ["packed", "continuous", "tree"])
@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_per_sequence_tables(mode, style):
    # B=2, S=2, Hq=2, Hkv=1, D=r=16, 4 rows per table. Codes stay <= 256 and
    # scales <= 2^7, so every product is exact in FP16.
    B, S, Hq, Hkv, D, r, cap = 2, 2, 2, 1, 16, 16, 4
    qkv = coded_qkv(B, S, Hq + 2 * Hkv, D)
    orig = qkv.copy()
    cs = batched_scale_table(B, cap, r)
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout = workloads.sentinel_fill((B, S, Hq, D))
    end = np.array([2, 4], dtype=np.int32)           # b0 slots 0,1; b1 slots 2,3
    if mode == "packed":
        oracle.packed(cs, qkv, cache, Hq, Hkv, style)
        pos = {(b, s): s for b in range(B) for s in range(S)}
        slot = pos
    elif mode == "continuous":
        oracle.continuous(cs, end, qkv, cache, qout, Hq, Hkv, style)
        pos = {(0, 0): 0, (0, 1): 1, (1, 0): 2, (1, 1): 3}
        slot = pos
    else:
        ids = np.array([[1, 1], [0, 3]], dtype=np.int32)
        oracle.tree(cs, end, ids, qkv, cache, qout, Hq, Hkv, style)
        pos = {(0, 0): 1, (0, 1): 1, (1, 0): 0, (1, 1): 3}
        slot = {(0, 0): 0, (0, 1): 1, (1, 0): 2, (1, 1): 3}
    for (b, s), p in pos.items():
        e = p + 4 * b                                   # table b, row p
        qdst = qkv[b, s, :Hq] if mode == "packed" else qout[b, s]
        for hq in range(Hq):
            want = rotated_scaled(val(orig[b, s, hq]), r, style, e)
            assert np.array_equal(val(qdst[hq]), want), (mode, b, s, hq)
        want_k = rotated_scaled(val(orig[b, s, Hq]), r, style, e)
        assert np.array_equal(val(cache[b, 0, 0, slot[(b, s)]]), want_k), (mode, b, s)
        assert np.array_equal(cache[b, 1, 0, slot[(b, s)]], orig[b, s, Hq + 1])


# ------------------------------------------- positions past the cos/sin table --

def _table_prefix(rows, r, extra=1):
    """A [1, rows, r] table that is the prefix of a larger array: a read of row
    `rows` (one past the end) stays inside allocated memory and returns a row
    of 2^10, which no pinned output may contain."""
    big = np.zeros((1, rows + extra, r), dtype=np.float32)
    big[0, :, : r // 2] = 1.0
    big[0, rows:, :] = 2.0 ** 10
    return big[:, :rows]


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_tree_position_at_table_end_is_skipped(style):
    # "Apply Rope Write KV", tree: the cos/sin row is tokenPosIds[b, s]; a
    # position equal to cosSinSeqLen has no row, so the token writes nothing.
    B, S, Hq, Hkv, D, r, cap = 1, 3, 2, 1, 16, 16, 8
    qkv = coded_qkv(B, S, 4, D)
    cs = _table_prefix(5, r)                          # rows 0..4
    end = np.array([3], dtype=np.int32)               # slots 0, 1, 2
    ids = np.array([[4, 5, 2]], dtype=np.int32)        # 5 == cosSinSeqLen
    cache = workloads.sentinel_fill((B, 2, Hkv, cap, D))
    qout = workloads.sentinel_fill((B, S, Hq, D))
    oracle.tree(cs, end, ids, qkv, cache, qout, Hq, Hkv, style)
    expect = {(0, 0, 0, 0): (0, 0, 2), (0, 1, 0, 0): (0, 0, 3),
              (0, 0, 0, 2): (0, 2, 2), (0, 1, 0, 2): (0, 2, 3)}
    _check_cache(cache, qkv, expect, {}, r, style, False)
    assert np.all(qout[0, 1] == SENT)
    assert np.array_equal(qout[0, 0], qkv[0, 0, :2]) and np.array_equal(qout[0, 2], qkv[0, 2, :2])


# ------------------------------------------------------ argument checks --

def _dims_case(B=2, S=2, Hq=2, Hkv=1, D=16, r=16, cs_batch=1, cap=4):
    qkv = coded_qkv(B, S, Hq + 2 * Hkv, D)
    cs = np.zeros((cs_batch, cap, r), dtype=np.float32)
    cs[:, :, : r // 2] = 1.0
    return (qkv, cs, np.full(B, S, np.int32), workloads.sentinel_fill((B, 2, Hkv, cap, D)),
            workloads.sentinel_fill((B, S, Hq, D)))


def _call(mode, qkv, cs, end, cache, qo, Hq, Hkv):
    B, S = qkv.shape[:2]
    D = qkv.shape[3]
    if mode == "packed":
        oracle.packed(cs, qkv, cache, Hq, Hkv, oracle.NEOX)
    elif mode == "continuous":
        oracle.continuous(cs, end, qkv, cache, qo, Hq, Hkv, oracle.NEOX)
    elif mode == "tree":
        pos = np.tile(np.arange(S, dtype=np.int32), (B, 1))
        oracle.tree(cs, end, pos, qkv, cache, qo, Hq, Hkv, oracle.NEOX)
    elif mode == "qknorm":
        w = f16(np.ones(D))
        oracle.continuous_qknorm(cs, end, qkv, cache, qo, w, w, 1e-6, Hq, Hkv, oracle.NEOX)
    else:
        c8 = np.zeros(cache.shape, dtype=np.uint8)
        oracle.continuous_fp8(cs, end, qkv, c8, qo, 1.0, 1.0, Hq, Hkv, oracle.NEOX)


@pytest.mark.parametrize("mode", ["packed", "continuous", "tree", "qknorm", "fp8"])
@pytest.mark.parametrize("bad", ["cos_sin_batch", "gqa_ratio", "odd_rotary_dim"])
def test_invalid_dims_are_rejected(mode, bad):
    """The table batch is 1 (shared) or B (one table per sequence), nothing
    else ("Apply Rope Write KV", cosSinCacheBatchSize); Q heads come in whole
    groups per KV head (sglang rope_cache.py, QH_PER_KH = qh // kh); the
    rotated dims form pairs. Each violation is an error that writes nothing,
    while the same call with valid dims succeeds."""
    Hq, Hkv, r, csb = 2, 1, 16, 1
    if bad == "cos_sin_batch":
        csb = 3                                    # B = 2
    elif bad == "gqa_ratio":
        Hq, Hkv = 3, 2
    else:
        r = 15
    qkv, cs, end, cache, qo = _dims_case(Hq=Hq, Hkv=Hkv, r=r, cs_batch=csb)
    with pytest.raises(ValueError):
        _call(mode, qkv, cs, end, cache, qo, Hq, Hkv)
    assert np.all(cache == SENT) and np.all(qo == SENT)
    assert np.array_equal(qkv, coded_qkv(2, 2, Hq + 2 * Hkv, 16))
    good = _dims_case(cs_batch=2)                 # batch of tables == B is valid
    _call(mode, *good, 2, 1)


def test_paged_plane_boundaries():
    """Canonical page ids are flat indices of the [2, numPages] pool ("Dflash
    Runtime Kernels", launchDFlashTargetKVCacheUpdate): a K write needs
    0 <= id < numPages, a V write numPages <= id < 2 * numPages, each plane
    decided on its own. numPages = 4, TPP = 4, one sequence, rows t at
    positions 1, 6, 11, 12 (logical pages 0..3):

        logical page   0   1   2   3
        K column       4   3   0  -1    (4 == numPages is a V-plane id)
        V column       5   7   8   3    (8 == 2 * numPages; 3 is a K-plane id)

    Logical page 0's K id, read as a flat index, is V-plane page 0, which no
    row writes: a K write there would show.
    """
    Hkv, D, r = 1, 16, 16
    table = np.array([[[4, 3, 0, -1], [5, 7, 8, 3]]], dtype=np.int32)
    positions = np.array([1, 6, 11, 12], dtype=np.int32)
    seqs = np.zeros(4, dtype=np.int32)
    t, d = np.meshgrid(np.arange(4), np.arange(D), indexing="ij")
    k = f16(1 + d + 17 * t)[:, None, :]
    v = f16(200 + d + 17 * t)[:, None, :]
    cs = np.zeros((4, r), dtype=np.float32)
    for i in range(4):
        cs[i, r // 2:] = 2.0 ** i
    pool = workloads.sentinel_fill((2, 4, 4, Hkv, D))
    oracle.paged(np.ascontiguousarray(k), np.ascontiguousarray(v), pool, cs, positions, seqs,
                 table, oracle.NEOX)
    want_k = {(0, 3, 2): 1, (0, 0, 3): 2}           # (plane, page, slot) <- row
    want_v = {(1, 1, 1): 0, (1, 3, 2): 1}
    written = np.zeros(pool.shape[:3], dtype=bool)
    for (pl, pg, sl), i in want_k.items():
        written[pl, pg, sl] = True
        assert np.array_equal(val(pool[pl, pg, sl, 0]), rotated_scaled(val(k[i, 0]), r, oracle.NEOX, i))
    for (pl, pg, sl), i in want_v.items():
        written[pl, pg, sl] = True
        assert np.array_equal(pool[pl, pg, sl, 0], v[i, 0])
    assert np.all(pool[~written] == SENT)


def test_packed_rejects_table_shorter_than_sequence():
    """The packed call's positions are 0 .. S-1 (an empty cache, filled from 0),
    so a table with fewer than S rows cannot serve it: an error that writes
    nothing, even though the cache is long enough."""
    qkv = coded_qkv(1, 5, 4, 16)
    cache = workloads.sentinel_fill((1, 2, 1, 8, 16))
    with pytest.raises(ValueError):
        oracle.packed(identity_table(4, 16), qkv, cache, 2, 1, oracle.NEOX)
    assert np.all(cache == SENT) and np.array_equal(qkv, coded_qkv(1, 5, 4, 16))
    oracle.packed(identity_table(5, 16), qkv, cache, 2, 1, oracle.NEOX)
