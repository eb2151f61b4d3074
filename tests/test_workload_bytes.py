"""Byte counts of the benchmark's workloads: the per-token formula of the
metric and the variant that counts each distinct cos/sin row once."""
import numpy as np

import workloads


def _tree(pos, cs_batch):
    B, S = len(pos), len(pos[0])
    Hq, Hkv, D, r, cap = 4, 2, 64, 32, 16
    rng = workloads.rng_for(0)
    qkv = workloads.fp16_normal(rng, (B, S, Hq + 2 * Hkv, D))
    cs = workloads.cos_sin_table(1e4, 8, r, batch=cs_batch)
    return workloads.ContiguousCase("tree", B, S, Hq, Hkv, D, r, cap, workloads.GPTJ, 1e4, cs,
                                    qkv, end_lens=np.full(B, S, np.int32),
                                    pos_ids=np.array(pos, dtype=np.int32))


def test_per_token_formula():
    c = _tree([[5, 6, 6, 7], [5, 5, 6, 1]], 1)
    per_tok = (4 + 4) * 64 * 2 + 32 * 4 + 4 * 64 * 2 + 2 * 2 * 64 * 2
    assert c.algorithmic_bytes() == 8 * per_tok


def test_distinct_rows_shared_and_per_sequence_tables():
    pos = [[5, 6, 6, 7], [5, 5, 6, 9]]              # 9 lies past the 8-row table
    shared, per_seq = _tree(pos, 1), _tree(pos, 2)
    base = shared.algorithmic_bytes() - 8 * 32 * 4
    assert shared.algorithmic_bytes_distinct_rows() == base + 3 * 32 * 4     # rows 5, 6, 7
    assert per_seq.algorithmic_bytes_distinct_rows() == base + 5 * 32 * 4    # (0,5..7), (1,5..6)


def test_distinct_rows_equal_per_token_for_one_prefill_sequence():
    c = workloads.make_continuous(1, 40, 4, 2, 64, 64, 64, workloads.NEOX, 1e4, seed=3,
                                  start_range=(0, 20), cs_seq=64)
    assert c.algorithmic_bytes_distinct_rows() == c.algorithmic_bytes()


def test_tree_config_within_one_percent():
    c = workloads.config("tree")
    a, d = c.algorithmic_bytes(), c.algorithmic_bytes_distinct_rows()
    assert 0 < a - d < 0.01 * a
