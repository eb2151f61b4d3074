"""Pins for the oracle's rotation of one head (x' = x*cos + rotate(x)*sin).

Each check is fixed by the pages or by mathematics, not by the oracle itself:
the printed rotate() layouts (sglang rope_cache.py), a closed-form worked
example, the identity at position 0, per-pair norm preservation, dependence of
<rope(q,m), rope(k,n)> on m-n only, and the NeoX/GPT-J equivalence under the
dim permutation. A dropped term, a wrong sign, a wrong partner or frequency
index, or swapped cos/sin halves each fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rotate_examples.json")
STYLES = {"neox": oracle.NEOX, "gptj": oracle.GPTJ}


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["neox", "gptj"])
def test_rotate_matches_printed_layout(golden, name):
    g = golden["rotate"][name]
    x = np.array([3.0, 5.0, 7.0, 11.0])
    want = np.array([s * x[i] for s, i in zip(g["sign"], g["index"])])
    assert np.array_equal(oracle.rotate_half(x, 4, STYLES[name]), want)


@pytest.mark.parametrize("name", ["neox", "gptj"])
def test_frequency_index_matches_stage_2_1(golden, name):
    want = golden["freq_index_r8"][name]["index"]
    assert [oracle.freq_index(d, 8, STYLES[name]) for d in range(8)] == want


def _row(angles):
    """A cos/sin table row [cos | sin] in FP32 for the given angles."""
    a = np.asarray(angles, dtype=np.float64)
    return np.concatenate([np.cos(a), np.sin(a)]).astype(np.float32)


def test_worked_example_neox():
    # D = r = 4, theta = 10000: inverse frequencies 10000^(-0/4) = 1 and
    # 10000^(-2/4) = 0.01; at position 1 the angles are 1 and 0.01.
    row = workloads.cos_sin_table(10000.0, 2, 4)[0, 1]
    assert row[0] == np.float32(math.cos(1.0)) and row[1] == np.float32(math.cos(0.01))
    assert row[2] == np.float32(math.sin(1.0)) and row[3] == np.float32(math.sin(0.01))
    c1, c2, s1, s2 = (float(v) for v in row)
    # NeoX pairs (0,2) with frequency 0 and (1,3) with frequency 1
    y = oracle.rope_head_f64(np.array([1.0, 0, 0, 0]), row, 4, oracle.NEOX)
    assert np.array_equal(y, [c1, 0.0, s1, 0.0])
    y = oracle.rope_head_f64(np.array([0, 1.0, 0, 0]), row, 4, oracle.NEOX)
    assert np.array_equal(y, [0.0, c2, 0.0, s2])
    y = oracle.rope_head_f64(np.array([0, 0, 1.0, 0]), row, 4, oracle.NEOX)
    assert np.array_equal(y, [-s1, 0.0, c1, 0.0])
    assert abs(c1 - 0.5403023058681398) < 1e-7 and abs(s1 - 0.8414709848078965) < 1e-7


def test_worked_example_gptj():
    row = workloads.cos_sin_table(10000.0, 2, 4)[0, 1]
    c1, c2, s1, s2 = (float(v) for v in row)
    # GPT-J pairs (0,1) with frequency 0 and (2,3) with frequency 1
    y = oracle.rope_head_f64(np.array([1.0, 0, 0, 0]), row, 4, oracle.GPTJ)
    assert np.array_equal(y, [c1, s1, 0.0, 0.0])
    y = oracle.rope_head_f64(np.array([0, 0, 1.0, 0]), row, 4, oracle.GPTJ)
    assert np.array_equal(y, [0.0, 0.0, c2, s2])
    y = oracle.rope_head_f64(np.array([0, 1.0, 0, 0]), row, 4, oracle.GPTJ)
    assert np.array_equal(y, [-s1, c1, 0.0, 0.0])


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
@pytest.mark.parametrize("D,r", [(64, 64), (128, 128), (128, 64), (256, 96)])
def test_position_zero_is_identity(style, D, r):
    rng = np.random.Generator(np.random.PCG64(7))
    row0 = workloads.cos_sin_table(5e5, 1, r)[0, 0]
    assert np.array_equal(row0, np.concatenate([np.ones(r // 2), np.zeros(r // 2)]).astype(np.float32))
    x = rng.standard_normal(D)
    y = oracle.rope_head_f64(x, row0, r, style)
    assert np.array_equal(y, x)


def _pairs(r, style):
    h = r // 2
    if style == oracle.NEOX:
        return [(i, i + h) for i in range(h)]
    return [(2 * i, 2 * i + 1) for i in range(h)]


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
@pytest.mark.parametrize("D,r", [(128, 128), (128, 64), (64, 32)])
def test_pair_norm_preserved_and_tail_untouched(style, D, r):
    rng = np.random.Generator(np.random.PCG64(11))
    table = workloads.cos_sin_table(5e5, 4096, r)[0]
    for _ in range(200):
        p = int(rng.integers(0, 4096))
        x = rng.standard_normal(D)
        y = oracle.rope_head_f64(x, table[p], r, style)
        for a, b in _pairs(r, style):
            nx = math.hypot(x[a], x[b])
            ny = math.hypot(y[a], y[b])
            assert abs(ny - nx) <= 1e-6 * max(nx, 1e-30)
        assert np.array_equal(y[r:], x[r:])


@pytest.mark.parametrize("style", [oracle.NEOX, oracle.GPTJ])
def test_dot_product_depends_only_on_offset(style):
    D = r = 128
    rng = np.random.Generator(np.random.PCG64(5))
    table = workloads.cos_sin_table(1e4, 2048, r)[0]
    for _ in range(100):
        q = rng.standard_normal(D)
        k = rng.standard_normal(D)
        m, n = (int(v) for v in rng.integers(0, 1024, size=2))
        delta = int(rng.integers(1, 1024))
        lhs = np.dot(oracle.rope_head_f64(q, table[m], r, style),
                     oracle.rope_head_f64(k, table[n], r, style))
        rhs = np.dot(oracle.rope_head_f64(q, table[m + delta], r, style),
                     oracle.rope_head_f64(k, table[n + delta], r, style))
        assert abs(lhs - rhs) <= 1e-5 * np.linalg.norm(q) * np.linalg.norm(k)


@pytest.mark.parametrize("D,r", [(128, 128), (128, 64), (64, 16)])
def test_gptj_equals_neox_under_dim_permutation(D, r):
    """With P moving NeoX dim i to GPT-J dim 2i and NeoX dim i+h to GPT-J dim
    2i+1 (dims >= r fixed): gptj(P x) == P neox(x), exactly."""
    h = r // 2
    perm = np.arange(D)
    for i in range(h):
        perm[2 * i] = i          # GPT-J dim 2i   <- NeoX dim i
        perm[2 * i + 1] = i + h  # GPT-J dim 2i+1 <- NeoX dim i+h
    rng = np.random.Generator(np.random.PCG64(3))
    table = workloads.cos_sin_table(5e5, 512, r)[0]
    for _ in range(50):
        x = rng.standard_normal(D)
        row = table[int(rng.integers(0, 512))]
        neox = oracle.rope_head_f64(x, row, r, oracle.NEOX)
        gptj = oracle.rope_head_f64(x[perm], row, r, oracle.GPTJ)
        assert np.array_equal(gptj, neox[perm])


def test_cos_sin_table_closed_form():
    r = 64
    t = workloads.cos_sin_table(1e4, 300, r)[0]
    for p in (0, 1, 17, 299):
        for i in range(r // 2):
            ang = p * 1e4 ** (-2.0 * i / r)
            assert t[p, i] == np.float32(math.cos(ang))
            assert t[p, r // 2 + i] == np.float32(math.sin(ang))
    c, s = t[:, : r // 2].astype(np.float64), t[:, r // 2:].astype(np.float64)
    assert np.max(np.abs(c * c + s * s - 1.0)) <= 2.0 ** -23
