"""GPU parity of the DFlash prologue entry points (delta metadata, cos/sin
gather) and of the one-launch fused update, against the oracle; and the fused
launch against the three-launch pipeline it replaces, bit for bit."""
import numpy as np
import pytest

import workloads
from parity import compare, dev_sentinel, pool_rotated, to_dev, to_host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
NEOX, GPTJ = workloads.NEOX, workloads.GPTJ


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rope_kv_cache_gb300 import build
    build.build_library()


def _i32(n):
    return torch.full((n,), 12345, dtype=torch.int32, device="cuda:0")


@pytest.mark.parametrize("B,W", [(1, 1), (3, 4), (128, 128), (7, 300), (1000, 17)])
def test_delta_metadata(B, W):
    import oracle
    import rope_kv_cache_gb300 as rk
    rng = workloads.rng_for(B * 1000 + W)
    old = rng.integers(-5, 40000, size=B).astype(np.int32)
    lens = rng.integers(-2, W + 3, size=B).astype(np.int32)
    pos, seq = _i32(B * W), _i32(B * W)
    rk.dflash_prepare_delta_metadata(to_dev(old), to_dev(lens), W, pos, seq)
    torch.cuda.synchronize()
    o_pos, o_seq = oracle.delta_metadata(old, lens, W)
    assert np.array_equal(pos.cpu().numpy(), o_pos)
    assert np.array_equal(seq.cpu().numpy(), o_seq)


@pytest.mark.parametrize("rows,with_state,r", [(1, False, 128), (3, True, 64), (4, False, 256),
                                               (2, True, 16)])
def test_gather_delta_rope(rows, with_state, r):
    import oracle
    import rope_kv_cache_gb300 as rk
    rng = workloads.rng_for(rows * 10 + r)
    B, N, cap = 6, 999, 500
    src = workloads.cos_sin_table(1e4, cap, r, batch=rows, pos_offset=np.arange(rows) * 77)
    pos = rng.integers(-3, cap + 5, size=N).astype(np.int32)
    seq = rng.integers(-1, B + 2, size=N).astype(np.int32)
    state = rng.integers(-1, rows + 1, size=B).astype(np.int32) if with_state else None
    out = torch.full((N, r), float("nan"), dtype=torch.float32, device="cuda:0")
    rk.dflash_gather_delta_rope(to_dev(src), out, to_dev(pos), to_dev(seq),
                                to_dev(state) if with_state else None, batch_size=B)
    torch.cuda.synchronize()
    want = oracle.gather_delta_rope(src, pos, seq, state, B)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def _run_fused(fc, stream=None):
    import rope_kv_cache_gb300 as rk
    pool = dev_sentinel(fc.pool_shape())
    rk.paged_kv_delta_update_fused(to_dev(fc.k_delta), to_dev(fc.v_delta), pool, to_dev(fc.source),
                                   to_dev(fc.old_lengths), to_dev(fc.delta_lengths),
                                   to_dev(fc.page_table),
                                   to_dev(fc.state) if fc.state is not None else None,
                                   style=fc.style, stream=stream)
    torch.cuda.synchronize()
    return pool


def _run_unfused(fc):
    """The three-launch pipeline on the GPU: metadata, gather, paged update."""
    import rope_kv_cache_gb300 as rk
    N, r = fc.N, fc.r
    pos, seq = _i32(N), _i32(N)
    rk.dflash_prepare_delta_metadata(to_dev(fc.old_lengths), to_dev(fc.delta_lengths), fc.W, pos, seq)
    cs = torch.empty((N, r), dtype=torch.float32, device="cuda:0")
    rk.dflash_gather_delta_rope(to_dev(fc.source), cs, pos, seq,
                                to_dev(fc.state) if fc.state is not None else None, batch_size=fc.B)
    pool = dev_sentinel(fc.pool_shape())
    rk.paged_kv_delta_update(to_dev(fc.k_delta), to_dev(fc.v_delta), pool, cs, pos, seq,
                             to_dev(fc.page_table), style=fc.style)
    torch.cuda.synchronize()
    return pool


SMALL = [
    # B, W, Hkv, D, r, tpp, mpps, numPages, style, source_rows, with_state, cache_capacity
    (5, 6, 2, 64, 64, 4, 8, 40, GPTJ, 3, True, None),
    (9, 33, 8, 128, 128, 16, 8, 72, NEOX, 1, False, None),
    (4, 20, 1, 256, 96, 8, 4, 16, NEOX, 2, False, None),
    (6, 40, 4, 128, 64, 16, 6, 36, GPTJ, 2, True, 50),   # positions past the cos/sin cache
    (40, 32, 8, 128, 128, 64, 2, 80, NEOX, 1, False, None),  # >= 1024 rows
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_fused_matches_oracle_and_pipeline(idx):
    import oracle
    B, W, Hkv, D, r, tpp, mpps, P, style, rows, st, cap = SMALL[idx]
    fc = workloads.make_paged_fused(B, W, Hkv, D, r, tpp, mpps, P, style, 1e4, seed=300 + idx,
                                    len_range=(0, W + 2), unmapped_frac=0.05, source_rows=rows,
                                    with_state=st, cache_capacity=cap, name=f"fused{idx}")
    if st:
        fc.state[0] = -1               # a sequence without a cos/sin row
    g = to_host_bits(_run_fused(fc))
    want = fc.new_pool()
    oracle.paged_fused(fc.k_delta, fc.v_delta, want, fc.source, fc.old_lengths, fc.delta_lengths,
                       fc.W, fc.state, fc.page_table, fc.style)
    compare(g, want, pool_rotated(want.shape, fc.r), fc.name)
    assert np.array_equal(g, to_host_bits(_run_unfused(fc)))


@pytest.mark.parametrize("style", [NEOX, GPTJ])
def test_fused_without_source_rows(style):
    """No cos/sin source rows (the source may then be NULL, as for the
    gather): every row's cos/sin is zero, so rotated K dims are written as
    zeros, exactly as the three-launch pipeline writes them."""
    import oracle
    fc = workloads.make_paged_fused(6, 21, 2, 128, 64, 8, 6, 40, style, 1e4, seed=350 + style,
                                    len_range=(0, 21), unmapped_frac=0.05, name="fused_nosrc")
    fc.source = np.ascontiguousarray(fc.source[:0])
    g = to_host_bits(_run_fused(fc))
    want = fc.new_pool()
    oracle.paged_fused(fc.k_delta, fc.v_delta, want, fc.source, fc.old_lengths, fc.delta_lengths,
                       fc.W, None, fc.page_table, fc.style)
    compare(g, want, pool_rotated(want.shape, fc.r), fc.name)
    assert np.array_equal(g, to_host_bits(_run_unfused(fc)))
    written = want[0] != workloads.SENTINEL
    rot = want[0][..., : fc.r][written[..., : fc.r]].view(np.float16)
    assert written.any() and np.all(rot == 0)            # +0 or -0


def test_config_paged_fused_full():
    """16384 rows into the 17.2 GB pool: every written row against the oracle
    composition, nothing else changed, and bit-identical to the pipeline."""
    import oracle
    fc = workloads.config("paged_fused")
    pool = _run_fused(fc)
    pos, seq = oracle.delta_metadata(fc.old_lengths, fc.delta_lengths, fc.W)
    cs = oracle.gather_delta_rope(fc.source, pos, seq, fc.state, fc.B)
    kd, vd, ko, vo = oracle.paged_rows(fc.k_delta, fc.v_delta, cs, pos, seq, fc.page_table,
                                       fc.num_pages, fc.tokens_per_page, fc.style)
    row = fc.Hkv * fc.D
    flat = pool.view(-1).view(torch.int16)
    ar = torch.arange(row, device=pool.device)
    for dest, out, plane in ((kd, ko, 0), (vd, vo, 1)):
        sel = np.nonzero(dest >= 0)[0]
        idx = torch.as_tensor(dest[sel], device=pool.device)[:, None] + ar[None, :]
        got = flat[idx.reshape(-1)].cpu().numpy().view(np.uint16).reshape(len(sel), fc.Hkv, fc.D)
        rot = (np.arange(fc.D) < fc.r)[None, None, :] if plane == 0 else np.zeros((1, 1, fc.D), bool)
        compare(got, out[sel], rot, f"paged_fused plane {plane}")
    n_written = int((kd >= 0).sum() + (vd >= 0).sum()) * row
    sent = np.uint16(workloads.SENTINEL).view(np.int16).item()
    v = pool.view(torch.int16).view(2 * fc.num_pages, -1)
    count = sum(int((v[c:c + 4096] != sent).sum().item()) for c in range(0, v.shape[0], 4096))
    assert count == n_written
    ref = _run_unfused(fc)
    same = sum(int((pool.view(torch.int16).view(-1)[c:c + (1 << 28)] !=
                    ref.view(torch.int16).view(-1)[c:c + (1 << 28)]).sum().item())
               for c in range(0, pool.numel(), 1 << 28))
    assert same == 0
