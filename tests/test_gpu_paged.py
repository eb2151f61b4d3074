"""GPU parity of the paged delta update against the oracle.

Small pools are compared element by element (every skip rule appears: padding
rows, sequences past batchSize, positions past the logical pages, unmapped and
out-of-plane page ids). The full paged workload (a 17.2 GB pool) is checked on
every written row plus a device-side count proving nothing else changed.
"""
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


def _run_gpu(pc, batch_size=None, stream=None):
    import rope_kv_cache_gb300 as rk
    pool = dev_sentinel(pc.pool_shape())
    rk.paged_kv_delta_update(to_dev(pc.k_delta), to_dev(pc.v_delta), pool, to_dev(pc.cos_sin_rows),
                             to_dev(pc.positions), to_dev(pc.seq_ids), to_dev(pc.page_table),
                             batch_size=batch_size, style=pc.style, stream=stream)
    torch.cuda.synchronize()
    return pool


def _check_full(pc, batch_size=None):
    import oracle
    g = to_host_bits(_run_gpu(pc, batch_size))
    want = pc.new_pool()
    pt = pc.page_table if batch_size is None else np.ascontiguousarray(pc.page_table[:batch_size])
    oracle.paged(pc.k_delta, pc.v_delta, want, pc.cos_sin_rows, pc.positions, pc.seq_ids, pt,
                 pc.style)
    return compare(g, want, pool_rotated(want.shape, pc.r), pc.name)


SMALL = [
    # N, B, Hkv, D, r, tpp, mpps, numPages, style
    (300, 4, 2, 64, 64, 16, 32, 128, GPTJ),
    (513, 5, 8, 128, 128, 64, 4, 20, NEOX),
    (97, 3, 1, 256, 128, 8, 16, 48, NEOX),
    (1500, 8, 4, 128, 64, 32, 8, 64, GPTJ),     # >= 1024 rows: two items per thread
    (64, 2, 32, 128, 128, 4, 64, 128, NEOX),    # 32 KV heads: several CTAs per row
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_small_pools(idx):
    N, B, Hkv, D, r, tpp, mpps, P, style = SMALL[idx]
    pc = workloads.make_paged(N, B, Hkv, D, r, tpp, mpps, P, style, 1e4, seed=200 + idx,
                              valid_rows=int(0.9 * N), len_range=(1, min(256, tpp * mpps)),
                              unmapped_frac=0.05, name=f"paged{idx}")
    _check_full(pc)


def test_every_skip_rule():
    """Out-of-plane ids, rows past batchSize and past the logical pages."""
    pc = workloads.make_paged(400, 6, 2, 128, 128, 16, 8, 48, NEOX, 5e5, seed=31,
                              valid_rows=360, len_range=(1, 100), unmapped_frac=0.05,
                              name="skips")
    pt = pc.page_table
    pt[0, 0, :4] = [48, 60, 95, -5]          # V-plane ids / garbage in the K column
    pt[1, 1, :4] = [0, 47, 96, -1]           # K-plane ids / 2*numPages in the V column
    pc.seq_ids[:5] = 6                        # == batchSize: skipped
    pc.positions[5:9] = 8 * 16 + np.arange(4)  # logical page 8 == maxPagesPerSeq
    pc.seq_ids[5:9] = 2
    _check_full(pc)
    # a smaller active batch skips the rows of the trailing sequences
    _check_full(pc, batch_size=4)


def test_empty_rows_is_no_op():
    import rope_kv_cache_gb300 as rk
    pc = workloads.make_paged(0, 2, 2, 64, 64, 16, 4, 8, NEOX, 1e4, seed=1, valid_rows=0,
                              len_range=(0, 0))
    pool = to_dev(pc.new_pool())
    rk.paged_kv_delta_update(to_dev(pc.k_delta), to_dev(pc.v_delta), pool, to_dev(pc.cos_sin_rows),
                             to_dev(pc.positions), to_dev(pc.seq_ids), to_dev(pc.page_table))
    torch.cuda.synchronize()
    assert np.all(to_host_bits(pool) == workloads.SENTINEL)


def test_config_paged_written_rows_and_untouched():
    import oracle
    pc = workloads.config("paged")
    pool = _run_gpu(pc)
    kd, vd, ko, vo = oracle.paged_rows(pc.k_delta, pc.v_delta, pc.cos_sin_rows, pc.positions,
                                       pc.seq_ids, pc.page_table, pc.num_pages,
                                       pc.tokens_per_page, pc.style)
    row = pc.Hkv * pc.D
    flat = pool.view(-1).view(torch.int16)
    rows_idx = torch.arange(row, device=pool.device)
    for dest, out, plane in ((kd, ko, 0), (vd, vo, 1)):
        sel = np.nonzero(dest >= 0)[0]
        idx = torch.as_tensor(dest[sel], device=pool.device)[:, None] + rows_idx[None, :]
        got = flat[idx.reshape(-1)].cpu().numpy().view(np.uint16).reshape(len(sel), pc.Hkv, pc.D)
        want = out[sel]
        rot = (np.arange(pc.D) < pc.r)[None, None, :] if plane == 0 else np.zeros((1, 1, pc.D), bool)
        compare(got, want, rot, f"paged plane {plane}")
    n_written = int((kd >= 0).sum() + (vd >= 0).sum()) * row
    sent = np.uint16(workloads.SENTINEL).view(np.int16).item()
    v = pool.view(torch.int16).view(2 * pc.num_pages, -1)
    count = 0
    for c in range(0, v.shape[0], 4096):
        count += int((v[c:c + 4096] != sent).sum().item())
    assert count == n_written
