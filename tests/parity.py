"""Shared helpers of the GPU parity tests: moving seeded inputs to the device,
calling the binding, and comparing device results with the oracle's.

Comparison rule (element by element):
* every element outside the rotated region (V, dims >= rotaryDim, untouched
  sentinel bytes) must be bit-identical to the oracle's;
* a rotated element is either bit-identical, or both values are finite and
  |gpu - oracle| <= 2^-10 * |oracle| + 1e-6 (+0 and -0 count as equal);
* and where |oracle| >= 2^-6 the two are at most one FP16 ulp apart. Below
  that magnitude the absolute term of the bound governs: a result that cancels
  down to ~1e-4 carries an FP32 rounding error of ~1e-7 from terms of size ~1,
  which is more than one FP16 ulp there (6e-8) yet far inside the bound.
"""
from __future__ import annotations

import contextlib

import numpy as np

try:
    import torch
except ImportError:  # pragma: no cover - torch is present wherever tests run
    torch = None

import workloads

TOL_REL = 2.0 ** -10
TOL_ABS = 1e-6
ULP_RULE_MIN = 2.0 ** -6


_DEVICE = [None]


def dev():
    """The device the helpers move inputs to (cuda:0 unless on_device says)."""
    return _DEVICE[0] or torch.device("cuda:0")


@contextlib.contextmanager
def on_device(device):
    """Run the helpers against `device` instead of cuda:0."""
    _DEVICE[0] = device
    try:
        yield
    finally:
        _DEVICE[0] = None


def to_dev(a: np.ndarray):
    """Host numpy array -> device tensor; FP16 bit arrays become float16 tensors."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev()).view(torch.float16)
    return torch.from_numpy(a).to(dev())


def dev_sentinel(shape):
    """A device FP16 buffer filled with the sentinel bits, made on the device."""
    return torch.full(tuple(shape), workloads.SENTINEL, dtype=torch.int16,
                      device=dev()).view(torch.float16)


def to_host_bits(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ordered(bits: np.ndarray) -> np.ndarray:
    """FP16 bits -> integers ordered like the values (so adjacent values differ by 1)."""
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def compare(got: np.ndarray, want: np.ndarray, rotated: np.ndarray, what: str = "") -> dict:
    """Assert the comparison rule; returns simple statistics."""
    assert got.shape == want.shape, (what, got.shape, want.shape)
    rotated = np.broadcast_to(rotated, got.shape)
    diff = got != want
    exact_bad = diff & ~rotated
    if exact_bad.any():
        idx = np.argwhere(exact_bad)[0]
        raise AssertionError(f"{what}: bit mismatch outside the rotated region at {tuple(idx)}: "
                             f"gpu {got[tuple(idx)]:#06x} oracle {want[tuple(idx)]:#06x} "
                             f"({int(exact_bad.sum())} elements)")
    rd = diff & rotated
    n_diff = int(rd.sum())
    max_ulp = 0
    max_err = 0.0
    if n_diff:
        g = got[rd]
        w = want[rd]
        gv = g.view(np.float16).astype(np.float64)
        wv = w.view(np.float16).astype(np.float64)
        finite = np.isfinite(gv) & np.isfinite(wv)
        if not finite.all():
            i = np.nonzero(~finite)[0][0]
            raise AssertionError(f"{what}: non-finite mismatch gpu {g[i]:#06x} oracle {w[i]:#06x}")
        ulp = np.abs(_ordered(g) - _ordered(w))
        zero_pair = (gv == 0) & (wv == 0)
        ulp = np.where(zero_pair, 0, ulp)
        err = np.abs(gv - wv)
        bad = ((ulp > 1) & (np.abs(wv) >= ULP_RULE_MIN)) | (err > TOL_REL * np.abs(wv) + TOL_ABS)
        if bad.any():
            i = np.nonzero(bad)[0][0]
            raise AssertionError(f"{what}: rotated element off by {ulp[i]} ulp / {err[i]:.3g} "
                                 f"(gpu {gv[i]!r} oracle {wv[i]!r}); {int(bad.sum())} bad")
        big = np.abs(wv) >= ULP_RULE_MIN
        max_ulp = int(ulp[big].max()) if big.any() else 0
        max_err = float(err.max())
    return {"n": int(got.size), "n_diff": n_diff, "max_ulp": max_ulp, "max_err": max_err}


# ----------------------------------------------------------- rotated masks --

def qout_rotated(shape, r):
    return (np.arange(shape[-1]) < r)[None, None, None, :]


def cache_rotated(shape, r):
    plane0 = (np.arange(2) == 0)[None, :, None, None, None]
    return plane0 & (np.arange(shape[-1]) < r)[None, None, None, None, :]


def qkv_rotated(Hq, Hkv, D, r):
    H = Hq + 2 * Hkv
    return ((np.arange(H) < Hq + Hkv)[:, None] & (np.arange(D) < r)[None, :])[None, None]


def pool_rotated(shape, r):
    return (np.arange(2) == 0)[:, None, None, None, None] & \
        (np.arange(shape[-1]) < r)[None, None, None, None, :]


# ------------------------------------------------------------- run a case --

def run_gpu_contiguous(case: workloads.ContiguousCase, stream=None):
    """Run the case's entry point on the device; returns host bit arrays
    (qkv after the call, cache, qOut or None)."""
    import rope_kv_cache_gb300 as rk
    cs = to_dev(case.cos_sin)
    qkv = to_dev(case.qkv)
    cache = to_dev(case.new_cache())
    if case.mode == "packed":
        rk.rope_write_kv_packed(cs, qkv, cache, case.Hq, case.Hkv, case.style, stream=stream)
        qout = None
    else:
        qout = to_dev(case.new_qout())
        end = to_dev(case.end_lens)
        if case.mode == "continuous" and case.norm is not None:
            qw, kw, eps = case.norm
            rk.rope_write_kv_continuous_qknorm(cs, end, qkv, cache, qout, to_dev(qw), to_dev(kw),
                                               eps, case.Hq, case.Hkv, case.style, stream=stream)
        elif case.mode == "continuous":
            rk.rope_write_kv_continuous(cs, end, qkv, cache, qout, case.Hq, case.Hkv, case.style,
                                        stream=stream)
        else:
            rk.rope_write_kv_tree(cs, end, to_dev(case.pos_ids), qkv, cache, qout, case.Hq,
                                  case.Hkv, case.style, stream=stream)
    torch.cuda.synchronize(dev())
    return to_host_bits(qkv), to_host_bits(cache), (to_host_bits(qout) if qout is not None else None)


def run_oracle_contiguous(case: workloads.ContiguousCase):
    import oracle
    qkv = case.qkv.copy()
    cache = case.new_cache()
    if case.mode == "packed":
        oracle.packed(case.cos_sin, qkv, cache, case.Hq, case.Hkv, case.style)
        return qkv, cache, None
    qout = case.new_qout()
    if case.mode == "continuous" and case.norm is not None:
        qw, kw, eps = case.norm
        oracle.continuous_qknorm(case.cos_sin, case.end_lens, qkv, cache, qout, qw, kw, eps,
                                 case.Hq, case.Hkv, case.style)
    elif case.mode == "continuous":
        oracle.continuous(case.cos_sin, case.end_lens, qkv, cache, qout, case.Hq, case.Hkv,
                          case.style)
    else:
        oracle.tree(case.cos_sin, case.end_lens, case.pos_ids, qkv, cache, qout, case.Hq,
                    case.Hkv, case.style)
    return qkv, cache, qout


def check_contiguous(case: workloads.ContiguousCase, stream=None) -> dict:
    g_qkv, g_cache, g_qout = run_gpu_contiguous(case, stream)
    o_qkv, o_cache, o_qout = run_oracle_contiguous(case)
    stats = {}
    # a normalized call computes every Q/K dim (none is a bit copy)
    r = case.D if case.norm is not None else case.r
    if case.mode == "packed":
        stats["qkv"] = compare(g_qkv, o_qkv, qkv_rotated(case.Hq, case.Hkv, case.D, case.r),
                               f"{case.name} qkv")
    else:
        assert np.array_equal(g_qkv, case.qkv), f"{case.name}: qkv modified by a read-only call"
        stats["qout"] = compare(g_qout, o_qout, qout_rotated(o_qout.shape, r),
                                f"{case.name} qOut")
    stats["cache"] = compare(g_cache, o_cache, cache_rotated(o_cache.shape, r),
                             f"{case.name} cache")
    return stats
