"""Benchmark of the fused RoPE + KV-cache write on GB300.

One step = one call of the entry point over one batch of the workload (one
kernel launch). The headline workload is the Llama-3-8B-shaped prefill
(B=4, S=2048, Hq=32, Hkv=8, D=r=128, NeoX, continuous cache of 8192 slots);
decode, tree, paged and the tiny packed case are measured in the same run and
reported under "workloads".

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA
graphs, bracketed by a barrier and torch.cuda.synchronize(); CUDA events on the
launching stream. Consecutive steps cycle through a ring of distinct input sets
(and distinct cache slots / pages) whose footprint exceeds twice the L2 size,
so no step reads what the previous one left in L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 (torchrun) every rank runs its own replica of the workload on its
GPU (the path has no exchange step: weak scaling, no collective on the data
path); value is the whole-job rate over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fused RoPE+KV-write tokens/s and effective HBM GB/s (% of GB300 peak)"
HEADLINE = "prefill"
EXTRA = ("decode", "decode_floor", "tree", "paged", "packed_tiny", "paged_fused", "paged_fused_3launch",
         "slotmap_prefill", "slotmap_decode", "prefill_qknorm", "decode_qknorm", "prefill_fp8",
         "decode_fp8")
NOMINAL_HBM_GBS = 8000.0
CACHE_RING_BUDGET = 16 * 2 ** 30  # device bytes for one contiguous cache per ring set
FALLBACK_HBM_GBS = 6800.0

DESCR = {
    "packed_tiny": "packed in-place, empty cache: B=1 S=16 Hq=4 Hkv=2 D=r=64 NeoX theta=1e4",
    "prefill": "Llama-3-8B-shaped prefill, continuous cache: B=4 S=2048 Hq=32 Hkv=8 D=r=128 "
               "NeoX theta=5e5, capacity 8192, start in [0,4096]",
    "decode": "decode, continuous cache: B=256 S=1 Hq=32 Hkv=8 D=r=128 NeoX theta=5e5, "
              "cache [256,2,8,8192,128], end lengths in [1,8192]",
    "tree": "tree speculative decoding: B=64 S=64 Hq=32 Hkv=8 D=128 r=64 GPT-J theta=1e4, "
            "depth 0..6, base in [128,4000], capacity 4096",
    "paged": "paged delta update: 16384 rows (15565 valid) over B=128, Hkv=8 D=r=128 NeoX, "
             "64 tokens/page, 512 pages/seq, 65536 pages per plane, 2% unmapped",
    "paged_fused": "DFlash step in one launch (delta metadata + cos/sin gather + paged update): "
                   "B=128 x deltaWidth 128 rows, lengths in [1,128], Hkv=8 D=r=128 NeoX, "
                   "64 tokens/page, 512 pages/seq, 65536 pages per plane",
    "paged_fused_3launch": "the same DFlash step as three launches (metadata, gather, update)",
    "slotmap_prefill": "the prefill behind the sglang-style interface: separate Q/K/V views of a "
                       "packed buffer, per-token positions and flat slots, block size 64, "
                       "16384 blocks",
    "slotmap_decode": "256 one-token decodes behind the sglang-style interface",
    "prefill_qknorm": "the prefill with pre-RoPE QK RMS norm fused in (weights [128], eps 1e-6)",
    "decode_qknorm": "the decode with pre-RoPE QK RMS norm fused in (weights [128], eps 1e-6)",
    "prefill_fp8": "the prefill with an E4M3 KV cache (k_scale 0.05, v_scale 0.04)",
    "decode_fp8": "the decode with an E4M3 KV cache (k_scale 0.05, v_scale 0.04)",
    "decode_floor": "the floor of one dependent decode-sized launch: a plain copy of decode's "
                    "bytes in decode's grid (512 CTAs x 96 threads, four 16-byte vectors per "
                    "thread), with decode's L2 prefetch, dependent-launch attribute and residency "
                    "cap, timed like decode",
    "decode_c1024": "decode as above with cache capacity 1024 (profiler-sized twin)",
    "paged_p8192": "paged as above with 64 pages/seq and 8192 pages per plane (profiler-sized twin)",
    "paged_fused_p8192": "paged_fused with 64 pages/seq and 8192 pages per plane (profiler-sized twin)",
    "slotmap_prefill_b4096": "slotmap_prefill with 4096 blocks per cache (profiler-sized twin)",
    "slotmap_decode_b4096": "slotmap_decode with 4096 blocks per cache (profiler-sized twin)",
    "decode_qknorm_c1024": "decode_qknorm with cache capacity 1024 (profiler-sized twin)",
    "decode_fp8_c1024": "decode_fp8 with cache capacity 1024 (profiler-sized twin)",
    "paged_fused_p8192_3launch": "paged_fused_p8192 as three launches (profiler-sized twin)",
}


# ------------------------------------------------------------------ utils --

def max_over_ranks(value: float, dist, device) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: int, steps: int, max_seconds: float) -> float:
    """Weak scaling: every rank processes its own replica of the workload, so
    the job's rate is all ranks' units over the slowest rank's time."""
    return world * units_per_rank * steps / max_seconds


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, the blank space of each line
    collapsed and blank lines dropped: a comment edit leaves it unchanged,
    any edit of the code (string literals, such as inline PTX, included)
    changes it."""
    out = []
    i, n = 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    lines = (" ".join(line.split()) for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


KERNEL_SOURCES = ("rope_kv_cache_gb300/csrc/ropekv_kernels.cuh",
                  "rope_kv_cache_gb300/csrc/ropekv_api.cu",
                  "rope_kv_cache_gb300/csrc/ropekv_floor.cu")


def source_sha():
    """Hash of the kernel sources' code (comments and blank space aside): the
    key that ties a profile capture to the kernels it measured."""
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode("utf-8"))
        h.update(b"\0")
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha()
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload and parts[3] == sha:
            return int(float(parts[2]))
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in a thread."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "n_samples": 0}
        inside = [p for t, p in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        note = "during the timed region"
        if len(inside) < 3:
            # short timed region: take the samples closest to it
            near = sorted(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[:5]
            inside = [p for _, p in near]
            note = "nearest samples (timed region shorter than the sampling interval)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "n_samples": len(inside), "window": note}


# --------------------------------------------------------- device workload --

class DeviceWorkload:
    """A workload resident in HBM: a ring of per-step input sets plus the
    shared cache / pool, and one bound call per ring slot."""

    def __init__(self, name: str, device, l2_bytes: int):
        import torch
        import rope_kv_cache_gb300 as rk
        self.torch = torch
        self.rk = rk
        self.name = name
        self.device = device
        self.three_launch = name.endswith("_3launch")
        self.case = workloads.config(name[: -len("_3launch")] if self.three_launch else name)
        self.paged = isinstance(self.case, workloads.PagedCase)
        self.fused = isinstance(self.case, workloads.PagedFusedCase)
        self.slotmap = isinstance(self.case, workloads.SlotMapCase)
        c = self.case
        if self.paged or self.fused:
            self.tokens = c.valid_rows
        else:
            self.tokens = c.tokens
        self.bytes = c.algorithmic_bytes()
        self.ring = max(2, min(96, math.ceil(2 * l2_bytes / max(self.bytes, 1))))
        t = lambda a: self._dev(a)
        self.sets = []
        if self.paged:
            self.pool = self._sentinel(c.pool_shape())
            k_base, v_base = t(c.k_delta), t(c.v_delta)
            cs, pos, seq = t(c.cos_sin_rows), t(c.positions), t(c.seq_ids)
            for k in range(self.ring):
                pt = t(workloads.step_variant(c, k))
                self.sets.append(dict(k=k_base.clone() if k else k_base,
                                      v=v_base.clone() if k else v_base,
                                      cs=cs.clone() if k else cs, pos=pos, seq=seq, pt=pt))
            self.bytes = int(np.mean([self._variant_bytes(k) for k in range(self.ring)]))
        elif self.fused:
            self.pool = self._sentinel(c.pool_shape())
            self.source = t(c.source)
            self.lens = t(c.delta_lengths)
            self.state = t(c.state) if c.state is not None else None
            k_base, v_base = t(c.k_delta), t(c.v_delta)
            for k in range(self.ring):
                old, pt = workloads.step_variant(c, k)
                st = dict(k=k_base.clone() if k else k_base, v=v_base.clone() if k else v_base,
                          old=t(old), pt=t(pt))
                if self.three_launch:
                    # the pipeline's intermediate arrays (owned by the caller)
                    st["pos"] = torch.empty(c.N, dtype=torch.int32, device=device)
                    st["seq"] = torch.empty(c.N, dtype=torch.int32, device=device)
                    st["cs"] = torch.empty((c.N, c.r), dtype=torch.float32, device=device)
                self.sets.append(st)
            self.bytes = int(np.mean([self._variant_bytes(k) for k in range(self.ring)]))
        elif self.slotmap:
            self.cos_sin = t(c.cos_sin)
            self.kc = self._sentinel(c.cache_shape())
            self.vc = self._sentinel(c.cache_shape())
            qkv_base = t(c.qkv)
            for k in range(self.ring):
                pos, slots = workloads.step_variant(c, k)
                self.sets.append(dict(qkv=qkv_base.clone() if k else qkv_base, pos=t(pos),
                                      slots=t(slots), qout=self._sentinel((c.T, c.Hq, c.D))))
        else:
            self.cos_sin = t(c.cos_sin)
            self.norm = None
            if c.norm is not None:
                self.norm = (t(c.norm[0]), t(c.norm[1]), float(c.norm[2]))
            self.fp8 = None
            if c.fp8_scales is not None:
                self.fp8 = tuple(torch.tensor([v], dtype=torch.float32, device=device)
                                 for v in c.fp8_scales)

            def new_cache():
                if c.fp8_scales is not None:
                    return torch.full((c.B, 2, c.Hkv, c.cap, c.D), workloads.SENTINEL8,
                                      dtype=torch.uint8, device=device)
                return (t(c.new_cache()) if c.cache_init == "zero"
                        else self._sentinel((c.B, 2, c.Hkv, c.cap, c.D)))
            # One cache per ring set where they fit, as the layers of a model
            # each write their own: no step rewrites slots that the previous
            # step left in L2. A shared cache (the 8.6 GB decode cache) is only
            # used where the sets' slots almost never meet (one random slot per
            # sequence).
            cache_bytes = c.B * 2 * c.Hkv * c.cap * c.D * (1 if c.fp8_scales is not None else 2)
            self.caches_per_set = self.ring * cache_bytes <= CACHE_RING_BUDGET
            self.cache = new_cache()
            qkv_base = t(c.qkv)
            for k in range(self.ring):
                end, pos = workloads.step_variant(c, k)
                s = dict(qkv=qkv_base.clone() if k else qkv_base)
                s["cache"] = new_cache() if (k and self.caches_per_set) else self.cache
                if c.mode != "packed":
                    s["end"] = t(end)
                    s["qout"] = self._sentinel((c.B, c.S, c.Hq, c.D))
                    if c.mode == "tree":
                        s["pos"] = t(pos)
                self.sets.append(s)
        torch.cuda.synchronize(device)

    def _dev(self, a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return self.torch.from_numpy(a.view(np.int16)).to(self.device).view(self.torch.float16)
        return self.torch.from_numpy(a).to(self.device)

    def _sentinel(self, shape):
        torch = self.torch
        return torch.full(shape, workloads.SENTINEL, dtype=torch.int16,
                          device=self.device).view(torch.float16)

    def _variant_bytes(self, k):
        c = self.case
        saved = (c.page_table, getattr(c, "old_lengths", None))
        v = workloads.step_variant(c, k)
        if self.fused:
            c.old_lengths, c.page_table = v
        else:
            c.page_table = v
        try:
            return c.algorithmic_bytes()
        finally:
            c.page_table = saved[0]
            if self.fused:
                c.old_lengths = saved[1]

    def footprint(self):
        return self.ring * self.bytes

    def call(self, k: int, stream):
        c, s, rk = self.case, self.sets[k % self.ring], self.rk
        if self.fused and self.three_launch:
            rk.dflash_prepare_delta_metadata(s["old"], self.lens, c.W, s["pos"], s["seq"],
                                             stream=stream)
            rk.dflash_gather_delta_rope(self.source, s["cs"], s["pos"], s["seq"], self.state,
                                        batch_size=c.B, stream=stream)
            rk.paged_kv_delta_update(s["k"], s["v"], self.pool, s["cs"], s["pos"], s["seq"],
                                     s["pt"], style=c.style, stream=stream)
        elif self.slotmap:
            qkv = s["qkv"]
            Hq, Hkv = c.Hq, c.Hkv
            rk.rope_write_kv_slot_mapping(self.cos_sin, s["pos"], qkv[:, :Hq], qkv[:, Hq:Hq + Hkv],
                                          qkv[:, Hq + Hkv:], s["slots"], self.kc, self.vc,
                                          s["qout"], None, style=c.style, stream=stream)
        elif self.fused:
            rk.paged_kv_delta_update_fused(s["k"], s["v"], self.pool, self.source, s["old"],
                                           self.lens, s["pt"], self.state, style=c.style,
                                           stream=stream)
        elif self.paged:
            rk.paged_kv_delta_update(s["k"], s["v"], self.pool, s["cs"], s["pos"], s["seq"],
                                     s["pt"], style=c.style, stream=stream)
        elif c.mode == "packed":
            rk.rope_write_kv_packed(self.cos_sin, s["qkv"], s["cache"], c.Hq, c.Hkv, c.style,
                                    stream=stream)
        elif c.mode == "tree":
            rk.rope_write_kv_tree(self.cos_sin, s["end"], s["pos"], s["qkv"], s["cache"],
                                  s["qout"], c.Hq, c.Hkv, c.style, stream=stream)
        elif self.fp8 is not None:
            rk.rope_write_kv_continuous_fp8(self.cos_sin, s["end"], s["qkv"], s["cache"],
                                            s["qout"], self.fp8[0], self.fp8[1], c.Hq, c.Hkv,
                                            c.style, stream=stream)
        elif self.norm is not None:
            qw, kw, eps = self.norm
            rk.rope_write_kv_continuous_qknorm(self.cos_sin, s["end"], s["qkv"], s["cache"],
                                               s["qout"], qw, kw, eps, c.Hq, c.Hkv, c.style,
                                               stream=stream)
        else:
            rk.rope_write_kv_continuous(self.cos_sin, s["end"], s["qkv"], s["cache"], s["qout"],
                                        c.Hq, c.Hkv, c.style, stream=stream)


class FloorWorkload:
    """The decode floor (include/ropekv_floor.h): per step one copy of the
    decode call's bytes in the decode call's grid -- two CTAs of 96 threads per
    token, 512 in all, four 16-byte vectors per thread, read and written --
    through a ring of source/destination buffers larger than twice the L2."""
    THREADS = 96
    CTAS = 512

    def __init__(self, name: str, device, l2_bytes: int):
        import torch
        import rope_kv_cache_gb300 as rk
        self.torch, self.rk, self.name, self.device = torch, rk, name, device
        self.three_launch = self.paged = self.fused = self.slotmap = False
        self.copy_bytes = self.CTAS * self.THREADS * 4 * 16
        self.bytes = 2 * self.copy_bytes
        self.tokens = self.CTAS
        self.ring = max(2, min(96, math.ceil(2 * l2_bytes / self.bytes)))
        n = self.copy_bytes // 2
        self.sets = [(torch.randint(-2 ** 15, 2 ** 15, (n,), dtype=torch.int16, device=device),
                      torch.empty(n, dtype=torch.int16, device=device)) for _ in range(self.ring)]
        torch.cuda.synchronize(device)

    def call(self, k: int, stream):
        src, dst = self.sets[k % self.ring]
        self.rk.ropekv_floor_copy(src, dst, self.THREADS, True, stream=stream)


def make_workload(name: str, device, l2_bytes: int):
    if name == "decode_floor":
        return FloorWorkload(name, device, l2_bytes)
    return DeviceWorkload(name, device, l2_bytes)


def make_graphs(wl: DeviceWorkload, steps: int, stream, chunk: int = 256):
    """CUDA graphs holding exactly `steps` launches: full chunks plus a tail."""
    torch = wl.torch
    graphs = []
    k = 0
    while k < steps:
        n = min(chunk, steps - k)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                wl.call(k + j, torch.cuda.current_stream())
        graphs.append(g)
        k += n
    return graphs


# ~0.2 ms at GB300's 2.07 GHz SM clock: longer than submitting a graph takes.
QUEUE_LEAD_CYCLES = 400_000


def time_steps(wl: DeviceWorkload, steps: int, warmup: int, stream, barrier=None):
    """Warm up, then time exactly `steps` launches; returns (seconds, t0, t1)."""
    torch = wl.torch
    with torch.cuda.stream(stream):
        for k in range(warmup):
            wl.call(k, stream)
    torch.cuda.synchronize(wl.device)
    graphs = make_graphs(wl, steps, stream)
    # CUDAGraph.replay() launches on torch's current stream: make it `stream`,
    # the stream the events are recorded on.
    with torch.cuda.stream(stream):
        # untimed replays: upload the graphs and bring the clocks up
        spin_end = time.time() + 0.3
        while True:
            for g in graphs:
                g.replay()
            torch.cuda.synchronize(wl.device)
            if time.time() >= spin_end:
                break
        for attempt in range(3):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            if barrier:
                barrier()
            torch.cuda.synchronize(wl.device)
            t0 = time.time()
            # Keep the stream busy (a bounded sleep kernel, before the start
            # event) while the host submits the graphs, so that the timed
            # region holds the launches' GPU time and not the GPU idling
            # until the first graph has been submitted.
            torch.cuda._sleep(QUEUE_LEAD_CYCLES)
            start.record(stream)
            for g in graphs:
                g.replay()
            end.record(stream)
            torch.cuda.synchronize(wl.device)
            t1 = time.time()
            sec = start.elapsed_time(end) / 1e3
            # The host clock around the same region must agree with the device
            # clock: events recorded on a stream the work does not run on read
            # near zero. (A host stall only lengthens the wall time; such a
            # region is timed again.)
            wall = t1 - t0
            if wall >= 0.9 * sec and not (wall > 0.05 and sec < 0.5 * wall):
                break
            if wall > 0.05 and sec < 0.05 * wall or attempt == 2:
                raise RuntimeError(f"event time {sec:.6f}s disagrees with wall time {wall:.6f}s")
    if barrier:
        barrier()
    return sec, t0, t1


def e2e_contiguous(wl: DeviceWorkload, steps: int):
    """End to end through the public API with host buffers.

    Every step copies its inputs (QKV, end lengths, tree positions) from pinned
    host memory to the device, launches the entry point, and copies its output
    (qOut; the rotated QKV for the packed call) back to pinned host memory; the
    cache stays resident on the device. Steps are software-pipelined over two
    device buffer sets and three streams, so the host-to-device copy of step k+1
    and the device-to-host copy of step k-1 overlap the kernel of step k.
    """
    torch = wl.torch
    c = wl.case
    dev = wl.device
    h_in = {"qkv": torch.from_numpy(c.qkv.view(np.int16)).pin_memory()}
    if c.mode != "packed":
        h_in["end"] = torch.from_numpy(np.ascontiguousarray(c.end_lens)).pin_memory()
    if c.mode == "tree":
        h_in["pos"] = torch.from_numpy(np.ascontiguousarray(c.pos_ids)).pin_memory()
    out_shape = tuple(c.qkv.shape) if c.mode == "packed" else (c.B, c.S, c.Hq, c.D)
    h_out = torch.empty(out_shape, dtype=torch.int16).pin_memory()
    d_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in h_in.items()}
            for _ in range(2)]
    # the packed call rotates its input in place: its output buffer is the input
    d_out = [d["qkv"] if c.mode == "packed" else
             torch.empty(out_shape, dtype=torch.int16, device=dev) for d in d_in]
    s_h2d, s_cmp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "cmp", "d2h")}
    rk = wl.rk

    def step(k):
        j = k % 2
        with torch.cuda.stream(s_h2d):
            if k >= 2:
                s_h2d.wait_event(ev["cmp"][j])      # kernel k-2 has read set j
                s_h2d.wait_event(ev["d2h"][j])      # and its output has been copied out
            for name, h in h_in.items():
                d_in[j][name].copy_(h, non_blocking=True)
            ev["h2d"][j].record(s_h2d)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev["h2d"][j])
            if k >= 2:
                s_cmp.wait_event(ev["d2h"][j])      # output of step k-2 copied out
            x = d_in[j]
            if c.mode == "packed":
                rk.rope_write_kv_packed(wl.cos_sin, x["qkv"].view(torch.float16), wl.cache,
                                        c.Hq, c.Hkv, c.style, stream=s_cmp)
            elif c.mode == "tree":
                rk.rope_write_kv_tree(wl.cos_sin, x["end"], x["pos"], x["qkv"].view(torch.float16),
                                      wl.cache, d_out[j].view(torch.float16), c.Hq, c.Hkv,
                                      c.style, stream=s_cmp)
            else:
                rk.rope_write_kv_continuous(wl.cos_sin, x["end"], x["qkv"].view(torch.float16),
                                            wl.cache, d_out[j].view(torch.float16), c.Hq, c.Hkv,
                                            c.style, stream=s_cmp)
            ev["cmp"][j].record(s_cmp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["cmp"][j])
            h_out.copy_(d_out[j], non_blocking=True)
            ev["d2h"][j].record(s_d2h)

    for k in range(3):
        step(k)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_h2d)
    for k in range(steps):
        step(k)
    s_d2h.wait_event(ev["d2h"][(steps - 1) % 2])
    end.record(s_d2h)
    torch.cuda.synchronize(dev)
    sec = start.elapsed_time(end) / 1e3
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = h_out.numel() * h_out.element_size()
    return {"value": c.tokens * steps / sec, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": sec * 1e3 / steps,
            "pipelined": "H2D of step k+1 and D2H of step k-1 overlap the kernel of step k"}


# ------------------------------------------------------------ CPU oracle --
#
# The CPU baseline is the oracle as it stands, timed on the host cores. A
# workload is cut into small independent oracle calls ("units") whose outputs
# land in small host buffers, so that no 8.6 GB cache or 17 GB pool is
# allocated on the host; the arithmetic per token is the oracle's, unchanged:
#   * contiguous-cache calls: one chunk of one sequence as a B = 1 call, with
#     the chunk's own slots and positions (the end length shifted to match);
#   * paged update: a chunk of delta rows through oracle.paged_rows (the
#     destinations and values; the pool write is a copy of those values);
#   * fused DFlash step: one sequence through oracle.delta_metadata,
#     oracle.gather_delta_rope and oracle.paged_rows (the oracle's own
#     composition of the three steps, without the pool);
#   * slot mapping: a chunk of tokens, their slots renumbered into a
#     chunk-sized cache.
# The oracle is single-threaded; all cores are used by running independent
# units in one spawned process per core.

def _oracle_base_name(name: str) -> str:
    return name[: -len("_3launch")] if name.endswith("_3launch") else name


class OracleUnits:
    """A workload's inputs cut into oracle calls of about `chunk` tokens.
    Each call returns its outputs; `meta[k]` says what unit k covers (the
    tests check the units against the oracle's call on the whole case)."""

    def __init__(self, name: str, chunk: int = 128, case=None):
        self.name = name
        c = case if case is not None else workloads.config(_oracle_base_name(name))
        self.case = c
        self.calls = []          # (callable, tokens it processes)
        self.meta = []
        if isinstance(c, workloads.PagedCase):
            kw, vw = c.plane_written()
            valid = kw | vw
            for t0 in range(0, c.N, chunk):
                sl = slice(t0, min(c.N, t0 + chunk))
                args = (np.ascontiguousarray(c.k_delta[sl]), np.ascontiguousarray(c.v_delta[sl]),
                        np.ascontiguousarray(c.cos_sin_rows[sl]),
                        np.ascontiguousarray(c.positions[sl]),
                        np.ascontiguousarray(c.seq_ids[sl]))
                self.calls.append((self._paged_call(args), int(valid[sl].sum())))
                self.meta.append(("rows", sl.start, sl.stop - sl.start))
            self.units_total = c.valid_rows
        elif isinstance(c, workloads.PagedFusedCase):
            kw, vw = c.plane_written()
            valid = (kw | vw).reshape(c.B, c.W)
            for b in range(c.B):
                self.calls.append((self._fused_call(b), int(valid[b].sum())))
                self.meta.append(("sequence", b))
            self.units_total = c.valid_rows
        elif isinstance(c, workloads.SlotMapCase):
            for t0 in range(0, c.T, chunk):
                n = min(c.T, t0 + chunk) - t0
                self.calls.append((self._slotmap_call(t0, n), n))
                self.meta.append(("tokens", t0, n))
            self.units_total = c.T
        else:
            nb = c.B if c.mode == "packed" else 1   # the packed call runs whole
            self._cache = (np.zeros((nb, 2, c.Hkv, c.cap, c.D), dtype=np.uint8)
                           if c.fp8_scales is not None else
                           np.zeros((nb, 2, c.Hkv, c.cap, c.D), dtype=np.uint16))
            if c.mode == "packed":
                self.calls.append((self._packed_call(), c.tokens))
                self.meta.append(("all",))
            else:
                n = min(chunk, c.S)
                self._qout = np.zeros((1, n, c.Hq, c.D), dtype=np.uint16)
                for b in range(c.B):
                    for s0 in range(0, c.S, n):
                        m = min(c.S, s0 + n) - s0
                        self.calls.append((self._contiguous_call(b, s0, m), m))
                        self.meta.append(("chunk", b, s0, m))
            self.units_total = c.tokens
        self.bytes_per_unit = c.algorithmic_bytes() / max(1, self.units_total)

    def _contiguous_call(self, b, s0, m):
        import oracle
        c = self.case
        qkv = np.ascontiguousarray(c.qkv[b:b + 1, s0:s0 + m])
        end = np.array([int(c.end_lens[b]) - c.S + s0 + m], dtype=np.int32)
        pos = np.ascontiguousarray(c.pos_ids[b:b + 1, s0:s0 + m]) if c.mode == "tree" else None
        qout = self._qout[:, :m] if m == self._qout.shape[1] else np.zeros(
            (1, m, c.Hq, c.D), dtype=np.uint16)
        cache = self._cache

        def run():
            if c.mode == "tree":
                oracle.tree(c.cos_sin, end, pos, qkv, cache, qout, c.Hq, c.Hkv, c.style)
            elif c.norm is not None:
                qw, kw, eps = c.norm
                oracle.continuous_qknorm(c.cos_sin, end, qkv, cache, qout, qw, kw, eps, c.Hq,
                                         c.Hkv, c.style)
            elif c.fp8_scales is not None:
                oracle.continuous_fp8(c.cos_sin, end, qkv, cache, qout, c.fp8_scales[0],
                                      c.fp8_scales[1], c.Hq, c.Hkv, c.style)
            else:
                oracle.continuous(c.cos_sin, end, qkv, cache, qout, c.Hq, c.Hkv, c.style)
            return qout, cache
        return run

    def _packed_call(self):
        import oracle
        c = self.case
        qkv = c.qkv.copy()

        def run():
            oracle.packed(c.cos_sin, qkv, self._cache, c.Hq, c.Hkv, c.style)
            return qkv, self._cache
        return run

    def _paged_call(self, args):
        import oracle
        c = self.case
        k, v, cs, pos, seq = args

        def run():
            return oracle.paged_rows(k, v, cs, pos, seq, c.page_table, c.num_pages,
                                     c.tokens_per_page, c.style)
        return run

    def _fused_call(self, b):
        import oracle
        c = self.case
        W = c.W
        old = np.ascontiguousarray(c.old_lengths[b:b + 1])
        lens = np.ascontiguousarray(c.delta_lengths[b:b + 1])
        state = np.ascontiguousarray(c.state[b:b + 1]) if c.state is not None else None
        table = np.ascontiguousarray(c.page_table[b:b + 1])
        k = np.ascontiguousarray(c.k_delta[b * W:(b + 1) * W])
        v = np.ascontiguousarray(c.v_delta[b * W:(b + 1) * W])

        def run():
            pos, seq = oracle.delta_metadata(old, lens, W)
            cs = oracle.gather_delta_rope(c.source, pos, seq, state, 1)
            return oracle.paged_rows(k, v, cs, pos, seq, table, c.num_pages, c.tokens_per_page,
                                     c.style)
        return run

    def _slotmap_call(self, t0, n):
        import oracle
        c = self.case
        qkv = np.ascontiguousarray(c.qkv[t0:t0 + n])
        pos = np.ascontiguousarray(c.positions[t0:t0 + n])
        slots = np.where(c.slots[t0:t0 + n] >= 0, np.arange(n), -1).astype(np.int64)
        blocks = -(-n // c.block_size)
        kc = np.zeros((blocks, c.block_size, c.Hkv, c.D), dtype=np.uint16)
        vc = np.zeros_like(kc)
        qout = np.zeros((n, c.Hq, c.D), dtype=np.uint16)
        Hq, Hkv = c.Hq, c.Hkv

        def run():
            oracle.slot_mapping(c.cos_sin, pos, qkv[:, :Hq], qkv[:, Hq:Hq + Hkv],
                                qkv[:, Hq + Hkv:], slots, kc, vc, qout, None, c.style)
            return qout, kc, vc, slots
        return run

    def run_units(self, first: int, count: int = 0, budget_s: float = 0.0):
        """Run units first, first+1, ... (wrapping): `count` of them, or as many
        as `budget_s` seconds allow (at least one). Returns (tokens, seconds)."""
        done, k = 0, 0
        n = len(self.calls)
        t0 = time.perf_counter()
        while True:
            fn, toks = self.calls[(first + k) % n]
            fn()
            done += toks
            k += 1
            if (count and k >= count) or (not count and time.perf_counter() - t0 >= budget_s):
                break
        return done, time.perf_counter() - t0


_W = {}


def _oracle_worker(job):
    """Pool worker: (name, chunk, first unit, count, budget) -> (tokens, seconds).
    Keeps the last workload's units, so that consecutive jobs reuse them."""
    name, chunk, first, count, budget_s = job
    key = (name, chunk)
    if _W.get("key") != key:
        import oracle
        oracle.build()
        _W.clear()
        _W["units"] = OracleUnits(name, chunk)
        _W["key"] = key
    return _W["units"].run_units(first, count, budget_s)


def oracle_process_pool():
    """One spawn-started process per host core (spawn: nothing of the parent's
    CUDA state is inherited)."""
    import multiprocessing
    import oracle
    oracle.build()
    procs = max(1, os.cpu_count() or 1)
    return multiprocessing.get_context("spawn").Pool(procs), procs


def oracle_rates(names, single_s: float, parallel_s: float, pool, procs) -> dict:
    """For every workload: the oracle's single-thread rate (this process) and
    its all-core rate (the sum of the pool processes' own rates)."""
    out = {}
    for name in names:
        units = OracleUnits(name)
        units.run_units(0, count=1)                       # warm-up
        tok1, sec1 = units.run_units(1, budget_s=single_s)
        n = len(units.calls)
        stride = max(1, n // procs)
        pool.map(_oracle_worker, [(name, 128, (j * stride) % n, 1, 0.0) for j in range(procs)])
        res = pool.map(_oracle_worker, [(name, 128, (j * stride + 1) % n, 0, parallel_s)
                                        for j in range(procs)])
        rate = sum(d / t for d, t in res)
        out[name] = {
            "value": rate, "unit": "tokens/s", "cores": procs, "kind": "oracle",
            "effective_gbs": rate * units.bytes_per_unit / 1e9,
            "sample": f"{procs} spawned processes, each running oracle calls of <= 128 tokens "
                      f"(rows) of this workload for {parallel_s:g} s "
                      f"({sum(d for d, _ in res)} tokens in all); value = sum of the "
                      f"processes' rates",
            "single_thread": {"value": tok1 / sec1, "cores": 1,
                              "effective_gbs": tok1 / sec1 * units.bytes_per_unit / 1e9,
                              "sample": f"{tok1} tokens in {sec1:.2f} s"},
        }
        del units
    return out


def run_reference(args):
    """The reference arm: the CPU oracle as it stands on the headline workload,
    one spawned process per host core; every step, each process runs one
    oracle call on its own chunk of a prefill sequence, the chunk sized so
    that warm-up and timed steps take about a minute."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_tok_s = 1.0 / 6000.0
    chunk = int(max(1, min(2048, 60.0 / per_tok_s / max(1, args.steps + args.warmup))))
    pool, procs = oracle_process_pool()
    try:
        n_units = len(OracleUnits(HEADLINE, chunk).calls)
        done = []

        def step(k):
            res = pool.map(_oracle_worker, [(HEADLINE, chunk, (k * procs + j) % n_units, 1, 0.0)
                                            for j in range(procs)])
            done.append(sum(d for d, _ in res))

        for k in range(args.warmup):
            step(k)
        done.clear()
        t0 = time.perf_counter()
        for k in range(args.steps):
            step(args.warmup + k)
        sec = time.perf_counter() - t0
    finally:
        pool.close()
        pool.join()
    value = sum(done) / sec
    sample = (f"oracle.continuous in {procs} spawned processes, one call per process per step on "
              f"{chunk} tokens of one prefill sequence each")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) FP16 QKV)",
        "config": {"workload": DESCR[HEADLINE], "tokens_per_step": sum(done) // args.steps},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": procs, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------- main --

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=list(workloads.CONFIG_NAMES) + list(workloads.PROFILE_NAMES)
                    + list(workloads.NEXT_NAMES)
                    + ["decode_floor", "paged_fused_3launch", "paged_fused_p8192_3launch"],
                    help="workload of the headline line (default: the prefill)")
    ap.add_argument("--extra-steps", type=int, default=4000,
                    help="timed launches per extra workload (decode, tree, paged, packed_tiny)")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU time budget of the headline's oracle baseline sample "
                         "(single thread, then all cores); 0 leaves the CPU baseline out "
                         "(profiling runs)")
    ap.add_argument("--cpu-seconds-extra", type=float, default=1.5,
                    help="the same for every other workload")
    ap.add_argument("--e2e-steps", type=int, default=100)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and (world > 1 or args.gpus > 1):
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch with torchrun")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    barrier = None
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        barrier = lambda: dist.barrier()

    from rope_kv_cache_gb300 import build as rkbuild
    rkbuild.build_library()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    peak, peak_src = measured_peak()
    uuid = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(local))
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    stream = torch.cuda.Stream(dev)

    name = args.workload
    wl = make_workload(name, dev, l2)
    sec, t0, t1 = time_steps(wl, args.steps, args.warmup, stream, barrier)
    if world > 1:
        sec = max_over_ranks(sec, dist, dev)
    launch_s = sec / args.steps
    achieved = wl.bytes / launch_s / 1e9
    clocks = sampler.summary(t0, t1) if sampler else None
    e2e = e2e_contiguous(wl, args.e2e_steps) \
        if isinstance(wl, DeviceWorkload) and not (
            wl.paged or wl.fused or wl.slotmap or wl.case.norm is not None
            or wl.case.fp8_scales is not None) else None
    tokens, bytes_step, ring = wl.tokens, wl.bytes, wl.ring
    per_set = getattr(wl, "caches_per_set", None)
    kernel = _kernel_name(wl)
    del wl
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extra:
        for xname in EXTRA:
            if xname == name:
                continue
            w = make_workload(xname, dev, l2)
            s_, _, _ = time_steps(w, args.extra_steps, args.warmup, stream, barrier)
            per = s_ / args.extra_steps
            gbs = w.bytes / per / 1e9
            extra[xname] = {"workload": DESCR[xname], "tokens_per_step": w.tokens,
                            "launches_per_step": 3 if w.three_launch else 1,
                            "bytes_per_step": w.bytes, "ring": w.ring,
                            "us_per_launch": per * 1e6, "tokens_per_s": w.tokens / per,
                            "effective_gbs": gbs, "frac_of_measured_peak": gbs / peak,
                            "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                            "launches_timed": args.extra_steps, "kernel": _kernel_name(w),
                            "cache_per_ring_set": getattr(w, "caches_per_set", None),
                            "dram_bytes_per_launch_ncu": ncu_traffic(xname)}
            case = getattr(w, "case", None)     # the floor copy has no case
            if isinstance(case, workloads.ContiguousCase) and case.mode == "tree":
                # the same launch with each distinct cos/sin row counted once
                # (siblings share their position's row)
                bd = case.algorithmic_bytes_distinct_rows()
                extra[xname]["bytes_per_step_distinct_rows"] = bd
                extra[xname]["effective_gbs_distinct_rows"] = bd / per / 1e9
            del w
            torch.cuda.empty_cache()
        floor = extra.get("decode_floor")
        if floor is not None:
            # decode-sized launches as a fraction of the floor of one dependent
            # launch in the same grid (time ratio: 1.0 = at the floor)
            floor["cpu_baseline"] = None
            floor["note"] = "a measurement reference, not a workload of the method: no oracle"
            for xname in ("decode", "decode_qknorm", "decode_fp8", "slotmap_decode"):
                if xname in extra:
                    extra[xname]["floor_us_per_launch"] = floor["us_per_launch"]
                    extra[xname]["frac_of_floor"] = (floor["us_per_launch"]
                                                     / extra[xname]["us_per_launch"])
    if sampler:
        sampler.stop()
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    cpu = {name: None}
    if args.cpu_seconds > 0:
        pool, procs = oracle_process_pool()
        try:
            if name != "decode_floor":
                cpu = oracle_rates([name], args.cpu_seconds, args.cpu_seconds, pool, procs)
            if extra:
                cpu.update(oracle_rates([x for x in EXTRA if x in extra and x != "decode_floor"
                                         and not x.endswith("_3launch")],
                                        args.cpu_seconds_extra, args.cpu_seconds_extra, pool,
                                        procs))
        finally:
            pool.close()
            pool.join()
    for xname, entry in extra.items():
        base = cpu.get(_oracle_base_name(xname))
        if base is not None:
            entry["cpu_baseline"] = dict(base)
            if xname.endswith("_3launch"):
                entry["cpu_baseline"]["note"] = "the same oracle work as the one-launch step"
    line = {
        "metric": METRIC,
        "value": whole_job_rate(world, tokens, args.steps, sec),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage": "f16 in/out, f32 cos/sin, f32 math",
        "data": "synthetic: seeded N(0,1) FP16 activations, FP32 RoPE table (no dataset, no weights)",
        "config": {"workload": DESCR.get(name, name), "tokens_per_step": tokens,
                   "bytes_per_step": bytes_step,
                   "parallelism": f"one independent replica per GPU x{world} (no exchange)",
                   "l2": f"inputs larger than L2: ring of {ring} input sets, "
                         f"{ring * bytes_step / 1e6:.0f} MB > 2 x L2 ({l2 / 1e6:.0f} MB)",
                   "timed_region": "CUDA events around exactly K launches replayed from CUDA "
                                   "graphs on one stream; a 0.2 ms sleep kernel queued ahead of "
                                   "the start event keeps the graph submission out of it",
                   "caches": None if per_set is None else
                   ("one KV cache per ring set (each step writes a cache the previous step did "
                    "not)" if per_set else "one KV cache shared by the ring sets")},
        "effective_gbs": achieved,
        "pct_of_peak": {"measured_copy": 100 * achieved / peak,
                        "nominal_8tbs": 100 * achieved / NOMINAL_HBM_GBS},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(name),
                     "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "kernel": kernel},
        "cpu_baseline": cpu[name],
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "workloads": extra,
    }
    print(json.dumps(line), flush=True)
    return 0


def _kernel_name(wl) -> str:
    if isinstance(wl, FloorWorkload):
        return "floor_copy_kernel (libropekv_floor.so)"
    c = wl.case
    if wl.slotmap:
        return f"rope_kv_slotmap_kernel<D={c.D}, {'NeoX' if c.style == 0 else 'GPT-J'}>"
    if wl.fused:
        if wl.three_launch:
            return "delta_metadata_kernel + gather_delta_rope_kernel + paged_delta_kernel"
        return f"paged_delta_kernel<D={c.D}, {'NeoX' if c.style == 0 else 'GPT-J'}, fused>"
    if wl.paged:
        return f"paged_delta_kernel<D={c.D}, {'NeoX' if c.style == 0 else 'GPT-J'}>"
    return (f"rope_kv_token_kernel<D={c.D}, {'NeoX' if c.style == 0 else 'GPT-J'}, "
            f"{c.mode}{', qk-norm' if c.norm is not None else ''}"
            f"{', e4m3 cache' if c.fp8_scales is not None else ''}>")


if __name__ == "__main__":
    sys.exit(main())
