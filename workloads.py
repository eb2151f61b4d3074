"""Seeded synthetic inputs for the fused RoPE + KV-cache write.

This module only draws inputs: FP16 activations, cos/sin tables, positions,
trees, page tables. It holds none of the rotation or cache-write arithmetic,
and both the CUDA path's tests/benchmark and the CPU oracle's tests take their
inputs from here. Every draw uses ``numpy.random.Generator(PCG64(seed))``.

Workload shapes follow the pages: Llama-style GQA (32 query heads, 8 KV heads,
head dim 128) for prefill, decode, tree speculative decoding (TensorRT-Edge-LLM
"Apply Rope Write KV") and the DFlash paged delta update (TensorRT-Edge-LLM
"Dflash Runtime Kernels", ``launchDFlashTargetKVCacheUpdate``). No dataset or
trained weight is involved; activations are N(0,1) rounded to FP16.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

NEOX = 0
GPTJ = 1

# FP16 bit pattern written into every output buffer before a call: a NaN that
# no finite input or rotated value can produce, so any byte the call did not
# write is recognisable afterwards.
SENTINEL = 0x7E5A
# The same for E4M3 caches: 0x7F is NaN there, and the saturating store never
# produces NaN from finite values.
SENTINEL8 = 0x7F


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def fp16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) samples rounded to FP16 (numpy's round-to-nearest-even), as bits."""
    return rng.standard_normal(size=shape).astype(np.float16).view(np.uint16)


def cos_sin_table(theta: float, seq_len: int, rotary_dim: int, batch: int = 1,
                  pos_offset: Optional[np.ndarray] = None) -> np.ndarray:
    """FP32 table [batch, seq_len, rotary_dim] = [cos_0..cos_{h-1} | sin_0..sin_{h-1}].

    Row p holds angle p * theta^(-2i/r) for frequency i < h = r/2, computed in
    double and rounded to FP32. ``pos_offset`` (per batch row) shifts the
    positions of each batch row, giving distinct per-sequence tables.
    """
    h = rotary_dim // 2
    i = np.arange(h, dtype=np.float64)
    inv_freq = theta ** (-(2.0 * i) / rotary_dim)
    out = np.empty((batch, seq_len, rotary_dim), dtype=np.float32)
    for b in range(batch):
        off = 0 if pos_offset is None else int(pos_offset[b])
        pos = np.arange(seq_len, dtype=np.float64) + off
        ang = pos[:, None] * inv_freq[None, :]
        out[b, :, :h] = np.cos(ang).astype(np.float32)
        out[b, :, h:] = np.sin(ang).astype(np.float32)
    return out


def sentinel_fill(shape) -> np.ndarray:
    return np.full(shape, SENTINEL, dtype=np.uint16)


# ------------------------------------------------------------- contiguous --

@dataclass
class ContiguousCase:
    """Inputs of the packed / continuous / tree entry points (host arrays)."""
    mode: str                 # "packed" | "continuous" | "tree"
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    r: int
    cap: int
    style: int
    theta: float
    cos_sin: np.ndarray       # [csB, csS, r] float32
    qkv: np.ndarray           # [B, S, Hq+2Hkv, D] uint16
    end_lens: Optional[np.ndarray] = None   # [B] int32
    pos_ids: Optional[np.ndarray] = None    # [B, S] int32
    cache_init: str = "sentinel"            # "sentinel" | "zero"
    name: str = ""
    # pre-RoPE QK RMS norm (continuous call only): (q_weight [D], k_weight [D]
    # uint16 FP16 bits, eps) or None
    norm: Optional[tuple] = None
    # FP8 (E4M3) cache (continuous call only): (k_scale, v_scale) or None
    fp8_scales: Optional[tuple] = None

    @property
    def H(self) -> int:
        return self.Hq + 2 * self.Hkv

    @property
    def tokens(self) -> int:
        return self.B * self.S

    def new_cache(self) -> np.ndarray:
        shape = (self.B, 2, self.Hkv, self.cap, self.D)
        if self.cache_init == "zero":
            return np.zeros(shape, dtype=np.uint16)
        return sentinel_fill(shape)

    def new_qout(self) -> np.ndarray:
        return sentinel_fill((self.B, self.S, self.Hq, self.D))

    def new_cache8(self) -> np.ndarray:
        """E4M3 cache filled with 0x7F, a NaN no saturating conversion produces."""
        return np.full((self.B, 2, self.Hkv, self.cap, self.D), SENTINEL8, dtype=np.uint8)

    def algorithmic_bytes(self) -> int:
        """QKV read + cos/sin read (one row per token) + Q, K, V written."""
        kv_elem = 1 if self.fp8_scales is not None else 2
        per_tok = (self.H * self.D * 2            # packed QKV row read
                   + self.r * 4                   # cos/sin row read
                   + self.Hq * self.D * 2         # Q written (qOut, or in place)
                   + 2 * self.Hkv * self.D * kv_elem)  # K and V cache rows written
        if self.mode == "packed":
            per_tok += self.Hkv * self.D * 2      # K also rotated in place in qkv
        return per_tok * self.tokens

    def positions(self) -> np.ndarray:
        """[B, S] RoPE position of every token (packed: s; continuous: end - S
        + s; tree: tokenPosIds)."""
        if self.mode == "tree":
            return np.asarray(self.pos_ids, dtype=np.int64)
        s = np.arange(self.S, dtype=np.int64)[None, :]
        if self.mode == "packed":
            return np.repeat(s, self.B, axis=0)
        return np.asarray(self.end_lens, dtype=np.int64)[:, None] - self.S + s

    def algorithmic_bytes_distinct_rows(self) -> int:
        """algorithmic_bytes with the cos/sin bytes counted once per distinct
        table row a launch reads rather than once per token (tree siblings
        share their position's row); tokens without a row in the table are
        left out."""
        pos = self.positions()
        csB, csS = self.cos_sin.shape[:2]
        table = np.broadcast_to(np.arange(self.B)[:, None] if csB > 1 else 0, pos.shape)
        ok = (pos >= 0) & (pos < csS)
        rows = len(set(zip(table[ok].tolist(), pos[ok].tolist())))
        return self.algorithmic_bytes() - self.r * 4 * self.tokens + self.r * 4 * rows


def norm_weights(seed: int, D: int, eps: float = 1e-6):
    """RMS-norm weights for Q and K heads, 1 + 0.1 N(0,1) rounded to FP16, and eps."""
    rng = rng_for(seed)
    w = (1.0 + 0.1 * rng.standard_normal((2, D))).astype(np.float16).view(np.uint16)
    return np.ascontiguousarray(w[0]), np.ascontiguousarray(w[1]), eps


def random_tree_depths(rng: np.random.Generator, n: int, max_parent_depth: int = 5) -> np.ndarray:
    """Depths of a random tree of n nodes: node 0 is the root (depth 0); node
    i > 0 picks its parent uniformly among earlier nodes of depth <= max_parent_depth."""
    depth = np.zeros(n, dtype=np.int32)
    for i in range(1, n):
        cands = np.nonzero(depth[:i] <= max_parent_depth)[0]
        parent = int(cands[rng.integers(0, len(cands))])
        depth[i] = depth[parent] + 1
    return depth


def make_packed(B, S, Hq, Hkv, D, r, cap, style, theta, seed, cs_seq=None, cs_batch=1,
                cache_init="zero", name="packed") -> ContiguousCase:
    rng = rng_for(seed)
    qkv = fp16_normal(rng, (B, S, Hq + 2 * Hkv, D))
    cs_seq = cap if cs_seq is None else cs_seq
    offs = None if cs_batch == 1 else rng.integers(0, 1000, size=cs_batch)
    cos_sin = cos_sin_table(theta, cs_seq, r, cs_batch, offs)
    return ContiguousCase("packed", B, S, Hq, Hkv, D, r, cap, style, theta, cos_sin, qkv,
                          cache_init=cache_init, name=name)


def make_continuous(B, S, Hq, Hkv, D, r, cap, style, theta, seed, end_lens=None,
                    start_range=None, cs_seq=None, cs_batch=1, name="continuous") -> ContiguousCase:
    """kvCacheEndLens = start_b + S with start_b uniform in start_range (inclusive),
    unless ``end_lens`` is given."""
    rng = rng_for(seed)
    qkv = fp16_normal(rng, (B, S, Hq + 2 * Hkv, D))
    if end_lens is None:
        lo, hi = start_range if start_range is not None else (0, cap - S)
        end_lens = rng.integers(lo, hi + 1, size=B).astype(np.int32) + np.int32(S)
    end_lens = np.asarray(end_lens, dtype=np.int32)
    cs_seq = cap if cs_seq is None else cs_seq
    offs = None if cs_batch == 1 else rng.integers(0, 1000, size=cs_batch)
    cos_sin = cos_sin_table(theta, cs_seq, r, cs_batch, offs)
    return ContiguousCase("continuous", B, S, Hq, Hkv, D, r, cap, style, theta, cos_sin, qkv,
                          end_lens=end_lens, name=name)


def make_tree(B, S, Hq, Hkv, D, r, cap, style, theta, seed, base_range, cs_seq=None,
              cs_batch=1, name="tree") -> ContiguousCase:
    """tokenPosIds[b, s] = base_b + depth_b[s] over a random tree per sequence;
    kvCacheEndLens[b] = base_b + S (tree tokens take linear slots)."""
    rng = rng_for(seed)
    qkv = fp16_normal(rng, (B, S, Hq + 2 * Hkv, D))
    base = rng.integers(base_range[0], base_range[1] + 1, size=B).astype(np.int32)
    depths = np.stack([random_tree_depths(rng, S) for _ in range(B)]) if S > 0 else \
        np.zeros((B, 0), dtype=np.int32)
    pos_ids = (base[:, None] + depths).astype(np.int32)
    end_lens = (base + S).astype(np.int32)
    cs_seq = cap if cs_seq is None else cs_seq
    offs = None if cs_batch == 1 else rng.integers(0, 1000, size=cs_batch)
    cos_sin = cos_sin_table(theta, cs_seq, r, cs_batch, offs)
    return ContiguousCase("tree", B, S, Hq, Hkv, D, r, cap, style, theta, cos_sin, qkv,
                          end_lens=end_lens, pos_ids=np.ascontiguousarray(pos_ids), name=name)


# ------------------------------------------------------------------ paged --

@dataclass
class PagedCase:
    """Inputs of the paged delta update (host arrays)."""
    N: int                    # numDeltaTokens
    B: int                    # batchSize
    Hkv: int
    D: int
    r: int
    num_pages: int
    max_pages_per_seq: int
    tokens_per_page: int
    style: int
    theta: float
    k_delta: np.ndarray       # [N, Hkv, D] uint16
    v_delta: np.ndarray       # [N, Hkv, D] uint16
    cos_sin_rows: np.ndarray  # [N, r] float32 (token-aligned: row t for delta row t)
    positions: np.ndarray     # [N] int32
    seq_ids: np.ndarray       # [N] int32
    page_table: np.ndarray    # [B, 2, maxPagesPerSeq] int32
    name: str = ""
    extra: dict = field(default_factory=dict)

    def pool_shape(self):
        return (2, self.num_pages, self.tokens_per_page, self.Hkv, self.D)

    def new_pool(self) -> np.ndarray:
        return sentinel_fill(self.pool_shape())

    def plane_written(self):
        """Boolean [N] masks: K plane written, V plane written (skip rules of
        launchDFlashTargetKVCacheUpdate); input bookkeeping for byte counts."""
        pos, seq = self.positions, self.seq_ids
        ok = (pos >= 0) & (seq >= 0) & (seq < self.B)
        lp = np.where(ok, pos // self.tokens_per_page, 0)
        ok &= lp < self.max_pages_per_seq
        s = np.where(ok, seq, 0)
        lpc = np.where(ok, lp, 0)
        idk = self.page_table[s, 0, lpc]
        idv = self.page_table[s, 1, lpc]
        kw = ok & (idk >= 0) & (idk < self.num_pages)
        vw = ok & (idv >= self.num_pages) & (idv < 2 * self.num_pages)
        return kw, vw

    def algorithmic_bytes(self) -> int:
        """Per row: 8 B of metadata; per written K plane: K read + cos/sin row +
        K written; per written V plane: V read + V written."""
        kw, vw = self.plane_written()
        row = self.Hkv * self.D * 2
        return int(self.N * 8 + kw.sum() * (2 * row + self.r * 4) + vw.sum() * 2 * row)

    @property
    def valid_rows(self) -> int:
        kw, vw = self.plane_written()
        return int((kw | vw).sum())


def make_paged(N, B, Hkv, D, r, tokens_per_page, max_pages_per_seq, num_pages, style, theta,
               seed, valid_rows=None, len_range=(1, 256), unmapped_frac=0.02,
               max_position=None, name="paged") -> PagedCase:
    """DFlash-style delta rows.

    * per-sequence delta lengths L_b uniform in len_range, then moved by +-1 on
      random sequences until sum(L_b) == valid_rows (default 95 % of N);
    * the N - valid_rows padding rows (position = sequence = -1) sit at random
      row indices; valid rows are grouped by sequence in order;
    * sequence b's rows take consecutive positions old_b .. old_b + L_b - 1 with
      old_b uniform in [0, max_position - L_b];
    * K-plane page ids are a random permutation of [0, num_pages) spread over
      the [B, maxPagesPerSeq] logical pages (cycled if there are more logical
      pages than physical); V-plane ids are num_pages + a separate permutation;
      then ``unmapped_frac`` of all table entries become -1;
    * cos/sin rows are gathered at each row's position (padding rows zero).
    """
    rng = rng_for(seed)
    if valid_rows is None:
        valid_rows = int(round(0.95 * N))
    if max_position is None:
        max_position = max_pages_per_seq * tokens_per_page
    lo, hi = len_range
    hi = min(hi, max_position)
    k_delta = fp16_normal(rng, (N, Hkv, D))
    v_delta = fp16_normal(rng, (N, Hkv, D))
    if B > 0:
        L = rng.integers(lo, hi + 1, size=B).astype(np.int64)
        if not (B * lo <= valid_rows <= B * hi):
            raise ValueError("valid_rows not reachable with len_range")
        while L.sum() != valid_rows:
            b = int(rng.integers(0, B))
            if L.sum() > valid_rows and L[b] > lo:
                L[b] -= 1
            elif L.sum() < valid_rows and L[b] < hi:
                L[b] += 1
    else:
        L = np.zeros(0, dtype=np.int64)
        valid_rows = 0
    old = np.array([rng.integers(0, max_position - int(l) + 1) for l in L], dtype=np.int64)
    seq_of_valid = np.repeat(np.arange(B, dtype=np.int32), L)
    pos_of_valid = np.concatenate([old[b] + np.arange(L[b]) for b in range(B)]).astype(np.int32) \
        if B > 0 else np.zeros(0, dtype=np.int32)
    pad_idx = np.sort(rng.choice(N, size=N - valid_rows, replace=False))
    is_pad = np.zeros(N, dtype=bool)
    is_pad[pad_idx] = True
    positions = np.full(N, -1, dtype=np.int32)
    seq_ids = np.full(N, -1, dtype=np.int32)
    positions[~is_pad] = pos_of_valid
    seq_ids[~is_pad] = seq_of_valid
    n_logical = B * max_pages_per_seq
    reps = -(-n_logical // max(num_pages, 1)) if num_pages > 0 else 0
    if num_pages > 0:
        kperm = np.concatenate([rng.permutation(num_pages) for _ in range(reps)])[:n_logical]
        vperm = np.concatenate([rng.permutation(num_pages) for _ in range(reps)])[:n_logical]
    else:
        kperm = np.full(n_logical, -1)
        vperm = np.full(n_logical, -1 - num_pages)
    table = np.empty((B, 2, max_pages_per_seq), dtype=np.int32)
    table[:, 0, :] = kperm.reshape(B, max_pages_per_seq)
    table[:, 1, :] = (vperm + num_pages).reshape(B, max_pages_per_seq)
    n_unmapped = int(round(unmapped_frac * table.size))
    if n_unmapped:
        flat = table.reshape(-1)
        flat[rng.choice(table.size, size=n_unmapped, replace=False)] = -1
    cs_full = cos_sin_table(theta, max_position, r)[0]
    cs_rows = np.zeros((N, r), dtype=np.float32)
    valid = positions >= 0
    cs_rows[valid] = cs_full[positions[valid]]
    return PagedCase(N, B, Hkv, D, r, num_pages, max_pages_per_seq, tokens_per_page, style, theta,
                     k_delta, v_delta, cs_rows, positions, seq_ids,
                     np.ascontiguousarray(table), name=name, extra={"lengths": L, "old": old})


# ----------------------------------------------------- fused DFlash update --

@dataclass
class PagedFusedCase:
    """Inputs of the one-launch DFlash update (metadata + gather + paged update):
    rows laid out [B, W]; row b*W + j is sequence b's delta token j."""
    B: int
    W: int                    # deltaWidth
    Hkv: int
    D: int
    r: int
    num_pages: int
    max_pages_per_seq: int
    tokens_per_page: int
    style: int
    theta: float
    k_delta: np.ndarray       # [B*W, Hkv, D] uint16
    v_delta: np.ndarray       # [B*W, Hkv, D] uint16
    source: np.ndarray        # [sourceRows, cacheCapacity, r] float32
    old_lengths: np.ndarray   # [B] int32
    delta_lengths: np.ndarray  # [B] int32
    state: Optional[np.ndarray]  # [B] int32 or None
    page_table: np.ndarray    # [B, 2, maxPagesPerSeq] int32
    name: str = ""

    @property
    def N(self) -> int:
        return self.B * self.W

    def pool_shape(self):
        return (2, self.num_pages, self.tokens_per_page, self.Hkv, self.D)

    def new_pool(self) -> np.ndarray:
        return sentinel_fill(self.pool_shape())

    def plane_written(self):
        """Boolean [B*W] masks of rows whose K / V plane is written (input
        bookkeeping for byte counts: layout, page-table and capacity rules)."""
        j = np.tile(np.arange(self.W), self.B)
        b = np.repeat(np.arange(self.B), self.W)
        pos = self.old_lengths[b].astype(np.int64) + j
        ok = (j < self.delta_lengths[b]) & (pos >= 0)
        lp = np.where(ok, pos // self.tokens_per_page, 0)
        ok &= lp < self.max_pages_per_seq
        lpc = np.where(ok, lp, 0)
        idk = self.page_table[b, 0, lpc]
        idv = self.page_table[b, 1, lpc]
        kw = ok & (idk >= 0) & (idk < self.num_pages)
        vw = ok & (idv >= self.num_pages) & (idv < 2 * self.num_pages)
        return kw, vw

    def algorithmic_bytes(self) -> int:
        """8 B of lengths per sequence; per written K plane: K read + cos/sin row
        + K written; per written V plane: V read + V written."""
        kw, vw = self.plane_written()
        row = self.Hkv * self.D * 2
        return int(self.B * 8 + kw.sum() * (2 * row + self.r * 4) + vw.sum() * 2 * row)

    @property
    def valid_rows(self) -> int:
        kw, vw = self.plane_written()
        return int((kw | vw).sum())


def make_paged_fused(B, W, Hkv, D, r, tokens_per_page, max_pages_per_seq, num_pages, style, theta,
                     seed, len_range=None, unmapped_frac=0.02, source_rows=1, with_state=False,
                     cache_capacity=None, name="paged_fused") -> PagedFusedCase:
    """Delta lengths uniform in len_range (default 1..W), old lengths uniform so
    that every token fits the sequence's logical pages, page ids as make_paged,
    a cos/sin source of `source_rows` tables (row k shifted by k*1000 positions)
    of cache_capacity positions, optional per-sequence state indices."""
    rng = rng_for(seed)
    k_delta = fp16_normal(rng, (B * W, Hkv, D))
    v_delta = fp16_normal(rng, (B * W, Hkv, D))
    lo, hi = len_range if len_range is not None else (1, W)
    lengths = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    max_position = max_pages_per_seq * tokens_per_page
    old = np.array([rng.integers(0, max(1, max_position - max(int(l), 0) + 1)) for l in lengths],
                   dtype=np.int32)
    n_logical = B * max_pages_per_seq
    reps = -(-n_logical // num_pages)
    kperm = np.concatenate([rng.permutation(num_pages) for _ in range(reps)])[:n_logical]
    vperm = np.concatenate([rng.permutation(num_pages) for _ in range(reps)])[:n_logical]
    table = np.empty((B, 2, max_pages_per_seq), dtype=np.int32)
    table[:, 0, :] = kperm.reshape(B, max_pages_per_seq)
    table[:, 1, :] = (vperm + num_pages).reshape(B, max_pages_per_seq)
    n_unmapped = int(round(unmapped_frac * table.size))
    if n_unmapped:
        flat = table.reshape(-1)
        flat[rng.choice(table.size, size=n_unmapped, replace=False)] = -1
    cap = max_position if cache_capacity is None else cache_capacity
    offs = np.arange(source_rows) * 1000
    source = cos_sin_table(theta, cap, r, batch=source_rows, pos_offset=offs)
    state = rng.integers(0, source_rows, size=B).astype(np.int32) if with_state else None
    return PagedFusedCase(B, W, Hkv, D, r, num_pages, max_pages_per_seq, tokens_per_page, style,
                          theta, k_delta, v_delta, source, old, lengths, state,
                          np.ascontiguousarray(table), name=name)


# ------------------------------------------------------ flat slot mapping --

@dataclass
class SlotMapCase:
    """Inputs of the sglang-style call: q, k, v are views into one packed
    [T, Hq + 2 Hkv, D] buffer; per-token positions and flat cache slots."""
    Hq: int
    Hkv: int
    D: int
    r: int
    style: int
    theta: float
    num_blocks: int
    block_size: int
    qkv: np.ndarray           # [T, Hq+2Hkv, D] uint16
    positions: np.ndarray     # [T] int64
    slots: np.ndarray         # [T] int64
    cos_sin: np.ndarray       # [rows, r] float32
    seq_lens: tuple = ()
    name: str = ""

    @property
    def T(self) -> int:
        return self.qkv.shape[0]

    @property
    def tokens(self) -> int:
        return self.T

    @property
    def q(self):
        return self.qkv[:, : self.Hq]

    @property
    def k(self):
        return self.qkv[:, self.Hq: self.Hq + self.Hkv]

    @property
    def v(self):
        return self.qkv[:, self.Hq + self.Hkv:]

    def cache_shape(self):
        return (self.num_blocks, self.block_size, self.Hkv, self.D)

    def algorithmic_bytes(self) -> int:
        """QKV read + cos/sin read + positions and slots read + Q, K, V written
        (K and V only for tokens with a valid slot)."""
        H = self.Hq + 2 * self.Hkv
        ok = (self.slots >= 0) & (self.slots < self.num_blocks * self.block_size)
        per_tok = H * self.D * 2 + self.r * 4 + 16 + self.Hq * self.D * 2
        return int(self.T * per_tok + ok.sum() * 2 * self.Hkv * self.D * 2)


def _slot_assignment(rng, seq_lens, block_size, num_blocks):
    """Each sequence's tokens fill consecutive offsets of its own blocks,
    starting at a random offset of its first block; blocks come from one
    random permutation of the pool (no block is shared)."""
    perm = rng.permutation(num_blocks)
    nxt = 0
    out = []
    for n in seq_lens:
        first = int(rng.integers(0, block_size))
        nblk = -(-(first + n) // block_size)
        blocks = perm[nxt: nxt + nblk]
        if len(blocks) < nblk:
            raise ValueError("not enough blocks for the sequences")
        nxt += nblk
        idx = first + np.arange(n)
        out.append(blocks[idx // block_size].astype(np.int64) * block_size + idx % block_size)
    return np.concatenate(out) if out else np.zeros(0, dtype=np.int64)


def make_slotmap(seq_lens, Hq, Hkv, D, r, style, theta, seed, block_size, num_blocks,
                 start_range, cs_rows, name="slotmap") -> SlotMapCase:
    rng = rng_for(seed)
    T = int(sum(seq_lens))
    qkv = fp16_normal(rng, (T, Hq + 2 * Hkv, D))
    starts = rng.integers(start_range[0], start_range[1] + 1, size=len(seq_lens))
    positions = np.concatenate([st + np.arange(n) for st, n in zip(starts, seq_lens)]) \
        .astype(np.int64) if T else np.zeros(0, dtype=np.int64)
    slots = _slot_assignment(rng, seq_lens, block_size, num_blocks)
    cos_sin = cos_sin_table(theta, cs_rows, r)[0]
    return SlotMapCase(Hq, Hkv, D, r, style, theta, num_blocks, block_size, qkv, positions,
                       np.ascontiguousarray(slots), np.ascontiguousarray(cos_sin),
                       tuple(int(x) for x in seq_lens), name=name)


# ------------------------------------------------------------ the configs --

CONFIG_NAMES = ("packed_tiny", "prefill", "decode", "tree", "paged")

# Smaller-footprint twins of workloads for profiler captures: the same
# tokens / rows per launch, a smaller cache (decode: capacity 1024) or pool
# (paged: 64 logical pages per sequence, 8192 pages per plane, positions < 4096).
PROFILE_NAMES = ("decode_c1024", "decode_qknorm_c1024", "decode_fp8_c1024", "paged_p8192",
                 "paged_fused_p8192", "slotmap_prefill_b4096", "slotmap_decode_b4096")

# Workloads of the next rows (built on the same kernels).
NEXT_NAMES = ("paged_fused", "slotmap_prefill", "slotmap_decode", "prefill_qknorm",
              "decode_qknorm", "prefill_fp8", "decode_fp8")


def config(name: str):
    """The five benchmark workloads, each drawn with its own seed (0..4)."""
    if name == "packed_tiny":
        # B=1, S=16, Hq=4, Hkv=2, D=r=64 NeoX, theta 1e4, table [1,64,64],
        # zero-initialised cache [1,2,2,64,64], positions 0..15.
        return make_packed(1, 16, 4, 2, 64, 64, 64, NEOX, 1e4, seed=0, cs_seq=64,
                           cache_init="zero", name=name)
    if name == "prefill":
        # Llama-3-8B-shaped prefill: B=4, S=2048, Hq=32, Hkv=8, D=r=128 NeoX,
        # theta 5e5, capacity 8192, end = start + 2048 with start in [0, 4096].
        return make_continuous(4, 2048, 32, 8, 128, 128, 8192, NEOX, 5e5, seed=1,
                               start_range=(0, 4096), cs_seq=8192, name=name)
    if name == "decode":
        # B=256 one-token decode, end lengths uniform in [1, 8192].
        rng = rng_for(2)
        qkv = fp16_normal(rng, (256, 1, 48, 128))
        end_lens = rng.integers(1, 8192 + 1, size=256).astype(np.int32)
        cos_sin = cos_sin_table(5e5, 8192, 128)
        return ContiguousCase("continuous", 256, 1, 32, 8, 128, 128, 8192, NEOX, 5e5, cos_sin,
                              qkv, end_lens=end_lens, name=name)
    if name == "tree":
        # B=64, 64 tree tokens, D=128, partial r=64 GPT-J, theta 1e4, base in
        # [128, 4000], capacity 4096.
        return make_tree(64, 64, 32, 8, 128, 64, 4096, GPTJ, 1e4, seed=3,
                         base_range=(128, 4000), cs_seq=4096, name=name)
    if name == "decode_c1024":
        rng = rng_for(2)
        qkv = fp16_normal(rng, (256, 1, 48, 128))
        end_lens = rng.integers(1, 1024 + 1, size=256).astype(np.int32)
        cos_sin = cos_sin_table(5e5, 1024, 128)
        return ContiguousCase("continuous", 256, 1, 32, 8, 128, 128, 1024, NEOX, 5e5, cos_sin,
                              qkv, end_lens=end_lens, name=name)
    if name in ("decode_qknorm_c1024", "decode_fp8_c1024"):
        # profiler-sized twins of decode_qknorm / decode_fp8 (capacity 1024)
        case = config("decode_c1024")
        if name.startswith("decode_qknorm"):
            case.norm = norm_weights(8, case.D)
        else:
            case.fp8_scales = (0.05, 0.04)
        case.name = name
        return case
    if name == "slotmap_decode_b4096":
        return make_slotmap([1] * 256, 32, 8, 128, 128, NEOX, 5e5, seed=7, block_size=64,
                            num_blocks=4096, start_range=(0, 8191), cs_rows=8192, name=name)
    if name == "paged_p8192":
        return make_paged(16384, 128, 8, 128, 128, 64, 64, 8192, NEOX, 5e5, seed=4,
                          valid_rows=15565, name=name)
    if name in ("prefill_qknorm", "decode_qknorm"):
        # the prefill / decode workloads with pre-RoPE QK RMS norm fused in
        case = config(name.split("_")[0])
        case.norm = norm_weights(8, case.D)
        case.name = name
        return case
    if name in ("prefill_fp8", "decode_fp8"):
        # the prefill / decode workloads with an E4M3 cache, per-tensor scales
        case = config(name.split("_")[0])
        case.fp8_scales = (0.05, 0.04)
        case.name = name
        return case
    if name == "slotmap_prefill":
        # the prefill above behind the sglang-style interface: 4 x 2048 tokens,
        # block size 64, 16384 blocks per cache, positions from start in [0, 4096]
        return make_slotmap([2048] * 4, 32, 8, 128, 128, NEOX, 5e5, seed=6, block_size=64,
                            num_blocks=16384, start_range=(0, 4096), cs_rows=8192, name=name)
    if name == "slotmap_decode":
        # 256 one-token sequences at positions in [0, 8191], one slot each
        return make_slotmap([1] * 256, 32, 8, 128, 128, NEOX, 5e5, seed=7, block_size=64,
                            num_blocks=16384, start_range=(0, 8191), cs_rows=8192, name=name)
    if name == "paged_fused_p8192":
        return make_paged_fused(128, 128, 8, 128, 128, 64, 64, 8192, NEOX, 5e5, seed=5,
                                name=name)
    if name == "slotmap_prefill_b4096":
        return make_slotmap([2048] * 4, 32, 8, 128, 128, NEOX, 5e5, seed=6, block_size=64,
                            num_blocks=4096, start_range=(0, 4096), cs_rows=8192, name=name)
    if name == "paged_fused":
        # the DFlash step in one launch: B=128 sequences x deltaWidth 128 rows
        # (16384 rows), delta lengths uniform in [1, 128], Hkv=8, D=r=128,
        # 64 tokens/page, 512 pages/seq, 65536 pages per plane, one shared
        # cos/sin table of 32768 positions.
        return make_paged_fused(128, 128, 8, 128, 128, 64, 512, 65536, NEOX, 5e5, seed=5,
                                name=name)
    if name == "paged":
        # 16384 delta rows over 128 sequences (15565 valid), Hkv=8, D=r=128,
        # 64 tokens/page, 512 logical pages per sequence, 65536 pages per plane.
        return make_paged(16384, 128, 8, 128, 128, 64, 512, 65536, NEOX, 5e5, seed=4,
                          valid_rows=15565, name=name)
    raise KeyError(name)


# ----------------------------------------------- per-step input variants --

def step_variant(case, k: int):
    """Index inputs of step k of a benchmark ring, drawn from the same
    distribution as the case's own (seed 1000 + k); step 0 is the case itself.

    Contiguous cases: (end_lens, pos_ids) -- new per-sequence start/end offsets
    (and tree bases) so every step writes different cache slots. Paged cases:
    page_table -- fresh page permutations with the same unmapped fraction, so
    every step writes different pages. Fused DFlash cases: (old_lengths,
    page_table).
    """
    if isinstance(case, SlotMapCase):
        if k == 0:
            return case.positions, case.slots
        rng = rng_for(1000 + k)
        lo, hi = int(case.positions.min()), int(case.positions.max())
        starts = rng.integers(0, max(1, hi - lo + 1), size=len(case.seq_lens))
        pos = np.concatenate([lo + st + np.arange(n) for st, n in zip(starts, case.seq_lens)])
        slots = _slot_assignment(rng, case.seq_lens, case.block_size, case.num_blocks)
        return pos.astype(np.int64), np.ascontiguousarray(slots)
    if k == 0:
        if isinstance(case, PagedCase):
            return case.page_table
        if isinstance(case, PagedFusedCase):
            return case.old_lengths, case.page_table
        return case.end_lens, case.pos_ids
    rng = rng_for(1000 + k)
    if isinstance(case, PagedFusedCase):
        max_position = case.max_pages_per_seq * case.tokens_per_page
        old = np.array([rng.integers(0, max(1, max_position - max(int(l), 0) + 1))
                        for l in case.delta_lengths], dtype=np.int32)
        t = case.page_table.copy()
        B, _, M = t.shape
        n = B * M
        reps = -(-n // case.num_pages)
        kp = np.concatenate([rng.permutation(case.num_pages) for _ in range(reps)])[:n]
        vp = np.concatenate([rng.permutation(case.num_pages) for _ in range(reps)])[:n]
        t[:, 0, :] = kp.reshape(B, M)
        t[:, 1, :] = (vp + case.num_pages).reshape(B, M)
        t[case.page_table < 0] = -1
        return old, np.ascontiguousarray(t)
    if isinstance(case, PagedCase):
        t = case.page_table.copy()
        B, _, M = t.shape
        n = B * M
        reps = -(-n // case.num_pages)
        kp = np.concatenate([rng.permutation(case.num_pages) for _ in range(reps)])[:n]
        vp = np.concatenate([rng.permutation(case.num_pages) for _ in range(reps)])[:n]
        t[:, 0, :] = kp.reshape(B, M)
        t[:, 1, :] = (vp + case.num_pages).reshape(B, M)
        unmapped = case.page_table < 0
        t[unmapped] = -1
        return np.ascontiguousarray(t)
    if case.mode == "packed":
        return None, None
    if case.mode == "tree":
        depth = case.pos_ids - (case.end_lens - case.S)[:, None]
        lo = int(case.end_lens.min() - case.S)
        hi = int(case.end_lens.max() - case.S)
        base = rng.integers(lo, hi + 1, size=case.B).astype(np.int32)
        return (base + case.S).astype(np.int32), np.ascontiguousarray((base[:, None] + depth).astype(np.int32))
    lo = int(case.end_lens.min())
    hi = int(case.end_lens.max())
    return rng.integers(lo, hi + 1, size=case.B).astype(np.int32), None
