// ropekv_kernels.cuh -- sm_103a kernels of the fused RoPE + KV-cache write.
//
// What is computed (sources cited by page title and section):
//   * x' = x*cos + rotate(x)*sin on the first rotaryDim dims of every Q and K
//     head (sglang rope_cache.py: _unit_rope; rotate() layouts of
//     _get_neox_rotated_x / _get_gptj_rotated_x; frequency index of kernel
//     Stage 2.1 with the half-width cos/sin table read as in _load_cos_sin).
//   * the contiguous-cache placement of TensorRT-Edge-LLM "Apply Rope Write KV"
//     (packed in place / continuous / tree), and
//   * the paged placement and skip rules of TensorRT-Edge-LLM "Dflash Runtime
//     Kernels", launchDFlashTargetKVCacheUpdate.
//
// Work decomposition. A head of D FP16 values is D/8 16-byte vectors. An
// "item" is two vectors of one head handled by one thread:
//   rotated region (item i < r/16): vectors i and i + r/16. For NeoX these are
//     partners (dims 8i+k and 8i+k+r/2 share frequency 8i+k), so the half swap
//     happens inside the thread's registers; for GPT-J each vector holds four
//     complete (2j, 2j+1) pairs, so the pair swap is inside one half2 word;
//   pass-through region (i >= r/16): two vectors past rotaryDim, copied as bits.
// V heads use the same vector pairs and are copied as bits. Items are numbered
// head-major inside a token, a CTA covers a contiguous run of one token's items
// and the block size is a multiple of D/16, so every thread keeps one item
// index i for all its heads: it loads its 8 cos + 8 sin values once per token
// and reuses them for every Q and K head it rotates. Loads are issued before
// the position / cos/sin chain resolves so their latencies overlap.
//
// All loads and stores are 16-byte vectors; a warp touches whole 32-byte
// sectors. Math is FP32 with round-to-nearest-even back to FP16. Invalid
// device-side indices are skipped; nothing traps or waits.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace ropekv {

enum Style : int { kNeox = 0, kGptj = 1 };
enum Mode : int { kPacked = 0, kContinuous = 1, kTree = 2 };

// Arguments of the contiguous-cache kernel (packed / continuous / tree).
struct TokenArgs {
    const float* cosSin;       // [csBatch, csSeq, r]
    const int32_t* endLens;    // [B]      (continuous, tree)
    const int32_t* posIds;     // [B, S]   (tree)
    const uint16_t* qkv;       // [B, S, Hq + 2 Hkv, D]
    uint16_t* qkvOut;          // same buffer as qkv for the packed in-place call
    uint16_t* cache;           // [B, 2, Hkv, cap, D]
    uint16_t* qOut;            // [B, S, Hq, D] (continuous, tree)
    const uint16_t* qNormW;    // [D] FP16 RMS-norm weight of Q heads (normalized call)
    const uint16_t* kNormW;    // [D] FP16 RMS-norm weight of K heads (normalized call)
    float eps;                 // RMS-norm epsilon (normalized call)
    uint8_t* cache8;           // [B, 2, Hkv, cap, D] E4M3 cache (FP8 call; replaces cache)
    const float* kScale;       // K scale of the FP8 cache (device scalar)
    const float* vScale;       // V scale of the FP8 cache (device scalar)
    int32_t S, Hq, Hkv, r, cap, csBatch, csSeq;
    int32_t itemsPerToken;     // (Hq + 2 Hkv) * D / 16
    int32_t ctasPerToken;      // CTAs sharing one token's items
};

// Arguments of the paged delta kernel.
struct PagedArgs {
    const uint16_t* kDelta;    // [N, Hkv, D]
    const uint16_t* vDelta;    // [N, Hkv, D]
    uint16_t* pool;            // [2, numPages, tpp, Hkv, D]
    const float* cosSin;       // [N, r] token-aligned; fused: [sourceRows, cacheCapacity, r]
    const int32_t* positions;  // [N]                 (explicit metadata)
    const int32_t* seqIds;     // [N]                 (explicit metadata)
    const int32_t* pageTable;  // [B, 2, mpps]
    const int32_t* oldLens;    // [B] draft cache lengths before the delta   (fused)
    const int32_t* deltaLens;  // [B] delta tokens per sequence             (fused)
    const int32_t* stateIdx;   // [B] cos/sin source row per sequence, or NULL (fused)
    int32_t B, Hkv, r, numPages, mpps, tpp;
    int32_t deltaWidth, sourceRows, cacheCapacity;  // (fused)
    int32_t widthShift;        // log2(deltaWidth) if it is a power of two, else -1 (fused)
    int32_t itemsPerRow;       // 2 * Hkv * D / 16 (K heads, then V heads)
    int32_t ctasPerRow;
};

// Arguments of the flat slot-mapping kernel (sglang-style separate Q/K/V).
struct SlotMapArgs {
    const float* cosSin;       // [csRows, r]
    const int64_t* positions;  // [T]
    const uint16_t* q;         // [T, Hq, D] with token stride qStride (elements)
    const uint16_t* k;         // [T, Hkv, D] with token stride kStride
    const uint16_t* v;         // [T, Hkv, D] with token stride vStride
    const int64_t* slots;      // [T] flat cache slots
    uint16_t* keyCache;        // [numBlocks, blockSize, Hkv, D]
    uint16_t* valueCache;      // [numBlocks, blockSize, Hkv, D]
    uint16_t* qOut;            // [T, Hq, D]
    uint16_t* kOut;            // [T, Hkv, D] or NULL
    int64_t qStride, kStride, vStride, numSlots;
    int32_t Hq, Hkv, r, csRows;
    int32_t itemsPerToken;     // (Hq + 2 Hkv) * D / 16
    int32_t ctasPerToken;
};

// Arguments of the DFlash delta-metadata and cos/sin gather kernels.
struct DeltaMetaArgs {
    const int32_t* oldLens;    // [B]
    const int32_t* deltaLens;  // [B]
    int32_t* positions;        // [B * width]
    int32_t* seqIds;           // [B * width]
    int32_t B, width;
};

struct GatherArgs {
    const float* source;       // [sourceRows, cacheCapacity, r]
    float* output;             // [N, r]
    const int32_t* positions;  // [N]
    const int32_t* seqIds;     // [N]
    const int32_t* stateIdx;   // [B] or NULL
    int32_t N, B, sourceRows, cacheCapacity, r;
};

// --------------------------------------------------------------- helpers --

// Compile-time memory/launch policy of a kernel instantiation (bit set).
//   kPdl:        the grid may be launched as a programmatic dependent of the
//                previous kernel in the stream. Every thread first lets the
//                next grid begin launching, then waits until the previous
//                grid has completed and its writes are visible, before it
//                reads or writes anything: safe whatever that grid did.
//   kStreamHint: activations and cache rows are touched once per call: load
//                them bypassing L1 and mark loads and stores evict-first in L2.
//   kTableKeep:  cos/sin rows are reused across tokens and calls: mark them
//                evict-last in L2 so the streaming traffic does not push
//                them out.
//   kPrefetch:   (with kPdl) before waiting for the previous grid, warm L2 with
//                the thread's input vectors and the token's index words
//                (end length and tree position, or position and slot).
//                Only L2 prefetches happen before the wait: nothing is read
//                into a register, so nothing stale can be consumed afterwards
//                (L2 is the point of coherence) and no thread stalls on memory
//                before the wait. (A blocking read of the position there, to
//                prefetch the cos/sin row, cost a memory round trip per CTA:
//                256-token decode 1.90 -> 2.12 us.)
enum Policy : int { kPdl = 1, kStreamHint = 2, kTableKeep = 4, kPrefetch = 8 };

__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

struct L2Policies {
    uint64_t stream;
    uint64_t keep;
};

template <int POL>
__device__ __forceinline__ L2Policies make_policies()
{
    L2Policies p{0, 0};
    if (POL & kStreamHint)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p.stream));
    if (POL & kTableKeep)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p.keep));
    return p;
}

template <int POL>
__device__ __forceinline__ void grid_dependency_sync()
{
    if (POL & kPdl) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
}

// 16-byte load of data that no thread of this grid writes.
template <int POL>
__device__ __forceinline__ uint4 load_ro(const uint16_t* p, const L2Policies& pol)
{
    if (POL & kStreamHint) {
        uint4 v;
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p), "l"(pol.stream));
        return v;
    }
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte load of data this grid later overwrites (the packed in-place call).
template <int POL>
__device__ __forceinline__ uint4 load_rw(const uint16_t* p, const L2Policies& pol)
{
    if (POL & kStreamHint) {
        uint4 v;
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p), "l"(pol.stream)
                     : "memory");
        return v;
    }
    return *reinterpret_cast<const uint4*>(p);
}

template <int POL>
__device__ __forceinline__ void store_v(uint16_t* p, const uint4& v, const L2Policies& pol)
{
    if (POL & kStreamHint) {
        asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                     :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol.stream)
                     : "memory");
        return;
    }
    *reinterpret_cast<uint4*>(p) = v;
}

template <int POL>
__device__ __forceinline__ float4 load_f4(const float* p, const L2Policies& pol)
{
    if (POL & kTableKeep) {
        float4 f;
        asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                     : "l"(p), "l"(pol.keep));
        return f;
    }
    return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ __half2& h2(uint32_t& w)
{
    return *reinterpret_cast<__half2*>(&w);
}

// The two vectors of item i (in units of 16-byte vectors inside a head).
template <int D>
__device__ __forceinline__ void item_vectors(int i, int r, int& va, int& vb)
{
    const int rot_items = r >> 4;
    if (i < rot_items) {
        va = i;
        vb = i + rot_items;
    } else {
        const int j = i - rot_items;
        va = (r >> 3) + j;
        vb = va + ((D - r) >> 4);
    }
}

// cos/sin of the frequencies item i uses, from one table row of r floats.
// NeoX: frequencies 8i..8i+7 (shared by both vectors).
// GPT-J: frequencies 4i..4i+3 (first vector) and r/4 + 4i .. +3 (second).
template <int STYLE, int POL>
__device__ __forceinline__ void load_cos_sin(const float* row, int i, int r, float c[8],
                                             float s[8], const L2Policies& pol)
{
    const int h = r >> 1;
    float4 a, b, e, f;
    if (STYLE == kNeox) {
        a = load_f4<POL>(row + 8 * i, pol);
        b = load_f4<POL>(row + 8 * i + 4, pol);
        e = load_f4<POL>(row + h + 8 * i, pol);
        f = load_f4<POL>(row + h + 8 * i + 4, pol);
    } else {
        a = load_f4<POL>(row + 4 * i, pol);
        b = load_f4<POL>(row + 4 * i + (r >> 2), pol);
        e = load_f4<POL>(row + h + 4 * i, pol);
        f = load_f4<POL>(row + h + 4 * i + (r >> 2), pol);
    }
    c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
    c[4] = b.x; c[5] = b.y; c[6] = b.z; c[7] = b.w;
    s[0] = e.x; s[1] = e.y; s[2] = e.z; s[3] = e.w;
    s[4] = f.x; s[5] = f.y; s[6] = f.z; s[7] = f.w;
}

// NeoX: va holds dims 8i..8i+7 (first half), vb the partner dims 8i+r/2...;
// a' = a*c - b*s, b' = b*c + a*s with the frequency of the pair.
__device__ __forceinline__ void rotate_neox(uint4& va, uint4& vb, const float c[8],
                                            const float s[8])
{
    uint32_t* wa = reinterpret_cast<uint32_t*>(&va);
    uint32_t* wb = reinterpret_cast<uint32_t*>(&vb);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 a = __half22float2(h2(wa[k]));
        const float2 b = __half22float2(h2(wb[k]));
        const float c0 = c[2 * k], c1 = c[2 * k + 1];
        const float s0 = s[2 * k], s1 = s[2 * k + 1];
        const float ax = fmaf(a.x, c0, -(b.x * s0));
        const float ay = fmaf(a.y, c1, -(b.y * s1));
        const float bx = fmaf(b.x, c0, a.x * s0);
        const float by = fmaf(b.y, c1, a.y * s1);
        h2(wa[k]) = __floats2half2_rn(ax, ay);
        h2(wb[k]) = __floats2half2_rn(bx, by);
    }
}

// GPT-J: each half2 word is one (2j, 2j+1) pair; word k of the vector uses
// frequency c[k] / s[k].
__device__ __forceinline__ void rotate_gptj(uint4& v, const float* c, const float* s)
{
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 x = __half22float2(h2(w[k]));
        const float e = fmaf(x.x, c[k], -(x.y * s[k]));
        const float o = fmaf(x.y, c[k], x.x * s[k]);
        h2(w[k]) = __floats2half2_rn(e, o);
    }
}

// Unpack / pack 8 FP16 values of a 16-byte vector to / from FP32.
__device__ __forceinline__ void unpack8(uint4 v, float f[8])
{
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 x = __half22float2(h2(w[k]));
        f[2 * k] = x.x;
        f[2 * k + 1] = x.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float f[8])
{
    uint4 v;
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        h2(w[k]) = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
    return v;
}

// 8 FP32 values -> 8 E4M3 bytes: round to nearest even, saturating to the
// largest finite value (CUDA's satfinite conversion).
__device__ __forceinline__ uint2 pack8_e4m3(const float f[8])
{
    const uint32_t p0 = __nv_cvt_float2_to_fp8x2(make_float2(f[0], f[1]), __NV_SATFINITE, __NV_E4M3);
    const uint32_t p1 = __nv_cvt_float2_to_fp8x2(make_float2(f[2], f[3]), __NV_SATFINITE, __NV_E4M3);
    const uint32_t p2 = __nv_cvt_float2_to_fp8x2(make_float2(f[4], f[5]), __NV_SATFINITE, __NV_E4M3);
    const uint32_t p3 = __nv_cvt_float2_to_fp8x2(make_float2(f[6], f[7]), __NV_SATFINITE, __NV_E4M3);
    return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

template <int POL>
__device__ __forceinline__ void store_v8(uint8_t* p, const uint2& v, const L2Policies& pol)
{
    if (POL & kStreamHint) {
        asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;"
                     :: "l"(p), "r"(v.x), "r"(v.y), "l"(pol.stream)
                     : "memory");
        return;
    }
    *reinterpret_cast<uint2*>(p) = v;
}

// The rotation of rotate_item on FP32 values (fa, fb: the item's two vectors).
template <int STYLE>
__device__ __forceinline__ void rotate_item_f32(float fa[8], float fb[8], const float c[8],
                                                const float s[8])
{
    if (STYLE == kNeox) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float x = fa[k], y = fb[k];
            fa[k] = fmaf(x, c[k], -(y * s[k]));
            fb[k] = fmaf(y, c[k], x * s[k]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float e = fa[2 * j], o = fa[2 * j + 1];
            fa[2 * j] = fmaf(e, c[j], -(o * s[j]));
            fa[2 * j + 1] = fmaf(o, c[j], e * s[j]);
            e = fb[2 * j];
            o = fb[2 * j + 1];
            fb[2 * j] = fmaf(e, c[4 + j], -(o * s[4 + j]));
            fb[2 * j + 1] = fmaf(o, c[4 + j], e * s[4 + j]);
        }
    }
}

template <int STYLE>
__device__ __forceinline__ void rotate_item(uint4& va, uint4& vb, const float c[8],
                                            const float s[8])
{
    if (STYLE == kNeox) {
        rotate_neox(va, vb, c, s);
    } else {
        rotate_gptj(va, c, s);
        rotate_gptj(vb, c + 4, s + 4);
    }
}

// ------------------------------------------------- contiguous-cache kernel --
//
// Grid: tokens * ctasPerToken CTAs; CTA (token, part) covers items
// [part * blockDim * IPT, (part + 1) * blockDim * IPT) of the token, each thread
// items tid + k * blockDim for k < IPT. blockDim is a multiple of D/16.
//
// NORM (continuous only): every Q and K head is first RMS-normalized over its D
// dims with its weight vector, x * rsqrt(mean(x^2) + eps) * w, in FP32, then
// rotated, then rounded once. A head's D/16 items sit in D/16 consecutive lanes
// of one warp (items are head-major and blocks are whole warps), so the sum of
// squares is one xor-shuffle reduction over those lanes.
//
// FP8 (continuous only): the cache is E4M3; K (after the rotation, in FP32)
// and V are multiplied by 1/kScale and 1/vScale and stored as 8-byte vectors
// ("rope_cache.py", Stage 3.3). Q is written in FP16 as usual.
template <int D, int STYLE, int MODE, int IPT, int POL, bool NORM = false, bool FP8 = false>
__global__ void __launch_bounds__(256) rope_kv_token_kernel(const TokenArgs a)
{
    constexpr int kItemsPerHead = D / 16;
    const int tok = blockIdx.x / a.ctasPerToken;
    const int part = blockIdx.x - tok * a.ctasPerToken;
    const int b = tok / a.S;
    const int s = tok - b * a.S;
    const int H = a.Hq + 2 * a.Hkv;
    const int i = threadIdx.x % kItemsPerHead;
    const int item0 = part * blockDim.x * IPT + threadIdx.x;

    int va, vb;
    item_vectors<D>(i, a.r, va, vb);
    const uint16_t* tokIn = a.qkv + (size_t)tok * H * D;

    if ((POL & kPdl) && (POL & kPrefetch)) {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const int item = item0 + k * blockDim.x;
            if (item < a.itemsPerToken) {
                const uint16_t* p = tokIn + (size_t)(item / kItemsPerHead) * D;
                prefetch_l2(p + 8 * va);
                prefetch_l2(p + 8 * vb);
            }
        }
        if (MODE != kPacked && threadIdx.x == 0) {
            prefetch_l2(a.endLens + b);
            if (MODE == kTree)
                prefetch_l2(a.posIds + tok);
        }
    }
    grid_dependency_sync<POL>();
    const L2Policies pol = make_policies<POL>();
    const bool rotItem = i < (a.r >> 4);
    const int bcRow = (a.csBatch == 1) ? 0 : b;
    float c[8], sn[8];

    // 1. this thread's QKV vectors (independent of the position chain)
    uint4 xa[IPT] = {}, xb[IPT] = {};
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const int item = item0 + k * blockDim.x;
        if (item < a.itemsPerToken) {
            const int head = item / kItemsPerHead;
            const uint16_t* p = tokIn + (size_t)head * D;
            if (MODE == kPacked) {
                xa[k] = load_rw<POL>(p + 8 * va, pol);
                xb[k] = load_rw<POL>(p + 8 * vb, pol);
            } else {
                xa[k] = load_ro<POL>(p + 8 * va, pol);
                xb[k] = load_ro<POL>(p + 8 * vb, pol);
            }
        }
    }

    // 2. position (cos/sin row) and cache slot of the token
    int pos, slot;
    if (MODE == kPacked) {
        pos = s;
        slot = s;
    } else {
        slot = __ldg(a.endLens + b) - a.S + s;
        pos = (MODE == kTree) ? __ldg(a.posIds + tok) : slot;
        if (slot < 0 || slot >= a.cap || pos < 0 || pos >= a.csSeq)
            return;  // skipped token: nothing written
    }

    // 3. cos/sin for this thread's frequencies
    if (rotItem) {
        const float* row = a.cosSin + ((size_t)bcRow * a.csSeq + pos) * a.r;
        load_cos_sin<STYLE, POL>(row, i, a.r, c, sn, pol);
    }

    if (NORM) {
        // weights of this lane's 16 dims, for Q heads and for K heads (kept
        // packed, unpacked where used)
        const uint4 wqa = __ldg(reinterpret_cast<const uint4*>(a.qNormW + 8 * va));
        const uint4 wqb = __ldg(reinterpret_cast<const uint4*>(a.qNormW + 8 * vb));
        const uint4 wka = __ldg(reinterpret_cast<const uint4*>(a.kNormW + 8 * va));
        const uint4 wkb = __ldg(reinterpret_cast<const uint4*>(a.kNormW + 8 * vb));
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const int item = item0 + k * blockDim.x;
            const int head = item / kItemsPerHead;
            const bool qk = item < a.itemsPerToken && head < a.Hq + a.Hkv;
            uint32_t* wa_ = reinterpret_cast<uint32_t*>(&xa[k]);
            uint32_t* wb_ = reinterpret_cast<uint32_t*>(&xb[k]);
            float ss = 0.0f;
            if (qk) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 x = __half22float2(h2(wa_[q]));
                    const float2 y = __half22float2(h2(wb_[q]));
                    ss = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(y.x, y.x, fmaf(y.y, y.y, ss))));
                }
            }
            // all lanes take part: a head's lanes are aligned groups of D/16
#pragma unroll
            for (int off = 1; off < kItemsPerHead; off <<= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (!qk)
                continue;
            const float inv = rsqrtf(ss * (1.0f / D) + a.eps);
            const bool isQ = head < a.Hq;
            uint4 wA = isQ ? wqa : wka;
            uint4 wB = isQ ? wqb : wkb;
            uint32_t* wA_ = reinterpret_cast<uint32_t*>(&wA);
            uint32_t* wB_ = reinterpret_cast<uint32_t*>(&wB);
            // one half2 word of each vector at a time: normalize, rotate, pack
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float2 x = __half22float2(h2(wa_[q]));
                float2 y = __half22float2(h2(wb_[q]));
                const float2 u = __half22float2(h2(wA_[q]));
                const float2 v = __half22float2(h2(wB_[q]));
                x.x = x.x * inv * u.x;
                x.y = x.y * inv * u.y;
                y.x = y.x * inv * v.x;
                y.y = y.y * inv * v.y;
                if (rotItem) {
                    if (STYLE == kNeox) {
                        // dims 2q, 2q+1 of vector a pair with the same dims of b
                        const float c0 = c[2 * q], c1 = c[2 * q + 1];
                        const float s0 = sn[2 * q], s1 = sn[2 * q + 1];
                        const float ax = fmaf(x.x, c0, -(y.x * s0));
                        const float ay = fmaf(x.y, c1, -(y.y * s1));
                        const float bx = fmaf(y.x, c0, x.x * s0);
                        const float by = fmaf(y.y, c1, x.y * s1);
                        x = make_float2(ax, ay);
                        y = make_float2(bx, by);
                    } else {
                        // word q is one (2j, 2j+1) pair: frequency q in a, 4 + q in b
                        x = make_float2(fmaf(x.x, c[q], -(x.y * sn[q])), fmaf(x.y, c[q], x.x * sn[q]));
                        y = make_float2(fmaf(y.x, c[4 + q], -(y.y * sn[4 + q])),
                                        fmaf(y.y, c[4 + q], y.x * sn[4 + q]));
                    }
                }
                h2(wa_[q]) = __floats2half2_rn(x.x, x.y);
                h2(wb_[q]) = __floats2half2_rn(y.x, y.y);
            }
        }
    }

    // 4. rotate and store
    float invK = 1.0f, invV = 1.0f;
    if (FP8) {
        invK = 1.0f / __ldg(a.kScale);
        invV = 1.0f / __ldg(a.vScale);
    }
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const int item = item0 + k * blockDim.x;
        if (item >= a.itemsPerToken)
            continue;
        const int head = item / kItemsPerHead;
        if (FP8 && head >= a.Hq) {
            // K or V into the E4M3 cache: FP32 value times the inverse scale
            float fa[8], fb[8];
            unpack8(xa[k], fa);
            unpack8(xb[k], fb);
            const bool isK = head < a.Hq + a.Hkv;
            if (isK && rotItem)
                rotate_item_f32<STYLE>(fa, fb, c, sn);
            const float inv = isK ? invK : invV;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                fa[j] *= inv;
                fb[j] *= inv;
            }
            const int plane = isK ? 0 : 1;
            const int hk = isK ? head - a.Hq : head - a.Hq - a.Hkv;
            uint8_t* dst = a.cache8 + ((((size_t)b * 2 + plane) * a.Hkv + hk) * a.cap + slot) * D;
            store_v8<POL>(dst + 8 * va, pack8_e4m3(fa), pol);
            store_v8<POL>(dst + 8 * vb, pack8_e4m3(fb), pol);
            continue;
        }
        uint16_t* dst;
        if (head < a.Hq + a.Hkv) {
            if (!NORM && rotItem)
                rotate_item<STYLE>(xa[k], xb[k], c, sn);
            if (head < a.Hq) {
                dst = (MODE == kPacked) ? a.qkvOut + (size_t)tok * H * D + (size_t)head * D
                                        : a.qOut + ((size_t)tok * a.Hq + head) * D;
            } else {
                const int hk = head - a.Hq;
                if (MODE == kPacked) {
                    uint16_t* q = a.qkvOut + (size_t)tok * H * D + (size_t)head * D;
                    store_v<POL>(q + 8 * va, xa[k], pol);
                    store_v<POL>(q + 8 * vb, xb[k], pol);
                }
                dst = a.cache + ((((size_t)b * 2 + 0) * a.Hkv + hk) * a.cap + slot) * D;
            }
        } else {
            const int hv = head - a.Hq - a.Hkv;
            dst = a.cache + ((((size_t)b * 2 + 1) * a.Hkv + hv) * a.cap + slot) * D;
        }
        store_v<POL>(dst + 8 * va, xa[k], pol);
        store_v<POL>(dst + 8 * vb, xb[k], pol);
    }
}

// --------------------------------------------------------- paged kernel --
//
// Grid: rows * ctasPerRow CTAs; items [0, Hkv*D/16) are K heads, the rest V
// heads, split across the CTAs of a row like the token kernel.
//
// FUSED = false: row t's position and sequence come from deltaPositions /
// deltaTokenToSequence and its cos/sin from row t of the token-aligned table
// ("Dflash Runtime Kernels", launchDFlashTargetKVCacheUpdate).
// FUSED = true: the same update with the two preceding DFlash steps folded in
// (launchDFlashPrepareDeltaMetadata, launchDFlashGatherDeltaRope): row
// t = b * deltaWidth + j is sequence b's token j when j < deltaLens[b], at
// position oldLens[b] + j, and its cos/sin row is read straight from the source
// cache at (state row of b, position) -- a zero row when that is out of range,
// exactly as the gather would have produced.
template <int D, int STYLE, int IPT, int POL, bool FUSED>
__global__ void __launch_bounds__(256) paged_delta_kernel(const PagedArgs a)
{
    constexpr int kItemsPerHead = D / 16;
    grid_dependency_sync<POL>();
    const L2Policies pol = make_policies<POL>();
    const int t = blockIdx.x / a.ctasPerRow;
    const int part = blockIdx.x - t * a.ctasPerRow;
    const int i = threadIdx.x % kItemsPerHead;
    const int item0 = part * blockDim.x * IPT + threadIdx.x;
    const int kItems = a.Hkv * kItemsPerHead;

    int pos, seq;
    if (FUSED) {
        // a shift instead of the division when the width allows (this sits
        // ahead of the row's first load: 13.82 -> 13.57 us on 128 x 128 rows)
        seq = a.widthShift >= 0 ? t >> a.widthShift : t / a.deltaWidth;
        const int j = t - seq * a.deltaWidth;
        if (j >= __ldg(a.deltaLens + seq))
            return;  // padding row of the [B, deltaWidth] layout
        pos = __ldg(a.oldLens + seq) + j;
    } else {
        pos = __ldg(a.positions + t);
        seq = __ldg(a.seqIds + t);
    }
    if (pos < 0 || seq < 0 || seq >= a.B)
        return;  // padding row
    const int lp = pos / a.tpp;
    if (lp >= a.mpps)
        return;  // past the sequence's logical pages
    const int inPage = pos - lp * a.tpp;

    int va, vb;
    item_vectors<D>(i, a.r, va, vb);

    // delta rows (issued before the page-table lookups resolve)
    const size_t rowOff = (size_t)t * a.Hkv * D;
    uint4 xa[IPT] = {}, xb[IPT] = {};
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const int item = item0 + k * blockDim.x;
        if (item < a.itemsPerRow) {
            const bool isK = item < kItems;
            const int head = (isK ? item : item - kItems) / kItemsPerHead;
            const uint16_t* p = (isK ? a.kDelta : a.vDelta) + rowOff + (size_t)head * D;
            xa[k] = load_ro<POL>(p + 8 * va, pol);
            xb[k] = load_ro<POL>(p + 8 * vb, pol);
        }
    }

    const int32_t* pt = a.pageTable + (size_t)seq * 2 * a.mpps + lp;
    const int idK = __ldg(pt);
    const int idV = __ldg(pt + a.mpps);
    const bool kOk = idK >= 0 && idK < a.numPages;
    const bool vOk = idV >= a.numPages && (int64_t)idV < 2 * (int64_t)a.numPages;

    // cos/sin are loaded whether or not the K page is mapped, so that their
    // address does not wait for the page-table lookup (measured ~1 % faster)
    float c[8], sn[8];
    const bool rotItem = i < (a.r >> 4);
    if (rotItem) {
        if (FUSED) {
            int state = -1;
            if (pos < a.cacheCapacity)
                state = a.stateIdx ? __ldg(a.stateIdx + seq) : (a.sourceRows == 1 ? 0 : seq);
            if (state >= 0 && state < a.sourceRows) {
                load_cos_sin<STYLE, POL>(a.cosSin + ((size_t)state * a.cacheCapacity + pos) * a.r,
                                         i, a.r, c, sn, pol);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    c[k] = 0.0f;
                    sn[k] = 0.0f;
                }
            }
        } else {
            load_cos_sin<STYLE, POL>(a.cosSin + (size_t)t * a.r, i, a.r, c, sn, pol);
        }
    }

    const size_t rowElems = (size_t)a.Hkv * D;
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const int item = item0 + k * blockDim.x;
        if (item >= a.itemsPerRow)
            continue;
        const bool isK = item < kItems;
        if (isK ? !kOk : !vOk)
            continue;
        const int head = (isK ? item : item - kItems) / kItemsPerHead;
        if (isK && rotItem)
            rotate_item<STYLE>(xa[k], xb[k], c, sn);
        const int id = isK ? idK : idV;  // flat page index of the [2, numPages] pool
        uint16_t* dst = a.pool + ((size_t)id * a.tpp + inPage) * rowElems + (size_t)head * D;
        store_v<POL>(dst + 8 * va, xa[k], pol);
        store_v<POL>(dst + 8 * vb, xb[k], pol);
    }
}

// ------------------------------------------------- slot-mapping kernel --
//
// sglang rope_cache.py, fused_qk_rope_reshape_and_cache (flash layout): Q, K, V
// come as separate token-strided tensors, each token carries its own RoPE
// position and one flat cache slot (block = slot / blockSize, offset =
// slot % blockSize, which for the [blocks, blockSize, Hkv, D] layout is simply
// row `slot`). Rotated Q always goes to qOut; a negative slot (or one past the
// caches) skips the K/V cache writes and kOut (Stage 3.1-3.5). Same item
// decomposition as rope_kv_token_kernel; every K/V vector has one writer, so no
// GQA group leader is needed.
template <int D, int STYLE, int IPT, int POL>
__global__ void __launch_bounds__(256) rope_kv_slotmap_kernel(const SlotMapArgs a)
{
    constexpr int kItemsPerHead = D / 16;
    const int tok = blockIdx.x / a.ctasPerToken;
    const int part = blockIdx.x - tok * a.ctasPerToken;
    const int i = threadIdx.x % kItemsPerHead;
    const int item0 = part * blockDim.x * IPT + threadIdx.x;
    const int qkHeads = a.Hq + a.Hkv;

    int va, vb;
    item_vectors<D>(i, a.r, va, vb);

    if ((POL & kPdl) && (POL & kPrefetch)) {
        // L2 prefetches only (see kPrefetch): inputs, the position and the slot
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const int item = item0 + k * blockDim.x;
            if (item < a.itemsPerToken) {
                const int head = item / kItemsPerHead;
                const uint16_t* p = head < a.Hq ? a.q + tok * a.qStride + (size_t)head * D
                                  : head < qkHeads ? a.k + tok * a.kStride + (size_t)(head - a.Hq) * D
                                  : a.v + tok * a.vStride + (size_t)(head - qkHeads) * D;
                prefetch_l2(p + 8 * va);
                prefetch_l2(p + 8 * vb);
            }
        }
        if (threadIdx.x == 0) {
            prefetch_l2(a.positions + tok);
            prefetch_l2(a.slots + tok);
        }
    }
    grid_dependency_sync<POL>();
    const L2Policies pol = make_policies<POL>();
    const bool rotItem = i < (a.r >> 4);
    float c[8], sn[8];

    uint4 xa[IPT] = {}, xb[IPT] = {};
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const int item = item0 + k * blockDim.x;
        if (item < a.itemsPerToken) {
            const int head = item / kItemsPerHead;
            const uint16_t* p;
            if (head < a.Hq)
                p = a.q + tok * a.qStride + (size_t)head * D;
            else if (head < qkHeads)
                p = a.k + tok * a.kStride + (size_t)(head - a.Hq) * D;
            else
                p = a.v + tok * a.vStride + (size_t)(head - qkHeads) * D;
            xa[k] = load_ro<POL>(p + 8 * va, pol);
            xb[k] = load_ro<POL>(p + 8 * vb, pol);
        }
    }

    const int64_t pos = __ldg(a.positions + tok);
    if (pos < 0 || pos >= a.csRows)
        return;  // no cos/sin row: nothing written for the token
    const int64_t slot = __ldg(a.slots + tok);
    const bool kvOk = slot >= 0 && slot < a.numSlots;

    if (rotItem)
        load_cos_sin<STYLE, POL>(a.cosSin + pos * a.r, i, a.r, c, sn, pol);

#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const int item = item0 + k * blockDim.x;
        if (item >= a.itemsPerToken)
            continue;
        const int head = item / kItemsPerHead;
        if (head < a.Hq) {
            if (rotItem)
                rotate_item<STYLE>(xa[k], xb[k], c, sn);
            uint16_t* dst = a.qOut + ((size_t)tok * a.Hq + head) * D;
            store_v<POL>(dst + 8 * va, xa[k], pol);
            store_v<POL>(dst + 8 * vb, xb[k], pol);
            continue;
        }
        if (!kvOk)
            continue;
        if (head < qkHeads) {
            const int hk = head - a.Hq;
            if (rotItem)
                rotate_item<STYLE>(xa[k], xb[k], c, sn);
            uint16_t* dst = a.keyCache + ((size_t)slot * a.Hkv + hk) * D;
            store_v<POL>(dst + 8 * va, xa[k], pol);
            store_v<POL>(dst + 8 * vb, xb[k], pol);
            if (a.kOut != nullptr) {
                uint16_t* ko = a.kOut + ((size_t)tok * a.Hkv + hk) * D;
                store_v<POL>(ko + 8 * va, xa[k], pol);
                store_v<POL>(ko + 8 * vb, xb[k], pol);
            }
        } else {
            uint16_t* dst = a.valueCache + ((size_t)slot * a.Hkv + (head - qkHeads)) * D;
            store_v<POL>(dst + 8 * va, xa[k], pol);
            store_v<POL>(dst + 8 * vb, xb[k], pol);
        }
    }
}

// ------------------------------------------------- DFlash prologue kernels --
//
// "Dflash Runtime Kernels", launchDFlashPrepareDeltaMetadata (signature only on
// the page; rows laid out [B, width]): one thread per row.
__global__ void __launch_bounds__(256) delta_metadata_kernel(const DeltaMetaArgs a)
{
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (long long)a.B * a.width)
        return;
    const int b = (int)(t / a.width);
    const int j = (int)(t - (long long)b * a.width);
    const bool valid = j < __ldg(a.deltaLens + b);
    a.positions[t] = valid ? __ldg(a.oldLens + b) + j : -1;
    a.seqIds[t] = valid ? b : -1;
}

// launchDFlashGatherDeltaRope (signature only on the page): one thread per
// float4 of an output row; zero rows where the source has no row.
__global__ void __launch_bounds__(256) gather_delta_rope_kernel(const GatherArgs a)
{
    const int q4 = a.r >> 2;
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= (long long)a.N * q4)
        return;
    const int t = (int)(g / q4);
    const int q = (int)(g - (long long)t * q4);
    const int pos = __ldg(a.positions + t);
    const int seq = __ldg(a.seqIds + t);
    int state = -1;
    if (pos >= 0 && seq >= 0 && seq < a.B && pos < a.cacheCapacity)
        state = a.stateIdx ? __ldg(a.stateIdx + seq) : (a.sourceRows == 1 ? 0 : seq);
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (state >= 0 && state < a.sourceRows)
        v = __ldg(reinterpret_cast<const float4*>(
                a.source + ((size_t)state * a.cacheCapacity + pos) * a.r) + q);
    reinterpret_cast<float4*>(a.output + (size_t)t * a.r)[q] = v;
}

}  // namespace ropekv
