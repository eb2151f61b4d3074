// ropekv_api.cu -- the C ABI of libropekv.so: host-side argument checks, the
// choice of kernel instantiation and launch shape, and one launch per call on
// the caller's stream. Declarations and the meaning of every argument are in
// include/ropekv.h. Nothing here allocates or synchronises; the only state is
// a per-kernel record of the devices on which its dynamic shared memory limit
// was raised (see residency_smem) and the process-wide residency-cap switch.
// Every entry point returns the status of its own launch: the library never
// reads or clears CUDA's per-thread "last error" for the caller.
#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include "ropekv.h"
#include "ropekv_kernels.cuh"

namespace {

using ropekv::PagedArgs;
using ropekv::TokenArgs;

bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

int check_head_dims(int32_t D, int32_t r)
{
    if (D != 64 && D != 128 && D != 256)
        return ROPEKV_ERR_HEAD_DIM;
    if (r < 16 || r > D || (r % 16) != 0)
        return ROPEKV_ERR_ROTARY_DIM;
    return ROPEKV_OK;
}

// Launch shape for `units` tokens (or rows) of `items` items each.
// Measured on GB300 over the prefill, decode, tree and paged workloads:
//   * two items per thread and up to 384 items per CTA: one 192-thread CTA per
//     token of 32 + 2 x 8 heads of 128 dims, one 64-thread CTA per paged row
//     of 8 + 8 heads. With dependent launch, the 8192-token prefill takes
//     30.30 us this way against 30.60 us with three 64-thread CTAs per token
//     (no dependent launch: at that CTA count its launch-rate cap hurt), and
//     the 4096-token tree 15.96 against 16.02 us;
//   * small launches (< 1024 units, decode) take up to 192 items per CTA --
//     two 96-thread CTAs per Llama token -- and add the residency cap below.
//     256 decode tokens, back to back: 2.15 -> 2.12 us (FP8 2.18 -> 2.15,
//     slot mapping 2.30 -> 2.28, QK-normalized 2.48 either way) against one
//     192-thread CTA per token; three 64-thread CTAs 2.14 us; one item per
//     thread in two or three CTAs per token 2.39 us;
//   * the large QK-normalized launch, ~3x the arithmetic per byte, keeps 32
//     threads x 4 items per CTA (more loads in flight per thread; 96 x 4 with
//     dependent launch: 31.60 us, the same), and the large FP8-cache launch
//     64 x 2 (8192 tokens: 28.53 us; 192 x 2 with dependent launch: 29.14 us).
// Blocks are whole warps; a warp's size is a multiple of every D/16, which
// keeps each thread on one item index.
struct Shape {
    int threads;
    int ipt;
    int ctasPerUnit;
    bool small;  // dependent launch with the prefetch prologue and a residency cap
};

enum class Work { kPlain, kNorm, kFp8 };

Shape pick_shape(int items, long long units, Work work = Work::kPlain)
{
    Shape sh;
    int perCta;
    sh.small = units < 1024;
    if (sh.small) {
        sh.ipt = 2;
        perCta = 192;
    } else if (work == Work::kPlain) {
        sh.ipt = 2;
        perCta = 384;
    } else if (work == Work::kNorm) {
        sh.ipt = 4;
        perCta = 128;
    } else {
        sh.ipt = 2;
        perCta = 128;
    }
    sh.ctasPerUnit = (items + perCta - 1) / perCta;
    const int per = (items + sh.ctasPerUnit * sh.ipt - 1) / (sh.ctasPerUnit * sh.ipt);
    sh.threads = ((per + 31) / 32) * 32;
    return sh;
}

// Kernel policies (see ropekv_kernels.cuh), measured on GB300:
//   * every launch: streaming L2 hints on activations and cache rows, and
//     cos/sin rows kept in L2 (evict-last; against no hint: paged update 21.25
//     -> 21.10 us, QK-normalized decode 2.47 -> 2.45 us, tree 16.04 -> 16.01,
//     the others within 0.2 %);
//   * small (decode-sized) token and slot-mapping launches: programmatic
//     dependent launch with the L2 prefetch prologue, which brings the
//     inputs and the index words into L2 while the previous kernel in the
//     stream drains (256 decode tokens: 3.01 -> 1.90 us per launch with the
//     residency cap below; the position -> cos/sin chain itself stays after
//     the wait, one L2 round trip longer than a plain copy);
//   * larger token and slot-mapping launches: dependent launch (tree: 16.56
//     -> 16.17 us) when the grid has at most kPdlMaxCtas CTAs or its CTAs
//     cover at least 256 items; plain continuous, packed and slot-mapping
//     launches also take the prefetch prologue (8192-token prefill 30.24 ->
//     29.99 us, 2048 one-token decodes 8.93 -> 8.33 us, 4096-token prefill
//     16.15 -> 15.65 us; slot mapping, 1024 one-token decodes 5.71 -> 5.39
//     us, 8192 tokens 30.55 -> 30.47 us), the QK-normalized and FP8-cache
//     ones do not (2048 tokens: 10.51 -> 11.53 and 8.77 -> 9.74 us with it;
//     8192 tokens unchanged), nor do tree launches (1024 tokens 5.35 -> 5.55
//     us with it, 4096 tokens 16.30 -> 16.25 us). The attribute
//     caps the CTA launch rate near one CTA per nanosecond, which starves
//     grids of many short CTAs (a 49 152-CTA prefill of 128-item CTAs: 29.9 ->
//     49.8 us); a 256-item CTA moves ~16 KB, more than HBM delivers in a
//     nanosecond. The paged kernels (128-item CTAs, many of them padding or
//     short) launch without it (the fused update: 13.9 -> 17.3 us with it).
// Kernels that do not wait on the previous grid (the DFlash metadata and
// gather kernels) never get the dependent-launch attribute.
constexpr int kPolLarge = ropekv::kStreamHint | ropekv::kTableKeep;
constexpr int kPolPdl = ropekv::kStreamHint | ropekv::kTableKeep | ropekv::kPdl;
constexpr int kPolSmall = ropekv::kStreamHint | ropekv::kTableKeep | ropekv::kPdl | ropekv::kPrefetch;
constexpr long long kPdlMaxCtas = 12288;

bool pdl_allowed(unsigned grid, const Shape& sh)
{
    return grid <= kPdlMaxCtas || sh.threads * sh.ipt >= 256;
}

// One launch; returns ROPEKV_OK or ROPEKV_ERR_LAUNCH from this launch's own
// result (cudaLaunchKernelEx reports configuration errors of this launch; an
// error left pending by earlier work in the context may also surface here).
template <typename Args>
int launch_k(void (*kern)(Args), unsigned grid, int threads, cudaStream_t st, bool pdl,
             const Args& a, size_t smem = 0)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? ROPEKV_OK : ROPEKV_ERR_LAUNCH;
}

// Process-wide switch of the residency cap below (ropekv_set_residency_cap).
std::atomic<int> g_residency_cap{1};

// Residency cap of a small dependent launch. A launch that starts while its
// predecessor still runs gets its CTAs placed densely: a per-warp timer trace
// of 512 decode CTAs of 192 threads found them on 61-66 of the 152 SMs, up to
// ten per SM, and the launch then lasts as long as the most loaded SMs take to
// issue their work. Dynamic shared memory that the kernel does not use, sized
// so that at most ceil(grid / SMs) CTAs fit on one SM, spreads the CTAs over
// the GPU (256 decode tokens: 2.40 -> 2.07 us per launch). Returns 0 (no cap)
// for grids of more than 8 CTAs per SM, when the caller switched the cap off
// or when the device cannot be queried (the launch then goes ahead uncapped);
// *optin receives the device's per-block shared memory limit.
size_t residency_smem(unsigned grid, int* optin)
{
    int dev = 0, sms = 0, perSm = 0, reserved = 0;
    *optin = 0;
    if (!g_residency_cap.load(std::memory_order_relaxed))
        return 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&perSm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess || sms <= 0) {
        return 0;
    }
    const unsigned cap = (grid + (unsigned)sms - 1) / (unsigned)sms;
    if (cap == 0 || cap > 8)
        return 0;
    long long bytes = (long long)perSm / cap - reserved;
    if (bytes > *optin)
        bytes = *optin;
    return bytes > 0 ? (size_t)(bytes & ~255LL) : 0;
}

// Launch of a small dependent kernel with its residency cap. A kernel's
// dynamic shared memory limit is raised from the default 48 KB to the
// device's maximum once per device (one bit per device ordinal below 64;
// higher ordinals raise it on every call) -- the only state the library keeps.
template <auto Kern, typename Args>
int launch_small(unsigned grid, int threads, cudaStream_t st, const Args& a)
{
    int optin = 0;
    size_t smem = residency_smem(grid, &optin);
    if (smem > 48 * 1024) {
        static std::atomic<unsigned long long> raised{0};
        int dev = 0;
        (void)cudaGetDevice(&dev);
        const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ULL << dev : 0;
        if (!bit || !(raised.load(std::memory_order_relaxed) & bit)) {
            if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) ==
                cudaSuccess) {
                raised.fetch_or(bit, std::memory_order_relaxed);
            } else {
                smem = 0;  // launch without the cap rather than fail
            }
        }
    }
    return launch_k(Kern, grid, threads, st, true, a, smem);
}

template <int D, int STYLE, int MODE, int IPT, bool NORM, bool FP8>
int launch_token_variant(const TokenArgs& a, unsigned grid, const Shape& sh, cudaStream_t st)
{
    if constexpr (IPT == 2) {
        if (sh.small)
            return launch_small<
                ropekv::rope_kv_token_kernel<D, STYLE, MODE, IPT, kPolSmall, NORM, FP8>>(
                grid, sh.threads, st, a);
    }
    constexpr int kPolMid =
        (MODE != ropekv::kTree && !NORM && !FP8) ? (kPolPdl | ropekv::kPrefetch) : kPolPdl;
    if (pdl_allowed(grid, sh))
        return launch_k(ropekv::rope_kv_token_kernel<D, STYLE, MODE, IPT, kPolMid, NORM, FP8>,
                        grid, sh.threads, st, true, a);
    return launch_k(ropekv::rope_kv_token_kernel<D, STYLE, MODE, IPT, kPolLarge, NORM, FP8>, grid,
                    sh.threads, st, false, a);
}

template <int D, int STYLE, int MODE, int IPT>
int launch_token(const TokenArgs& a, long long tokens, const Shape& sh, cudaStream_t st)
{
    const unsigned grid = (unsigned)(tokens * sh.ctasPerUnit);
    if constexpr (MODE == ropekv::kContinuous) {
        if (a.qNormW != nullptr)
            return launch_token_variant<D, STYLE, MODE, IPT, true, false>(a, grid, sh, st);
        if (a.cache8 != nullptr) {
            if constexpr (IPT != 4)
                return launch_token_variant<D, STYLE, MODE, IPT, false, true>(a, grid, sh, st);
            return ROPEKV_ERR_LAUNCH;  // pick_shape never gives the FP8 call 4 items
        }
    }
    if constexpr (IPT != 4)
        return launch_token_variant<D, STYLE, MODE, IPT, false, false>(a, grid, sh, st);
    return ROPEKV_ERR_LAUNCH;  // 4 items per thread: the normalized call only
}

template <int D, int STYLE, int MODE>
int dispatch_ipt(const TokenArgs& a, long long tokens, const Shape& sh, cudaStream_t st)
{
    if (sh.ipt == 4) {
        if constexpr (MODE == ropekv::kContinuous)
            return launch_token<D, STYLE, MODE, 4>(a, tokens, sh, st);  // the normalized call only
        return ROPEKV_ERR_LAUNCH;
    }
    return launch_token<D, STYLE, MODE, 2>(a, tokens, sh, st);
}

template <int D, int MODE>
int dispatch_style(const TokenArgs& a, int style, long long tokens, const Shape& sh,
                   cudaStream_t st)
{
    if (style == ROPEKV_GPTJ)
        return dispatch_ipt<D, ropekv::kGptj, MODE>(a, tokens, sh, st);
    return dispatch_ipt<D, ropekv::kNeox, MODE>(a, tokens, sh, st);
}

template <int MODE>
int dispatch_token(const TokenArgs& a, int D, int style, long long tokens, const Shape& sh,
                   cudaStream_t st)
{
    switch (D) {
    case 64: return dispatch_style<64, MODE>(a, style, tokens, sh, st);
    case 128: return dispatch_style<128, MODE>(a, style, tokens, sh, st);
    default: return dispatch_style<256, MODE>(a, style, tokens, sh, st);
    }
}

template <int D, int STYLE, bool FUSED>
int launch_paged(const PagedArgs& a, long long rows, const Shape& sh, cudaStream_t st)
{
    // pick_shape gives the paged rows (never "heavy") two items per thread
    const unsigned grid = (unsigned)(rows * sh.ctasPerUnit);
    return launch_k(ropekv::paged_delta_kernel<D, STYLE, 2, kPolLarge, FUSED>, grid, sh.threads,
                    st, false, a);
}

template <bool FUSED>
int dispatch_paged(const PagedArgs& a, int D, int style, long long rows, const Shape& sh,
                   cudaStream_t st)
{
    const bool gptj = style == ROPEKV_GPTJ;
    switch (D) {
    case 64:
        return gptj ? launch_paged<64, ropekv::kGptj, FUSED>(a, rows, sh, st)
                    : launch_paged<64, ropekv::kNeox, FUSED>(a, rows, sh, st);
    case 128:
        return gptj ? launch_paged<128, ropekv::kGptj, FUSED>(a, rows, sh, st)
                    : launch_paged<128, ropekv::kNeox, FUSED>(a, rows, sh, st);
    default:
        return gptj ? launch_paged<256, ropekv::kGptj, FUSED>(a, rows, sh, st)
                    : launch_paged<256, ropekv::kNeox, FUSED>(a, rows, sh, st);
    }
}

// Checks shared by both paged calls (sizes and style).
int check_paged_sizes(int32_t numRows, int32_t batchSize, int32_t numKVHeads, int32_t headDim,
                      int32_t rotaryDim, int32_t numPages, int32_t maxPagesPerSeq,
                      int32_t tokensPerPage, int32_t style)
{
    if (style != ROPEKV_NEOX && style != ROPEKV_GPTJ)
        return ROPEKV_ERR_STYLE;
    int rc = check_head_dims(headDim, rotaryDim);
    if (rc != ROPEKV_OK)
        return rc;
    if (numKVHeads <= 0)
        return ROPEKV_ERR_HEADS;
    if (numRows < 0 || batchSize < 0 || numPages < 0 || maxPagesPerSeq < 0 || tokensPerPage <= 0)
        return ROPEKV_ERR_SHAPE;
    if (2LL * numKVHeads * (headDim / 16) > (1LL << 30))
        return ROPEKV_ERR_SHAPE;
    return ROPEKV_OK;
}

int launch_paged_rows(PagedArgs& a, long long rows, int D, int style, bool fused, cudaStream_t st)
{
    const Shape sh = pick_shape(a.itemsPerRow, rows);
    if (rows * sh.ctasPerUnit > 0x7FFFFFFFLL)
        return ROPEKV_ERR_SHAPE;
    a.ctasPerRow = sh.ctasPerUnit;
    return fused ? dispatch_paged<true>(a, D, style, rows, sh, st)
                 : dispatch_paged<false>(a, D, style, rows, sh, st);
}

// Checks shared by the three contiguous-cache calls. On success fills the
// kernel arguments that depend only on the sizes and returns the token count.
int check_dims(const ropekv_dims* d, long long* tokens)
{
    if (d == nullptr)
        return ROPEKV_ERR_NULL_POINTER;
    if (d->style != ROPEKV_NEOX && d->style != ROPEKV_GPTJ)
        return ROPEKV_ERR_STYLE;
    int rc = check_head_dims(d->headDim, d->rotaryDim);
    if (rc != ROPEKV_OK)
        return rc;
    if (d->numQHeads <= 0 || d->numKVHeads <= 0 || d->numQHeads % d->numKVHeads != 0)
        return ROPEKV_ERR_HEADS;
    if (d->batch < 0 || d->seqLen < 0 || d->kvCapacity < 0 || d->cosSinSeqLen < 0)
        return ROPEKV_ERR_SHAPE;
    if (d->cosSinBatch != 1 && d->cosSinBatch != d->batch)
        return ROPEKV_ERR_COS_SIN_BATCH;
    const long long H = (long long)d->numQHeads + 2LL * d->numKVHeads;
    if (H * (d->headDim / 16) > (1LL << 30))
        return ROPEKV_ERR_SHAPE;
    *tokens = (long long)d->batch * d->seqLen;
    return ROPEKV_OK;
}

TokenArgs token_args(const ropekv_dims* d)
{
    TokenArgs a = {};
    a.S = d->seqLen;
    a.Hq = d->numQHeads;
    a.Hkv = d->numKVHeads;
    a.r = d->rotaryDim;
    a.cap = d->kvCapacity;
    a.csBatch = d->cosSinBatch;
    a.csSeq = d->cosSinSeqLen;
    a.itemsPerToken = (d->numQHeads + 2 * d->numKVHeads) * (d->headDim / 16);
    return a;
}

int launch_contiguous(TokenArgs a, const ropekv_dims* d, long long tokens, int mode,
                      cudaStream_t st)
{
    const Shape sh = pick_shape(a.itemsPerToken, tokens,
                                a.qNormW != nullptr  ? Work::kNorm
                                : a.cache8 != nullptr ? Work::kFp8
                                                      : Work::kPlain);
    if (tokens * sh.ctasPerUnit > 0x7FFFFFFFLL)
        return ROPEKV_ERR_SHAPE;
    a.ctasPerToken = sh.ctasPerUnit;
    switch (mode) {
    case ropekv::kPacked:
        return dispatch_token<ropekv::kPacked>(a, d->headDim, d->style, tokens, sh, st);
    case ropekv::kContinuous:
        return dispatch_token<ropekv::kContinuous>(a, d->headDim, d->style, tokens, sh, st);
    default:
        return dispatch_token<ropekv::kTree>(a, d->headDim, d->style, tokens, sh, st);
    }
}

template <int D>
int launch_slotmap(const ropekv::SlotMapArgs& a, bool gptj, unsigned grid, const Shape& sh,
                   cudaStream_t st)
{
    using ropekv::rope_kv_slotmap_kernel;
    if (sh.small)
        return gptj ? launch_small<rope_kv_slotmap_kernel<D, ropekv::kGptj, 2, kPolSmall>>(
                          grid, sh.threads, st, a)
                    : launch_small<rope_kv_slotmap_kernel<D, ropekv::kNeox, 2, kPolSmall>>(
                          grid, sh.threads, st, a);
    if (pdl_allowed(grid, sh))
        return gptj ? launch_k(rope_kv_slotmap_kernel<D, ropekv::kGptj, 2, kPolPdl | ropekv::kPrefetch>, grid,
                               sh.threads, st, true, a)
                    : launch_k(rope_kv_slotmap_kernel<D, ropekv::kNeox, 2, kPolPdl | ropekv::kPrefetch>, grid,
                               sh.threads, st, true, a);
    return gptj ? launch_k(rope_kv_slotmap_kernel<D, ropekv::kGptj, 2, kPolLarge>, grid,
                           sh.threads, st, false, a)
                : launch_k(rope_kv_slotmap_kernel<D, ropekv::kNeox, 2, kPolLarge>, grid,
                           sh.threads, st, false, a);
}

}  // namespace

extern "C" {

int rope_write_kv_packed(const float* cosSin, uint16_t* qkv, uint16_t* kvCache,
                         const ropekv_dims* dims, void* stream)
{
    long long tokens = 0;
    int rc = check_dims(dims, &tokens);
    if (rc != ROPEKV_OK)
        return rc;
    if (dims->seqLen > dims->kvCapacity || dims->seqLen > dims->cosSinSeqLen)
        return ROPEKV_ERR_CAPACITY;
    if (tokens == 0)
        return ROPEKV_OK;
    if (!cosSin || !qkv || !kvCache)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(cosSin) || !aligned16(qkv) || !aligned16(kvCache))
        return ROPEKV_ERR_MISALIGNED;
    TokenArgs a = token_args(dims);
    a.cosSin = cosSin;
    a.qkv = qkv;
    a.qkvOut = qkv;
    a.cache = kvCache;
    return launch_contiguous(a, dims, tokens, ropekv::kPacked, (cudaStream_t)stream);
}

int rope_write_kv_continuous(const float* cosSin, const int32_t* kvCacheEndLens,
                             const uint16_t* qkv, uint16_t* kvCache, uint16_t* qOut,
                             const ropekv_dims* dims, void* stream)
{
    long long tokens = 0;
    int rc = check_dims(dims, &tokens);
    if (rc != ROPEKV_OK)
        return rc;
    if (tokens == 0)
        return ROPEKV_OK;
    if (!cosSin || !kvCacheEndLens || !qkv || !kvCache || !qOut)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(cosSin) || !aligned16(kvCacheEndLens) || !aligned16(qkv) ||
        !aligned16(kvCache) || !aligned16(qOut))
        return ROPEKV_ERR_MISALIGNED;
    TokenArgs a = token_args(dims);
    a.cosSin = cosSin;
    a.endLens = kvCacheEndLens;
    a.qkv = qkv;
    a.cache = kvCache;
    a.qOut = qOut;
    return launch_contiguous(a, dims, tokens, ropekv::kContinuous, (cudaStream_t)stream);
}

int rope_write_kv_continuous_qknorm(const float* cosSin, const int32_t* kvCacheEndLens,
                                    const uint16_t* qkv, uint16_t* kvCache, uint16_t* qOut,
                                    const uint16_t* qNormWeight, const uint16_t* kNormWeight,
                                    float eps, const ropekv_dims* dims, void* stream)
{
    long long tokens = 0;
    int rc = check_dims(dims, &tokens);
    if (rc != ROPEKV_OK)
        return rc;
    if (!(eps >= 0.0f) || eps > 1.0e30f)
        return ROPEKV_ERR_SHAPE;
    if (tokens == 0)
        return ROPEKV_OK;
    if (!cosSin || !kvCacheEndLens || !qkv || !kvCache || !qOut || !qNormWeight || !kNormWeight)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(cosSin) || !aligned16(kvCacheEndLens) || !aligned16(qkv) ||
        !aligned16(kvCache) || !aligned16(qOut) || !aligned16(qNormWeight) ||
        !aligned16(kNormWeight))
        return ROPEKV_ERR_MISALIGNED;
    TokenArgs a = token_args(dims);
    a.cosSin = cosSin;
    a.endLens = kvCacheEndLens;
    a.qkv = qkv;
    a.cache = kvCache;
    a.qOut = qOut;
    a.qNormW = qNormWeight;
    a.kNormW = kNormWeight;
    a.eps = eps;
    return launch_contiguous(a, dims, tokens, ropekv::kContinuous, (cudaStream_t)stream);
}

int rope_write_kv_continuous_fp8(const float* cosSin, const int32_t* kvCacheEndLens,
                                 const uint16_t* qkv, uint8_t* kvCache8, uint16_t* qOut,
                                 const float* kScale, const float* vScale,
                                 const ropekv_dims* dims, void* stream)
{
    long long tokens = 0;
    int rc = check_dims(dims, &tokens);
    if (rc != ROPEKV_OK)
        return rc;
    if (tokens == 0)
        return ROPEKV_OK;
    if (!cosSin || !kvCacheEndLens || !qkv || !kvCache8 || !qOut || !kScale || !vScale)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(cosSin) || !aligned16(kvCacheEndLens) || !aligned16(qkv) ||
        !aligned16(kvCache8) || !aligned16(qOut) || !aligned16(kScale) || !aligned16(vScale))
        return ROPEKV_ERR_MISALIGNED;
    TokenArgs a = token_args(dims);
    a.cosSin = cosSin;
    a.endLens = kvCacheEndLens;
    a.qkv = qkv;
    a.cache8 = kvCache8;
    a.qOut = qOut;
    a.kScale = kScale;
    a.vScale = vScale;
    return launch_contiguous(a, dims, tokens, ropekv::kContinuous, (cudaStream_t)stream);
}

int rope_write_kv_tree(const float* cosSin, const int32_t* kvCacheEndLens,
                       const int32_t* tokenPosIds, const uint16_t* qkv, uint16_t* kvCache,
                       uint16_t* qOut, const ropekv_dims* dims, void* stream)
{
    long long tokens = 0;
    int rc = check_dims(dims, &tokens);
    if (rc != ROPEKV_OK)
        return rc;
    if (tokens == 0)
        return ROPEKV_OK;
    if (!cosSin || !kvCacheEndLens || !tokenPosIds || !qkv || !kvCache || !qOut)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(cosSin) || !aligned16(kvCacheEndLens) || !aligned16(tokenPosIds) ||
        !aligned16(qkv) || !aligned16(kvCache) || !aligned16(qOut))
        return ROPEKV_ERR_MISALIGNED;
    TokenArgs a = token_args(dims);
    a.cosSin = cosSin;
    a.endLens = kvCacheEndLens;
    a.posIds = tokenPosIds;
    a.qkv = qkv;
    a.cache = kvCache;
    a.qOut = qOut;
    return launch_contiguous(a, dims, tokens, ropekv::kTree, (cudaStream_t)stream);
}

int paged_kv_delta_update(const uint16_t* kDelta, const uint16_t* vDelta, uint16_t* kvCache,
                          const float* tokenAlignedCosSin, const int32_t* deltaPositions,
                          const int32_t* deltaTokenToSequence, const int32_t* pageTable,
                          int32_t numDeltaTokens, int32_t batchSize, int32_t numKVHeads,
                          int32_t headDim, int32_t rotaryDim, int32_t numPages,
                          int32_t maxPagesPerSeq, int32_t tokensPerPage, int32_t style,
                          void* stream)
{
    int rc = check_paged_sizes(numDeltaTokens, batchSize, numKVHeads, headDim, rotaryDim,
                               numPages, maxPagesPerSeq, tokensPerPage, style);
    if (rc != ROPEKV_OK)
        return rc;
    if (numDeltaTokens == 0)
        return ROPEKV_OK;
    if (!kDelta || !vDelta || !kvCache || !tokenAlignedCosSin || !deltaPositions ||
        !deltaTokenToSequence || (!pageTable && batchSize > 0))
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(kDelta) || !aligned16(vDelta) || !aligned16(kvCache) ||
        !aligned16(tokenAlignedCosSin) || !aligned16(deltaPositions) ||
        !aligned16(deltaTokenToSequence) || !aligned16(pageTable))
        return ROPEKV_ERR_MISALIGNED;
    if (batchSize == 0)
        return ROPEKV_OK;  // every row names a sequence >= batchSize: nothing to write
    PagedArgs a = {};
    a.kDelta = kDelta;
    a.vDelta = vDelta;
    a.pool = kvCache;
    a.cosSin = tokenAlignedCosSin;
    a.positions = deltaPositions;
    a.seqIds = deltaTokenToSequence;
    a.pageTable = pageTable;
    a.B = batchSize;
    a.Hkv = numKVHeads;
    a.r = rotaryDim;
    a.numPages = numPages;
    a.mpps = maxPagesPerSeq;
    a.tpp = tokensPerPage;
    a.itemsPerRow = 2 * numKVHeads * (headDim / 16);
    return launch_paged_rows(a, numDeltaTokens, headDim, style, false, (cudaStream_t)stream);
}

int paged_kv_delta_update_fused(const uint16_t* kDelta, const uint16_t* vDelta,
                                uint16_t* kvCache, const float* cosSinSource,
                                const int32_t* oldDraftCacheLengths,
                                const int32_t* deltaLengths, int32_t deltaWidth,
                                const int32_t* stateIndices, const int32_t* pageTable,
                                int32_t batchSize, int32_t numKVHeads, int32_t headDim,
                                int32_t rotaryDim, int32_t numPages, int32_t maxPagesPerSeq,
                                int32_t tokensPerPage, int32_t sourceRows,
                                int32_t cacheCapacity, int32_t style, void* stream)
{
    if (deltaWidth < 0 || sourceRows < 0 || cacheCapacity < 0)
        return ROPEKV_ERR_SHAPE;
    const long long rows = (long long)batchSize * deltaWidth;
    if (rows > 0x7FFFFFFFLL)
        return ROPEKV_ERR_SHAPE;
    int rc = check_paged_sizes((int32_t)rows, batchSize, numKVHeads, headDim, rotaryDim,
                               numPages, maxPagesPerSeq, tokensPerPage, style);
    if (rc != ROPEKV_OK)
        return rc;
    if (rows == 0)
        return ROPEKV_OK;
    // as the gather: without source rows there is nothing to read, and every
    // rotated K dim is written as zero
    if (!kDelta || !vDelta || !kvCache || (!cosSinSource && sourceRows > 0) ||
        !oldDraftCacheLengths || !deltaLengths || !pageTable)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(kDelta) || !aligned16(vDelta) || !aligned16(kvCache) ||
        !aligned16(cosSinSource) || !aligned16(oldDraftCacheLengths) ||
        !aligned16(deltaLengths) || !aligned16(stateIndices) || !aligned16(pageTable))
        return ROPEKV_ERR_MISALIGNED;
    PagedArgs a = {};
    a.kDelta = kDelta;
    a.vDelta = vDelta;
    a.pool = kvCache;
    a.cosSin = cosSinSource;
    a.pageTable = pageTable;
    a.oldLens = oldDraftCacheLengths;
    a.deltaLens = deltaLengths;
    a.stateIdx = stateIndices;
    a.B = batchSize;
    a.Hkv = numKVHeads;
    a.r = rotaryDim;
    a.numPages = numPages;
    a.mpps = maxPagesPerSeq;
    a.tpp = tokensPerPage;
    a.deltaWidth = deltaWidth;
    a.widthShift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == deltaWidth)
            a.widthShift = sh;
    a.sourceRows = sourceRows;
    a.cacheCapacity = cacheCapacity;
    a.itemsPerRow = 2 * numKVHeads * (headDim / 16);
    return launch_paged_rows(a, rows, headDim, style, true, (cudaStream_t)stream);
}

int dflash_prepare_delta_metadata(const int32_t* oldDraftCacheLengths,
                                  const int32_t* deltaLengths, int32_t deltaWidth,
                                  int32_t* deltaPositions, int32_t* deltaTokenToSequence,
                                  int32_t batchSize, void* stream)
{
    if (deltaWidth < 0 || batchSize < 0)
        return ROPEKV_ERR_SHAPE;
    const long long rows = (long long)batchSize * deltaWidth;
    if (rows > 0x7FFFFFFFLL)
        return ROPEKV_ERR_SHAPE;
    if (rows == 0)
        return ROPEKV_OK;
    if (!oldDraftCacheLengths || !deltaLengths || !deltaPositions || !deltaTokenToSequence)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(oldDraftCacheLengths) || !aligned16(deltaLengths) ||
        !aligned16(deltaPositions) || !aligned16(deltaTokenToSequence))
        return ROPEKV_ERR_MISALIGNED;
    ropekv::DeltaMetaArgs a = {oldDraftCacheLengths, deltaLengths, deltaPositions,
                               deltaTokenToSequence, batchSize, deltaWidth};
    const unsigned grid = (unsigned)((rows + 255) / 256);
    return launch_k(ropekv::delta_metadata_kernel, grid, 256, (cudaStream_t)stream, false, a);
}

int dflash_gather_delta_rope(const float* source, float* output, const int32_t* deltaPositions,
                             const int32_t* deltaTokenToSequence, const int32_t* stateIndices,
                             int32_t numDeltaTokens, int32_t batchSize, int32_t sourceRows,
                             int32_t cacheCapacity, int32_t rotaryDim, void* stream)
{
    if (rotaryDim < 16 || rotaryDim > 256 || (rotaryDim % 16) != 0)
        return ROPEKV_ERR_ROTARY_DIM;
    if (numDeltaTokens < 0 || batchSize < 0 || sourceRows < 0 || cacheCapacity < 0)
        return ROPEKV_ERR_SHAPE;
    if (numDeltaTokens == 0)
        return ROPEKV_OK;
    if (!output || !deltaPositions || !deltaTokenToSequence || (!source && sourceRows > 0))
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(source) || !aligned16(output) || !aligned16(deltaPositions) ||
        !aligned16(deltaTokenToSequence) || !aligned16(stateIndices))
        return ROPEKV_ERR_MISALIGNED;
    ropekv::GatherArgs a = {source, output, deltaPositions, deltaTokenToSequence, stateIndices,
                            numDeltaTokens, batchSize, sourceRows, cacheCapacity, rotaryDim};
    const long long n = (long long)numDeltaTokens * (rotaryDim / 4);
    const unsigned grid = (unsigned)((n + 255) / 256);
    return launch_k(ropekv::gather_delta_rope_kernel, grid, 256, (cudaStream_t)stream, false, a);
}

int rope_write_kv_slot_mapping(const float* cosSin, const int64_t* positions, const uint16_t* q,
                               int64_t qTokenStride, const uint16_t* k, int64_t kTokenStride,
                               const uint16_t* v, int64_t vTokenStride,
                               const int64_t* slotMapping, uint16_t* keyCache,
                               uint16_t* valueCache, uint16_t* qOut, uint16_t* kOut,
                               int32_t numTokens, int32_t numQHeads, int32_t numKVHeads,
                               int32_t headDim, int32_t rotaryDim, int32_t cosSinRows,
                               int64_t numBlocks, int32_t blockSize, int32_t style, void* stream)
{
    if (style != ROPEKV_NEOX && style != ROPEKV_GPTJ)
        return ROPEKV_ERR_STYLE;
    int rc = check_head_dims(headDim, rotaryDim);
    if (rc != ROPEKV_OK)
        return rc;
    if (numQHeads <= 0 || numKVHeads <= 0 || numQHeads % numKVHeads != 0)
        return ROPEKV_ERR_HEADS;
    if (numTokens < 0 || cosSinRows < 0 || numBlocks < 0 || blockSize <= 0 ||
        numBlocks > (1LL << 40) || numBlocks > INT64_MAX / blockSize)
        return ROPEKV_ERR_SHAPE;
    if (qTokenStride < (int64_t)numQHeads * headDim || kTokenStride < (int64_t)numKVHeads * headDim ||
        vTokenStride < (int64_t)numKVHeads * headDim || (qTokenStride % 8) != 0 ||
        (kTokenStride % 8) != 0 || (vTokenStride % 8) != 0)
        return ROPEKV_ERR_SHAPE;
    const long long items = ((long long)numQHeads + 2LL * numKVHeads) * (headDim / 16);
    if (items > (1LL << 30))
        return ROPEKV_ERR_SHAPE;
    if (numTokens == 0)
        return ROPEKV_OK;
    if (!cosSin || !positions || !q || !k || !v || !slotMapping || !keyCache || !valueCache ||
        !qOut)
        return ROPEKV_ERR_NULL_POINTER;
    if (!aligned16(cosSin) || !aligned16(positions) || !aligned16(q) || !aligned16(k) ||
        !aligned16(v) || !aligned16(slotMapping) || !aligned16(keyCache) ||
        !aligned16(valueCache) || !aligned16(qOut) || !aligned16(kOut))
        return ROPEKV_ERR_MISALIGNED;
    ropekv::SlotMapArgs a = {};
    a.cosSin = cosSin;
    a.positions = positions;
    a.q = q;
    a.k = k;
    a.v = v;
    a.slots = slotMapping;
    a.keyCache = keyCache;
    a.valueCache = valueCache;
    a.qOut = qOut;
    a.kOut = kOut;
    a.qStride = qTokenStride;
    a.kStride = kTokenStride;
    a.vStride = vTokenStride;
    a.numSlots = numBlocks * (int64_t)blockSize;
    a.Hq = numQHeads;
    a.Hkv = numKVHeads;
    a.r = rotaryDim;
    a.csRows = cosSinRows;
    a.itemsPerToken = (int32_t)items;
    const Shape sh = pick_shape(a.itemsPerToken, numTokens);
    if ((long long)numTokens * sh.ctasPerUnit > 0x7FFFFFFFLL)
        return ROPEKV_ERR_SHAPE;
    a.ctasPerToken = sh.ctasPerUnit;
    const unsigned grid = (unsigned)((long long)numTokens * sh.ctasPerUnit);
    cudaStream_t st = (cudaStream_t)stream;
    const bool gptj = style == ROPEKV_GPTJ;
    switch (headDim) {
    case 64: return launch_slotmap<64>(a, gptj, grid, sh, st);
    case 128: return launch_slotmap<128>(a, gptj, grid, sh, st);
    default: return launch_slotmap<256>(a, gptj, grid, sh, st);
    }
}

int ropekv_set_residency_cap(int enable)
{
    return g_residency_cap.exchange(enable ? 1 : 0, std::memory_order_relaxed);
}

int rope_check_capacity(int32_t cosSinSeqLen, int32_t kvCapacity)
{
    return cosSinSeqLen > kvCapacity ? ROPEKV_ERR_CAPACITY : ROPEKV_OK;
}

const char* ropekv_status_string(int status)
{
    switch (status) {
    case ROPEKV_OK: return "ok";
    case ROPEKV_ERR_NULL_POINTER: return "a required pointer is NULL";
    case ROPEKV_ERR_MISALIGNED: return "a tensor pointer is not 16-byte aligned";
    case ROPEKV_ERR_HEAD_DIM: return "headDim must be 64, 128 or 256";
    case ROPEKV_ERR_ROTARY_DIM: return "rotaryDim must be a multiple of 16 in [16, headDim]";
    case ROPEKV_ERR_HEADS: return "head counts must be positive, numQHeads a multiple of numKVHeads";
    case ROPEKV_ERR_SHAPE: return "a size is negative or too large";
    case ROPEKV_ERR_COS_SIN_BATCH: return "cosSinBatch must be 1 or batch";
    case ROPEKV_ERR_CAPACITY: return "capacity check failed";
    case ROPEKV_ERR_STYLE: return "style must be ROPEKV_NEOX or ROPEKV_GPTJ";
    case ROPEKV_ERR_LAUNCH: return "CUDA kernel launch failed";
    default: return "unknown status";
    }
}

}  // extern "C"
