/*
 * ropekv.h -- C ABI of the fused RoPE + KV-cache write library (libropekv.so).
 *
 * One call = one CUDA kernel launch on the caller's stream that, for every
 * token and head, reads the packed FP16 QKV row (or the K/V delta rows) and the
 * FP32 cos/sin row of the token's position, rotates the first rotaryDim dims
 * of Q and K, x' = x*cos + rotate(x)*sin, and writes rotated Q, rotated K and
 * unchanged V. Sources (web pages, cited by title and section):
 *
 *   [ARW] TensorRT-Edge-LLM 0.4.0 C++ API, "Apply Rope Write KV"
 *         (launchApplyRopeWriteKVPackedQKV, launchApplyRopeWriteKVContinuousQAndKVCache,
 *         launchApplyRopeWriteKVTreeDecoding).
 *   [DRK] TensorRT-Edge-LLM C++ API, "Dflash Runtime Kernels"
 *         (launchDFlashTargetKVCacheUpdate, checkDFlashRopeCapacity,
 *         launchDFlashPrepareDeltaMetadata, launchDFlashGatherDeltaRope).
 *   [MIR] libmir-cuda 0.1.0 backend/attention/graph/execution.rs (qkv_postprocess:
 *         QK normalization before RoPE, then the KV store).
 *   [RC]  sglang rope_cache.py (_get_neox_rotated_x, _get_gptj_rotated_x,
 *         _unit_rope, _load_cos_sin, kernel Stage 2.1; the
 *         fused_qk_rope_reshape_and_cache interface, Stages 3.1-3.5).
 *
 * Common rules for every entry point:
 *   - FP16 tensors are uint16_t arrays holding IEEE binary16 bits; FP32 tables
 *     are float; indices are int32_t. All tensors are dense, row-major, in the
 *     layouts stated per call.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller and must be
 *     16-byte aligned. The library allocates nothing and never synchronises;
 *     results are ready when the stream says so. Its only state is a record,
 *     per kernel and device, that the kernel's dynamic shared memory limit was
 *     raised, and the residency-cap switch (ropekv_set_residency_cap):
 *     decode-sized launches (fewer than 1024 tokens) reserve shared memory
 *     they do not use so that their CTAs spread over all SMs.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls are asynchronous and may be captured in a CUDA graph.
 *     The calling thread's current CUDA device must be the device that holds
 *     the tensors and the stream (as for any kernel launch): the launch and
 *     the residency cap use the current device.
 *   - cos/sin rows hold rotaryDim floats: cos_0..cos_{r/2-1} then
 *     sin_0..sin_{r/2-1} ([RC] _load_cos_sin and the half-width table rule).
 *     Dims i and partner use frequency i: NeoX pairs (i, i + r/2), GPT-J pairs
 *     (2i, 2i + 1) ([RC] rotate layouts and Stage 2.1). Dims >= rotaryDim and
 *     all V heads are copied bit for bit.
 *   - Return value: ROPEKV_OK (0), or a negative ropekv_status when the host
 *     rejected the arguments (nothing launched) or the launch failed. A
 *     launch failure is read from that launch's own result
 *     (cudaLaunchKernelEx); the library never calls cudaGetLastError or
 *     cudaPeekAtLastError, so it neither reports nor clears an error that the
 *     caller left pending. (An error that earlier work left in the context can
 *     still make the launch itself fail.)
 *     Data-dependent invalid indices found on the device (negative or
 *     out-of-range positions, sequences, slots or pages) are skipped: nothing
 *     is written for them, and no error is raised ([DRK] skip rules).
 *   - Supported shapes: headDim in {64, 128, 256}; rotaryDim a multiple of 16
 *     with 16 <= rotaryDim <= headDim; numQHeads a multiple of numKVHeads.
 *     Element counts of every tensor must fit in int64.
 *   - Two tokens that resolve to the same cache slot race (last writer wins
 *     in no fixed order); the pages' producers never generate them.
 */
#ifndef ROPEKV_H
#define ROPEKV_H

#include <stdint.h>

#if defined(__GNUC__)
#define ROPEKV_API __attribute__((visibility("default")))
#else
#define ROPEKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Pairing of rotated dims: GPT-NeoX half split or GPT-J interleaved pairs. */
typedef enum { ROPEKV_NEOX = 0, ROPEKV_GPTJ = 1 } ropekv_style;

typedef enum {
    ROPEKV_OK = 0,
    ROPEKV_ERR_NULL_POINTER = -1,    /* a required pointer is NULL              */
    ROPEKV_ERR_MISALIGNED = -2,      /* a tensor pointer is not 16-byte aligned */
    ROPEKV_ERR_HEAD_DIM = -3,        /* headDim not in {64, 128, 256}           */
    ROPEKV_ERR_ROTARY_DIM = -4,      /* rotaryDim not a multiple of 16 in [16, headDim] */
    ROPEKV_ERR_HEADS = -5,           /* numQHeads/numKVHeads <= 0 or not divisible */
    ROPEKV_ERR_SHAPE = -6,           /* negative size, or a size too large       */
    ROPEKV_ERR_COS_SIN_BATCH = -7,   /* cosSinBatch neither 1 nor batch          */
    ROPEKV_ERR_CAPACITY = -8,        /* capacity check failed (see each call)    */
    ROPEKV_ERR_STYLE = -9,           /* style not a ropekv_style                 */
    ROPEKV_ERR_LAUNCH = -10          /* the CUDA launch reported an error        */
} ropekv_status;

/* Sizes of the contiguous-cache entry points ([ARW]). */
typedef struct {
    int32_t batch;        /* B: sequences                                        */
    int32_t seqLen;       /* S: runtime tokens per sequence                      */
    int32_t numQHeads;    /* Hq                                                  */
    int32_t numKVHeads;   /* Hkv (= Hk = Hv)                                     */
    int32_t headDim;      /* D                                                   */
    int32_t rotaryDim;    /* r: leading dims of each Q/K head that are rotated   */
    int32_t kvCapacity;   /* slots per sequence in the cache                     */
    int32_t cosSinBatch;  /* 1 (one table for all sequences) or B (one per seq)  */
    int32_t cosSinSeqLen; /* rows (positions) per table                          */
    int32_t style;        /* a ropekv_style                                      */
} ropekv_dims;

/*
 * [ARW] launchApplyRopeWriteKVPackedQKV: the cache is empty.
 *   cosSin  [cosSinBatch, cosSinSeqLen, rotaryDim] FP32, read.
 *   qkv     [B, S, Hq + 2*Hkv, headDim] FP16, heads ordered Q, K, V; read and
 *           written IN PLACE: Q and K heads are rotated, V heads are left as is.
 *   kvCache [B, 2, Hkv, kvCapacity, headDim] FP16, written: plane 0 = rotated K,
 *           plane 1 = V, at slots 0..S-1 (an empty cache fills from slot 0); token s
 *           uses cos/sin row s. Slots >= S are not touched.
 * Host errors: S > kvCapacity or S > cosSinSeqLen -> ROPEKV_ERR_CAPACITY.
 */
ROPEKV_API int rope_write_kv_packed(const float* cosSin, uint16_t* qkv, uint16_t* kvCache,
                                    const ropekv_dims* dims, void* stream);

/*
 * [ARW] launchApplyRopeWriteKVContinuousQAndKVCache: the cache already holds
 * tokens. kvCacheEndLens[b] is where sequence b ends once this call's tokens
 * are written, so token s of
 * sequence b takes slot = position = kvCacheEndLens[b] - S + s.
 *   cosSin         [cosSinBatch, cosSinSeqLen, rotaryDim] FP32, read.
 *   kvCacheEndLens [B] INT32, read on the device.
 *   qkv            [B, S, Hq + 2*Hkv, headDim] FP16, read only.
 *   kvCache        [B, 2, Hkv, kvCapacity, headDim] FP16, written at the slots.
 *   qOut           [B, S, Hq, headDim] FP16, written (rotated Q).
 * A token whose slot is < 0, >= kvCapacity or >= cosSinSeqLen writes nothing
 * (neither its qOut row nor its cache slots).
 */
ROPEKV_API int rope_write_kv_continuous(const float* cosSin, const int32_t* kvCacheEndLens,
                                        const uint16_t* qkv, uint16_t* kvCache,
                                        uint16_t* qOut, const ropekv_dims* dims,
                                        void* stream);

/*
 * rope_write_kv_continuous with pre-RoPE RMS normalization of Q and K fused in
 * (libmir-cuda execution.rs: qkv_postprocess normalizes Q and K with
 * query_norm / key_norm weights and an epsilon before RoPE, then the KV store
 * runs; "Dflash Runtime Kernels" takes its K input already normalized).
 * Every Q head x becomes x[d] / sqrt(mean_d' x[d']^2 + eps) * qNormWeight[d]
 * (K heads with kNormWeight), in FP32, before the rotation; the result is
 * rounded to FP16 once. V is copied as bits. Dims >= rotaryDim of Q and K are normalized too.
 *   qNormWeight, kNormWeight  [headDim] FP16, read.
 *   eps                       >= 0.
 * Everything else as rope_write_kv_continuous.
 */
ROPEKV_API int rope_write_kv_continuous_qknorm(const float* cosSin,
                                               const int32_t* kvCacheEndLens,
                                               const uint16_t* qkv, uint16_t* kvCache,
                                               uint16_t* qOut, const uint16_t* qNormWeight,
                                               const uint16_t* kNormWeight, float eps,
                                               const ropekv_dims* dims, void* stream);

/*
 * rope_write_kv_continuous with an FP8 cache ([RC] kernel Stage 3.3: rotated K
 * and V are multiplied by 1/k_scale and 1/v_scale and stored in the cache's FP8
 * type). Cache elements are OCP E4M3 ("e4m3fn") bytes: plane 0 =
 * e4m3(rotated K * (1 / *kScale)), plane 1 = e4m3(V * (1 / *vScale)), rounded to
 * nearest even from FP32 and saturated to +-448. Rotated Q goes to qOut in FP16.
 *   kvCache8        [B, 2, Hkv, kvCapacity, headDim] uint8 (E4M3), written at the slots.
 *   kScale, vScale  one FP32 each, device memory, read by the kernel (> 0).
 * Everything else as rope_write_kv_continuous.
 */
ROPEKV_API int rope_write_kv_continuous_fp8(const float* cosSin, const int32_t* kvCacheEndLens,
                                            const uint16_t* qkv, uint8_t* kvCache8,
                                            uint16_t* qOut, const float* kScale,
                                            const float* vScale, const ropekv_dims* dims,
                                            void* stream);

/*
 * [ARW] launchApplyRopeWriteKVTreeDecoding: tree attention for speculative
 * decoding. As the continuous call, except that the RoPE position of token
 * (b, s) is tokenPosIds[b, s], the token's position in its sequence; the cache
 * slot stays kvCacheEndLens[b] - S + s, so sibling nodes that share a position
 * keep distinct slots.
 *   tokenPosIds [B, S] INT32, read on the device.
 * A token whose position is < 0 or >= cosSinSeqLen, or whose slot is outside
 * [0, kvCapacity), writes nothing.
 */
ROPEKV_API int rope_write_kv_tree(const float* cosSin, const int32_t* kvCacheEndLens,
                                  const int32_t* tokenPosIds, const uint16_t* qkv,
                                  uint16_t* kvCache, uint16_t* qOut,
                                  const ropekv_dims* dims, void* stream);

/*
 * [DRK] launchDFlashTargetKVCacheUpdate: RoPE on token-major K delta rows, and
 * K/V delta rows written into their sequences' pages of a paged pool.
 *   kDelta, vDelta        [numDeltaTokens, numKVHeads, headDim] FP16, read
 *                         (K not yet rotated).
 *   kvCache               [2, numPages, tokensPerPage, numKVHeads, headDim] FP16,
 *                         written at the destinations below, untouched elsewhere.
 *   tokenAlignedCosSin    [numDeltaTokens, rotaryDim] FP32: row t serves delta row t.
 *   deltaPositions        [numDeltaTokens] INT32 absolute KV positions.
 *   deltaTokenToSequence  [numDeltaTokens] INT32 owning sequence.
 *   pageTable             [batchSize, 2, maxPagesPerSeq] INT32 canonical page ids:
 *                         plane 0 entries in [0, numPages) name K pages, plane 1
 *                         entries in [numPages, 2*numPages) name V pages; the id
 *                         is the flat page index of the [2, numPages] pool.
 * Row t with pos = deltaPositions[t], seq = deltaTokenToSequence[t] and logical
 * page lp = pos / tokensPerPage writes rotated K to flat page
 * pageTable[seq, 0, lp] and V to flat page pageTable[seq, 1, lp], both at
 * in-page slot pos % tokensPerPage. The row is skipped when pos < 0, seq < 0,
 * seq >= batchSize or lp >= maxPagesPerSeq; each plane is skipped on its own
 * when its id is unmapped (negative) or outside that plane's range.
 * tokensPerPage is a runtime argument here (a compile-time constant on the page).
 * Host errors: tokensPerPage <= 0, numPages or maxPagesPerSeq < 0.
 */
ROPEKV_API int paged_kv_delta_update(const uint16_t* kDelta, const uint16_t* vDelta,
                                     uint16_t* kvCache, const float* tokenAlignedCosSin,
                                     const int32_t* deltaPositions,
                                     const int32_t* deltaTokenToSequence,
                                     const int32_t* pageTable, int32_t numDeltaTokens,
                                     int32_t batchSize, int32_t numKVHeads, int32_t headDim,
                                     int32_t rotaryDim, int32_t numPages,
                                     int32_t maxPagesPerSeq, int32_t tokensPerPage,
                                     int32_t style, void* stream);

/*
 * [RC] fused_qk_rope_reshape_and_cache with the flash cache layout: the same
 * fused RoPE + KV write behind sglang's interface. Q, K and V are separate
 * token-major tensors that may be views into one packed QKV buffer; every token
 * carries its own RoPE position and one flat cache slot.
 *   cosSin       [cosSinRows, rotaryDim] FP32, row = position.
 *   positions    [numTokens] INT64 RoPE position of each token.
 *   q            [numTokens, numQHeads, headDim] FP16, token stride qTokenStride
 *                elements (>= numQHeads*headDim, a multiple of 8); k, v likewise
 *                with numKVHeads heads and their own strides. Read only.
 *   slotMapping  [numTokens] INT64 flat slot: block slot / blockSize, offset
 *                slot % blockSize.
 *   keyCache, valueCache  [numBlocks, blockSize, numKVHeads, headDim] FP16, written
 *                at the slots (rotated K; V bits).
 *   qOut         [numTokens, numQHeads, headDim] FP16, rotated Q, written.
 *   kOut         [numTokens, numKVHeads, headDim] FP16 rotated K, or NULL.
 * A negative slot, or one >= numBlocks*blockSize, skips the cache writes and
 * kOut for that token (its qOut row is still written). A position outside
 * [0, cosSinRows) skips the whole token.
 * Host errors: strides too small or not multiples of 8 -> ROPEKV_ERR_SHAPE.
 */
ROPEKV_API int rope_write_kv_slot_mapping(const float* cosSin, const int64_t* positions,
                                          const uint16_t* q, int64_t qTokenStride,
                                          const uint16_t* k, int64_t kTokenStride,
                                          const uint16_t* v, int64_t vTokenStride,
                                          const int64_t* slotMapping, uint16_t* keyCache,
                                          uint16_t* valueCache, uint16_t* qOut, uint16_t* kOut,
                                          int32_t numTokens, int32_t numQHeads,
                                          int32_t numKVHeads, int32_t headDim,
                                          int32_t rotaryDim, int32_t cosSinRows,
                                          int64_t numBlocks, int32_t blockSize, int32_t style,
                                          void* stream);

/*
 * The DFlash target-KV step as ONE launch: launchDFlashPrepareDeltaMetadata,
 * launchDFlashGatherDeltaRope and launchDFlashTargetKVCacheUpdate of [DRK]
 * folded together, so the per-row positions, sequences and cos/sin rows never
 * go through memory. The result is exactly that of calling
 * dflash_prepare_delta_metadata, dflash_gather_delta_rope and
 * paged_kv_delta_update in that order on the same arguments.
 *   kDelta, vDelta         [batchSize * deltaWidth, numKVHeads, headDim] FP16: row
 *                          b * deltaWidth + j is sequence b's delta token j.
 *   kvCache, pageTable     as paged_kv_delta_update.
 *   cosSinSource           [sourceRows, cacheCapacity, rotaryDim] FP32 cos/sin cache.
 *   oldDraftCacheLengths   [batchSize] INT32, draft cache lengths before the delta.
 *   deltaLengths           [batchSize] INT32, delta tokens of each sequence; rows
 *                          j >= deltaLengths[b] are padding.
 *   stateIndices           [batchSize] INT32 source row of each sequence, or NULL
 *                          (then row 0 when sourceRows == 1, else row b).
 *   cosSinSource may be NULL when sourceRows == 0 (as for the gather): every
 *   row's cos/sin is then zero.
 * Token j of sequence b sits at position oldDraftCacheLengths[b] + j. When its
 * position is >= cacheCapacity or its source row is outside [0, sourceRows) the
 * gather yields a zero cos/sin row, so rotated K dims are written as zeros.
 * Host errors: as paged_kv_delta_update; deltaWidth, sourceRows or
 * cacheCapacity negative, or batchSize * deltaWidth >= 2^31 -> ROPEKV_ERR_SHAPE.
 */
ROPEKV_API int paged_kv_delta_update_fused(const uint16_t* kDelta, const uint16_t* vDelta,
                                           uint16_t* kvCache, const float* cosSinSource,
                                           const int32_t* oldDraftCacheLengths,
                                           const int32_t* deltaLengths, int32_t deltaWidth,
                                           const int32_t* stateIndices, const int32_t* pageTable,
                                           int32_t batchSize, int32_t numKVHeads,
                                           int32_t headDim, int32_t rotaryDim, int32_t numPages,
                                           int32_t maxPagesPerSeq, int32_t tokensPerPage,
                                           int32_t sourceRows, int32_t cacheCapacity,
                                           int32_t style, void* stream);

/*
 * [DRK] launchDFlashPrepareDeltaMetadata (the page prints only the signature).
 * Reading used here: delta rows are laid out [batchSize, deltaWidth]; row
 * t = b * deltaWidth + j gets deltaPositions[t] = oldDraftCacheLengths[b] + j and
 * deltaTokenToSequence[t] = b when j < deltaLengths[b], else -1 and -1 (padding).
 * (The target length after the delta is oldDraftCacheLengths[b] + deltaLength,
 * as [DRK] launchDFlashPrepareProposalInputs states.)
 *   oldDraftCacheLengths, deltaLengths  [batchSize] INT32, read.
 *   deltaPositions, deltaTokenToSequence [batchSize * deltaWidth] INT32, written.
 * Host errors: negative sizes or batchSize * deltaWidth >= 2^31 -> ROPEKV_ERR_SHAPE.
 */
ROPEKV_API int dflash_prepare_delta_metadata(const int32_t* oldDraftCacheLengths,
                                             const int32_t* deltaLengths, int32_t deltaWidth,
                                             int32_t* deltaPositions,
                                             int32_t* deltaTokenToSequence, int32_t batchSize,
                                             void* stream);

/*
 * [DRK] launchDFlashGatherDeltaRope (the page prints only the signature).
 * Reading used here: output row t is the tokenAlignedCosSin row of delta row t,
 *   output[t, :] = source[state, deltaPositions[t], :],
 * with state = stateIndices[seq] (stateIndices may be NULL: then 0 when
 * sourceRows == 1, else seq) and seq = deltaTokenToSequence[t]; the row is zero
 * when the position is negative or >= cacheCapacity, seq is negative or
 * >= batchSize, or state is outside [0, sourceRows).
 *   source  [sourceRows, cacheCapacity, rotaryDim] FP32, read.
 *   output  [numDeltaTokens, rotaryDim] FP32, written (every row).
 * Host errors: rotaryDim not a multiple of 16 in [16, 256] -> ROPEKV_ERR_ROTARY_DIM;
 * negative sizes -> ROPEKV_ERR_SHAPE.
 */
ROPEKV_API int dflash_gather_delta_rope(const float* source, float* output,
                                        const int32_t* deltaPositions,
                                        const int32_t* deltaTokenToSequence,
                                        const int32_t* stateIndices, int32_t numDeltaTokens,
                                        int32_t batchSize, int32_t sourceRows,
                                        int32_t cacheCapacity, int32_t rotaryDim, void* stream);

/*
 * [DRK] checkDFlashRopeCapacity: the RoPE table must cover every position the
 * paged update can write. kvCapacity is the page-aligned per-sequence capacity
 * (maxPagesPerSeq * tokensPerPage); the table may be shorter than it, so only
 * cosSinSeqLen > kvCapacity is rejected. Host only; returns ROPEKV_OK or
 * ROPEKV_ERR_CAPACITY (the page's version throws instead).
 */
ROPEKV_API int rope_check_capacity(int32_t cosSinSeqLen, int32_t kvCapacity);

/*
 * Process-wide switch of the residency cap of decode-sized launches (fewer
 * than 1024 tokens or rows): 1 (the default) = on, 0 = off. Returns the
 * previous setting. Thread-safe; takes effect for launches made after it.
 *
 * With the cap on, a decode-sized launch reserves dynamic shared memory that
 * its kernel does not use, sized so that at most ceil(grid / SMs) of its CTAs
 * fit on one SM. A launch that starts while its predecessor in the stream
 * still runs (programmatic dependent launch) otherwise has its CTAs packed
 * onto a minority of the SMs, and it lasts as long as the busiest SM (on
 * GB300, 256 decode tokens: 2.40 us uncapped, about 2.1 us capped). The cost
 * falls on concurrent work: while a kernel on another stream holds shared
 * memory on an SM, a capped CTA may not fit there and waits for another SM,
 * and the capped CTAs in turn keep other kernels' shared-memory-hungry CTAs
 * off the SMs they occupy. A caller that overlaps these writes with
 * shared-memory-heavy kernels (attention, GEMMs) can switch the cap off.
 * Results are identical either way. (Not in the pages: a launch-shape choice.)
 */
ROPEKV_API int ropekv_set_residency_cap(int enable);

/* Static, human-readable text for a status code (never NULL). */
ROPEKV_API const char* ropekv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ROPEKV_H */
