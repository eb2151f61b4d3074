/*
 * ropekv_oracle.h -- CPU oracle for the fused RoPE + KV-cache write.
 *
 * TEST INFRASTRUCTURE. This is the plain, slow, double-precision statement of
 * what the fused RoPE + KV-cache write computes. Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it. The library's
 * product path never calls it, and the two share no code, header, table or
 * helper.
 *
 * Sources, cited by page title and section:
 *   [ARW] TensorRT-Edge-LLM 0.4.0 C++ API, "Apply Rope Write KV":
 *         launchApplyRopeWriteKVPackedQKV, launchApplyRopeWriteKVContinuousQAndKVCache,
 *         launchApplyRopeWriteKVTreeDecoding (parameter lists: layouts, in/out roles).
 *   [RC]  sglang python/sglang/kernels/ops/kvcache/rope_cache.py:
 *         _get_neox_rotated_x, _get_gptj_rotated_x, _unit_rope, _load_cos_sin,
 *         kernel Stage 2.1 (frequency index) and the wrapper's cos_sin width rule.
 *   [RC]  (also) fused_qk_rope_reshape_and_cache, flash layout: separate Q/K/V,
 *         a flat slot mapping, the KV write skipped for negative slots.
 *   [DRK] TensorRT-Edge-LLM C++ API, "Dflash Runtime Kernels":
 *         launchDFlashTargetKVCacheUpdate, checkDFlashRopeCapacity,
 *         launchDFlashPrepareDeltaMetadata, launchDFlashGatherDeltaRope,
 *         launchDFlashPrepareProposalInputs (target length after the delta).
 *
 * Conventions shared by every function below:
 *   - FP16 tensors are passed as uint16_t arrays of IEEE 754 binary16 bits.
 *   - cos/sin rows hold r = rotaryDim FP32 values: cos_0..cos_{r/2-1} then
 *     sin_0..sin_{r/2-1} ([RC] _load_cos_sin reads sin at the cos index plus
 *     the frequency count; the wrapper's half-width rule fixes that count at r/2).
 *   - style 0 = GPT-NeoX half split, style 1 = GPT-J interleaved pairs.
 *   - All buffers are host memory owned by the caller. Functions return 0 on
 *     success and -1 when the sizes are inconsistent (nothing is written then).
 *
 * Parity status: every function here is pinned by tests under tests/ (worked
 * examples, closed forms, invariants and brute-force placement tables).
 */
#ifndef ROPEKV_ORACLE_H
#define ROPEKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE 754 binary16 bits -> double (exact). */
double ropekv_oracle_f16_to_f64(uint16_t bits);

/* double -> IEEE 754 binary16 bits, round to nearest, ties to even;
 * overflow goes to infinity, NaN stays NaN. */
uint16_t ropekv_oracle_f64_to_f16(double x);

/* rotate(x) of [RC] _get_neox_rotated_x / _get_gptj_rotated_x over the first
 * r dims of one head: NeoX [x0,x1,x2,x3] -> [-x2,-x3,x0,x1],
 * GPT-J [x0,x1,x2,x3] -> [-x1,x0,-x3,x2]. Writes out[0..r). */
void ropekv_oracle_rotate_half(const double* x, int r, int style, double* out);

/* Frequency index of dim d (< r), [RC] kernel Stage 2.1 with the half-width
 * table: NeoX d mod (r/2), GPT-J d / 2. */
int ropekv_oracle_freq_index(int d, int r, int style);

/* [RC] _unit_rope on one head, in double: y[d] = x[d]*cos[f(d)] + rotate(x)[d]*sin[f(d)]
 * for d < r; y[d] = x[d] for r <= d < D. cs_row is the r-float table row. */
void ropekv_oracle_rope_head_f64(const double* x, const float* cs_row, int D, int r,
                                 int style, double* y);

/* [ARW] launchApplyRopeWriteKVPackedQKV. Empty cache: position = cache slot = s.
 * qkv [B,S,Hq+2Hkv,D] is rotated in place (Q and K heads; V heads untouched),
 * kvCache [B,2,Hkv,cap,D] receives rotated K (plane 0) and V bits (plane 1) at
 * slots 0..S-1. cosSin [csBatch,csSeq,r]; csBatch is 1 (shared) or B. */
int ropekv_oracle_packed(const float* cosSin, uint16_t* qkv, uint16_t* kvCache,
                         int B, int S, int Hq, int Hkv, int D, int r, int cap,
                         int csBatch, int csSeq, int style);

/* [ARW] launchApplyRopeWriteKVContinuousQAndKVCache. slot = pos =
 * kvCacheEndLens[b] - S + s. qkv is read only; rotated Q goes to qOut
 * [B,S,Hq,D]; rotated K and V bits go to the cache at slot. A token whose slot
 * is negative, >= cap or >= csSeq writes nothing. */
int ropekv_oracle_continuous(const float* cosSin, const int32_t* kvCacheEndLens,
                             const uint16_t* qkv, uint16_t* kvCache, uint16_t* qOut,
                             int B, int S, int Hq, int Hkv, int D, int r, int cap,
                             int csBatch, int csSeq, int style);

/* [ARW] launchApplyRopeWriteKVTreeDecoding. RoPE position = tokenPosIds[b,s];
 * cache slot = kvCacheEndLens[b] - S + s (linear order). A token with a
 * negative or >= csSeq position, or a slot outside [0,cap), writes nothing. */
int ropekv_oracle_tree(const float* cosSin, const int32_t* kvCacheEndLens,
                       const int32_t* tokenPosIds, const uint16_t* qkv,
                       uint16_t* kvCache, uint16_t* qOut,
                       int B, int S, int Hq, int Hkv, int D, int r, int cap,
                       int csBatch, int csSeq, int style);

/* [DRK] launchDFlashTargetKVCacheUpdate, per delta row, without a pool.
 * For row t: kDest[t] / vDest[t] receive the element offset, inside a pool laid
 * out [2, numPages, tokensPerPage, Hkv, D], of the row's [Hkv, D] block in the
 * K / V plane, or -1 when that plane is skipped. kOut / vOut [numDeltaTokens,Hkv,D]
 * receive the values written there (rotated K with cos/sin row t; V bits);
 * rows whose plane is skipped are left as they were. */
int ropekv_oracle_paged_rows(const uint16_t* kDelta, const uint16_t* vDelta,
                             const float* tokenAlignedCosSin,
                             const int32_t* deltaPositions, const int32_t* deltaTokenToSequence,
                             const int32_t* pageTable,
                             int numDeltaTokens, int batchSize, int Hkv, int D, int r,
                             int numPages, int maxPagesPerSeq, int tokensPerPage, int style,
                             int64_t* kDest, int64_t* vDest, uint16_t* kOut, uint16_t* vOut);

/* [DRK] launchDFlashTargetKVCacheUpdate into a host pool
 * kvCache [2, numPages, tokensPerPage, Hkv, D]: the rows above, stored at their
 * destinations. */
int ropekv_oracle_paged(const uint16_t* kDelta, const uint16_t* vDelta, uint16_t* kvCache,
                        const float* tokenAlignedCosSin,
                        const int32_t* deltaPositions, const int32_t* deltaTokenToSequence,
                        const int32_t* pageTable,
                        int numDeltaTokens, int batchSize, int Hkv, int D, int r,
                        int numPages, int maxPagesPerSeq, int tokensPerPage, int style);

/* [DRK] launchDFlashPrepareDeltaMetadata (the page gives the signature only).
 * Reading: delta rows are laid out [batchSize, deltaWidth]; row b*deltaWidth + j
 * is sequence b's j-th new token when j < deltaLengths[b] (a negative length
 * counts as 0): position oldDraftCacheLengths[b] + j (the draft cache
 * length before the delta, plus the offset inside the delta), sequence b.
 * Every other row is padding: position -1, sequence -1. Writes
 * batchSize*deltaWidth entries of each output. */
int ropekv_oracle_delta_metadata(const int32_t* oldDraftCacheLengths, const int32_t* deltaLengths,
                                 int deltaWidth, int32_t* deltaPositions,
                                 int32_t* deltaTokenToSequence, int batchSize);

/* [DRK] launchDFlashGatherDeltaRope (the page gives the signature only).
 * Reading: source is a FP32 cos/sin cache [sourceRows, cacheCapacity, rotaryDim];
 * output [numDeltaTokens, rotaryDim] is the token-aligned table of the paged
 * update. Row t takes pos = deltaPositions[t], seq = deltaTokenToSequence[t] and
 * the source row state = stateIndices[seq] (or, without stateIndices, 0 when
 * sourceRows == 1, else seq); it copies source[state, pos, :] and is zero when
 * pos < 0, seq < 0, seq >= batchSize, pos >= cacheCapacity or state is outside
 * [0, sourceRows). stateIndices may be NULL. */
int ropekv_oracle_gather_delta_rope(const float* source, float* output,
                                    const int32_t* deltaPositions,
                                    const int32_t* deltaTokenToSequence,
                                    const int32_t* stateIndices, int numDeltaTokens,
                                    int batchSize, int sourceRows, int cacheCapacity,
                                    int rotaryDim);

/* The DFlash target-KV step as one call: delta metadata, the cos/sin gather and
 * the paged update above, in that order, on batchSize*deltaWidth delta rows.
 * Defined as exactly that composition (scratch arrays are the oracle's own). */
int ropekv_oracle_paged_fused(const uint16_t* kDelta, const uint16_t* vDelta, uint16_t* kvCache,
                              const float* source, const int32_t* oldDraftCacheLengths,
                              const int32_t* deltaLengths, int deltaWidth,
                              const int32_t* stateIndices, const int32_t* pageTable,
                              int batchSize, int Hkv, int D, int r, int numPages,
                              int maxPagesPerSeq, int tokensPerPage, int sourceRows,
                              int cacheCapacity, int style);

/* Pre-RoPE QK RMS normalization fused into the continuous call (libmir-cuda
 * execution.rs: qkv_postprocess normalizes Q and K with query_norm / key_norm
 * weights and epsilon, then applies RoPE, then the KV store; "Dflash Runtime
 * Kernels": its kDelta is K already normalized, not yet rotated). Reading:
 * each Q head x [D] becomes
 *   x_hat[d] = x[d] / sqrt(mean_{d'} x[d']^2 + eps) * qNormWeight[d]
 * (K heads with kNormWeight), then RoPE on x_hat, rounded to FP16 once; V is
 * copied as bits. Weights are FP16 [D]. Placement and skips: as the continuous
 * call. Dims >= r of Q and K are normalized (no longer bit copies). */
int ropekv_oracle_continuous_qknorm(const float* cosSin, const int32_t* kvCacheEndLens,
                                    const uint16_t* qkv, uint16_t* kvCache, uint16_t* qOut,
                                    const uint16_t* qNormWeight, const uint16_t* kNormWeight,
                                    float eps, int B, int S, int Hq, int Hkv, int D, int r,
                                    int cap, int csBatch, int csSeq, int style);

/* RMS normalization of one head in double (the first step above). */
void ropekv_oracle_rms_norm_f64(const double* x, const uint16_t* weight, double eps, int D,
                                double* y);

/* OCP FP8 E4M3 ("e4m3fn": 4 exponent bits, bias 7, 3 fraction bits, no
 * infinities, 0x7F / 0xFF NaN, largest finite 448) bits -> double (exact). */
double ropekv_oracle_e4m3_to_f64(uint8_t bits);

/* double -> E4M3 bits: round to nearest, ties to even; magnitudes above 448
 * (and infinities) saturate to +-448; NaN -> 0x7F. */
uint8_t ropekv_oracle_f64_to_e4m3(double x);

/* The continuous call with an FP8 cache ([RC] kernel Stage 3.3: K and V are
 * multiplied by 1/k_scale and 1/v_scale before the cache store, which converts
 * them to the cache's FP8 type). kvCache8 [B, 2, Hkv, cap, D] holds E4M3 bytes:
 * plane 0 = e4m3(rope(K) / kScale), plane 1 = e4m3(V / vScale); rotated Q goes
 * to qOut in FP16 as in the continuous call. */
int ropekv_oracle_continuous_fp8(const float* cosSin, const int32_t* kvCacheEndLens,
                                 const uint16_t* qkv, uint8_t* kvCache8, uint16_t* qOut,
                                 float kScale, float vScale, int B, int S, int Hq, int Hkv, int D,
                                 int r, int cap, int csBatch, int csSeq, int style);

/* [RC] fused_qk_rope_reshape_and_cache with the flash cache layout.
 * Token t (of T) has RoPE position positions[t] (row of cosSin [cosSinRows, r])
 * and flat cache slot slotMapping[t]. Q [T, Hq, D], K and V [T, Hkv, D] are read
 * with token strides qStride / kStride / vStride (elements). Rotated Q goes to
 * qOut [T, Hq, D]. When 0 <= slot < numBlocks*blockSize, rotated K goes to
 * keyCache[slot / blockSize, slot % blockSize] and to kOut [T, Hkv, D] (kOut
 * may be NULL), and V's bits go to valueCache at the same place; both caches
 * are [numBlocks, blockSize, Hkv, D]. A negative slot (or one past the caches)
 * skips those writes only. A position outside [0, cosSinRows) skips the token. */
int ropekv_oracle_slot_mapping(const float* cosSin, const int64_t* positions,
                               const uint16_t* q, int64_t qStride, const uint16_t* k,
                               int64_t kStride, const uint16_t* v, int64_t vStride,
                               const int64_t* slotMapping, uint16_t* keyCache,
                               uint16_t* valueCache, uint16_t* qOut, uint16_t* kOut, int T,
                               int Hq, int Hkv, int D, int r, int cosSinRows, int64_t numBlocks,
                               int blockSize, int style);

/* [DRK] checkDFlashRopeCapacity: 1 when the pair is rejected
 * (cosSinSeqLen > kvCapacity), else 0. */
int ropekv_oracle_capacity_rejected(int32_t cosSinSeqLen, int32_t kvCapacity);

#ifdef __cplusplus
}
#endif

#endif /* ROPEKV_ORACLE_H */
