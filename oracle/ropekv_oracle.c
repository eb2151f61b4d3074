/*
 * ropekv_oracle.c -- CPU oracle for the fused RoPE + KV-cache write.
 *
 * TEST INFRASTRUCTURE: the plain, slow, double-precision definition that the
 * CUDA path is checked against. Only tests, the smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code with the CUDA path.
 * Sources and conventions are listed in ropekv_oracle.h.
 *
 * Everything is written the plain way: one loop per index of the definition,
 * each element converted FP16 -> double, rotated in double, and rounded back
 * to FP16 with round-to-nearest-even. Bits that the method copies (dims past
 * rotaryDim, V heads) are copied as bits, never through a float.
 */
#include "ropekv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { STYLE_NEOX = 0, STYLE_GPTJ = 1 };

/* ---------------------------------------------------------------- FP16 ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = fraction * 2^-24; exponent 31: inf / NaN;
 * otherwise value = (1024 + fraction) * 2^(exponent - 25). */
double ropekv_oracle_f16_to_f64(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1F;
    int f = bits & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f != 0) ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Round to the nearest binary16 value, ties to even. Scaling by a power of two
 * is exact in double, so nearbyint (default mode: to nearest, ties to even)
 * applied to the scaled value rounds the exact input. */
uint16_t ropekv_oracle_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00u);
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: multiples of 2^-24; 1024 * 2^-24 is the smallest
         * normal, whose encoding 0x0400 is exactly the integer 1024. */
        double k = nearbyint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)k);
    }
    int E;
    (void)frexp(a, &E);
    E -= 1; /* 2^E <= a < 2^(E+1) */
    double q = nearbyint(ldexp(a, 10 - E)); /* significand * 2^10, in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    if (E > 15)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* ---------------------------------------------------------------- FP8 ----- */

/* E4M3: exponent field 0 is subnormal, value = fraction * 2^-9; otherwise
 * value = (8 + fraction) * 2^(exponent - 10); S.1111.111 is NaN. */
double ropekv_oracle_e4m3_to_f64(uint8_t bits)
{
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int f = bits & 0x7;
    double v;
    if (e == 15 && f == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

uint8_t ropekv_oracle_f64_to_e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80u : 0u;
    double a = fabs(x);
    if (isinf(a)) /* saturates like any magnitude above 448 */
        return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormals: multiples of 2^-9; 8 * 2^-9 is the smallest normal 0x08 */
        double k = nearbyint(ldexp(a, 9));
        return (uint8_t)(sign | (uint8_t)k);
    }
    int E;
    (void)frexp(a, &E);
    E -= 1; /* 2^E <= a < 2^(E+1) */
    double q = nearbyint(ldexp(a, 3 - E)); /* significand * 8, in [8, 16] */
    if (q == 16.0) {
        q = 8.0;
        E += 1;
    }
    int field = E + 7;
    /* saturate: 448 = S.1111.110 is the largest finite value, S.1111.111 is NaN */
    if (field > 15 || (field == 15 && q - 8.0 > 6.0))
        return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)(field << 3) | (uint8_t)(q - 8.0));
}

/* ---------------------------------------------------------------- RoPE ---- */

void ropekv_oracle_rotate_half(const double* x, int r, int style, double* out)
{
    int h = r / 2;
    for (int d = 0; d < r; ++d) {
        if (style == STYLE_NEOX) {
            /* first half takes minus the second half; second half takes the first */
            out[d] = (d < h) ? -x[d + h] : x[d - h];
        } else {
            /* each pair (2i, 2i+1) becomes (-x_{2i+1}, x_{2i}) */
            out[d] = (d % 2 == 0) ? -x[d + 1] : x[d - 1];
        }
    }
}

int ropekv_oracle_freq_index(int d, int r, int style)
{
    int h = r / 2;
    return (style == STYLE_NEOX) ? (d % h) : (d / 2);
}

void ropekv_oracle_rope_head_f64(const double* x, const float* cs_row, int D, int r,
                                 int style, double* y)
{
    int h = r / 2;
    double* rot = (double*)calloc((size_t)(r > 0 ? r : 1), sizeof(double));
    ropekv_oracle_rotate_half(x, r, style, rot);
    for (int d = 0; d < r; ++d) {
        int f = ropekv_oracle_freq_index(d, r, style);
        double c = (double)cs_row[f];
        double s = (double)cs_row[h + f];
        y[d] = x[d] * c + rot[d] * s;
    }
    for (int d = r; d < D; ++d)
        y[d] = x[d];
    free(rot);
}

/* Rotate one FP16 head (src, D elements) with table row cs and write it to dst:
 * rotated dims rounded to FP16, dims >= r copied as bits. src and dst may be
 * the same array (the in-place packed case). */
static void rope_head_f16(const uint16_t* src, const float* cs, int D, int r, int style,
                          uint16_t* dst)
{
    double* x = (double*)calloc((size_t)D, sizeof(double));
    double* y = (double*)calloc((size_t)D, sizeof(double));
    for (int d = 0; d < D; ++d)
        x[d] = ropekv_oracle_f16_to_f64(src[d]);
    ropekv_oracle_rope_head_f64(x, cs, D, r, style, y);
    uint16_t* out = (uint16_t*)calloc((size_t)D, sizeof(uint16_t));
    for (int d = 0; d < r; ++d)
        out[d] = ropekv_oracle_f64_to_f16(y[d]);
    for (int d = r; d < D; ++d)
        out[d] = src[d];
    memcpy(dst, out, sizeof(uint16_t) * (size_t)D);
    free(out);
    free(y);
    free(x);
}

static int dims_ok(int B, int S, int Hq, int Hkv, int D, int r, int cap, int csBatch,
                   int csSeq, int style)
{
    if (B < 0 || S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || cap < 0 || csSeq < 0)
        return 0;
    if (Hq % Hkv != 0)
        return 0;
    if (r <= 0 || r % 2 != 0 || r > D)
        return 0;
    if (csBatch != 1 && csBatch != B)
        return 0;
    if (style != STYLE_NEOX && style != STYLE_GPTJ)
        return 0;
    return 1;
}

/* Element offsets of the contiguous layouts of "Apply Rope Write KV". */
static size_t qkv_at(int b, int s, int head, int S, int H, int D)
{
    return (((size_t)b * S + s) * H + head) * (size_t)D;
}
static size_t cache_at(int b, int plane, int hk, int slot, int Hkv, int cap, int D)
{
    return ((((size_t)b * 2 + plane) * Hkv + hk) * (size_t)cap + slot) * (size_t)D;
}
static size_t qout_at(int b, int s, int hq, int S, int Hq, int D)
{
    return (((size_t)b * S + s) * Hq + hq) * (size_t)D;
}
static const float* cs_row_at(const float* cosSin, int b, int pos, int csBatch, int csSeq,
                              int r)
{
    int bc = (csBatch == 1) ? 0 : b;
    return cosSin + ((size_t)bc * csSeq + pos) * (size_t)r;
}

/* One token of the contiguous-cache paths: Q heads to qDst (a pointer to the
 * token's first Q head in either qkv or qOut), K heads to plane 0 and V bits to
 * plane 1 of the cache at slot. */
static void token_write(const uint16_t* qkv_tok, uint16_t* qDst, uint16_t* kvCache,
                        const float* cs, int b, int slot, int Hq, int Hkv, int D, int r,
                        int cap, int style, int k_in_place, uint16_t* qkv_tok_mut)
{
    for (int hq = 0; hq < Hq; ++hq)
        rope_head_f16(qkv_tok + (size_t)hq * D, cs, D, r, style, qDst + (size_t)hq * D);
    for (int hk = 0; hk < Hkv; ++hk) {
        uint16_t* kc = kvCache + cache_at(b, 0, hk, slot, Hkv, cap, D);
        rope_head_f16(qkv_tok + (size_t)(Hq + hk) * D, cs, D, r, style, kc);
        if (k_in_place)
            memcpy(qkv_tok_mut + (size_t)(Hq + hk) * D, kc, sizeof(uint16_t) * (size_t)D);
    }
    for (int hv = 0; hv < Hkv; ++hv) {
        uint16_t* vc = kvCache + cache_at(b, 1, hv, slot, Hkv, cap, D);
        memcpy(vc, qkv_tok + (size_t)(Hq + Hkv + hv) * D, sizeof(uint16_t) * (size_t)D);
    }
}

int ropekv_oracle_packed(const float* cosSin, uint16_t* qkv, uint16_t* kvCache,
                         int B, int S, int Hq, int Hkv, int D, int r, int cap,
                         int csBatch, int csSeq, int style)
{
    if (!dims_ok(B, S, Hq, Hkv, D, r, cap, csBatch, csSeq, style))
        return -1;
    if (S > cap || S > csSeq)
        return -1;
    int H = Hq + 2 * Hkv;
    for (int b = 0; b < B; ++b) {
        for (int s = 0; s < S; ++s) {
            int pos = s; /* empty cache: the tokens fill it from slot 0 */
            int slot = s;
            uint16_t* tok = qkv + qkv_at(b, s, 0, S, H, D);
            const float* cs = cs_row_at(cosSin, b, pos, csBatch, csSeq, r);
            /* Q rotated in place; K rotated into the cache and back into qkv */
            token_write(tok, tok, kvCache, cs, b, slot, Hq, Hkv, D, r, cap, style, 1, tok);
        }
    }
    return 0;
}

int ropekv_oracle_continuous(const float* cosSin, const int32_t* kvCacheEndLens,
                             const uint16_t* qkv, uint16_t* kvCache, uint16_t* qOut,
                             int B, int S, int Hq, int Hkv, int D, int r, int cap,
                             int csBatch, int csSeq, int style)
{
    if (!dims_ok(B, S, Hq, Hkv, D, r, cap, csBatch, csSeq, style))
        return -1;
    int H = Hq + 2 * Hkv;
    for (int b = 0; b < B; ++b) {
        for (int s = 0; s < S; ++s) {
            /* kvCacheEndLens is where the sequence ends once the S new
             * tokens are in: they take slots end-S .. end-1, and their
             * positions equal their slots. */
            long long slot = (long long)kvCacheEndLens[b] - S + s;
            long long pos = slot;
            if (slot < 0 || slot >= cap || pos >= csSeq)
                continue;
            const uint16_t* tok = qkv + qkv_at(b, s, 0, S, H, D);
            const float* cs = cs_row_at(cosSin, b, (int)pos, csBatch, csSeq, r);
            token_write(tok, qOut + qout_at(b, s, 0, S, Hq, D), kvCache, cs, b, (int)slot,
                        Hq, Hkv, D, r, cap, style, 0, NULL);
        }
    }
    return 0;
}

int ropekv_oracle_tree(const float* cosSin, const int32_t* kvCacheEndLens,
                       const int32_t* tokenPosIds, const uint16_t* qkv,
                       uint16_t* kvCache, uint16_t* qOut,
                       int B, int S, int Hq, int Hkv, int D, int r, int cap,
                       int csBatch, int csSeq, int style)
{
    if (!dims_ok(B, S, Hq, Hkv, D, r, cap, csBatch, csSeq, style))
        return -1;
    int H = Hq + 2 * Hkv;
    for (int b = 0; b < B; ++b) {
        for (int s = 0; s < S; ++s) {
            /* RoPE position from the tree; cache slot in linear token order */
            long long pos = tokenPosIds[(size_t)b * S + s];
            long long slot = (long long)kvCacheEndLens[b] - S + s;
            if (pos < 0 || pos >= csSeq || slot < 0 || slot >= cap)
                continue;
            const uint16_t* tok = qkv + qkv_at(b, s, 0, S, H, D);
            const float* cs = cs_row_at(cosSin, b, (int)pos, csBatch, csSeq, r);
            token_write(tok, qOut + qout_at(b, s, 0, S, Hq, D), kvCache, cs, b, (int)slot,
                        Hq, Hkv, D, r, cap, style, 0, NULL);
        }
    }
    return 0;
}

int ropekv_oracle_paged_rows(const uint16_t* kDelta, const uint16_t* vDelta,
                             const float* tokenAlignedCosSin,
                             const int32_t* deltaPositions, const int32_t* deltaTokenToSequence,
                             const int32_t* pageTable,
                             int numDeltaTokens, int batchSize, int Hkv, int D, int r,
                             int numPages, int maxPagesPerSeq, int tokensPerPage, int style,
                             int64_t* kDest, int64_t* vDest, uint16_t* kOut, uint16_t* vOut)
{
    if (numDeltaTokens < 0 || batchSize < 0 || Hkv <= 0 || D <= 0 || r <= 0 || r % 2 != 0 ||
        r > D || numPages < 0 || maxPagesPerSeq < 0 || tokensPerPage <= 0 ||
        (style != STYLE_NEOX && style != STYLE_GPTJ))
        return -1;
    size_t rowElems = (size_t)Hkv * D;
    for (int t = 0; t < numDeltaTokens; ++t) {
        kDest[t] = -1;
        vDest[t] = -1;
        int32_t pos = deltaPositions[t];
        int32_t seq = deltaTokenToSequence[t];
        /* negative position or sequence: padding row */
        if (pos < 0 || seq < 0 || seq >= batchSize)
            continue;
        int32_t lp = pos / tokensPerPage; /* logical page of the sequence */
        if (lp >= maxPagesPerSeq)         /* outside the sequence's capacity */
            continue;
        int32_t inPage = pos % tokensPerPage;
        int32_t idK = pageTable[((size_t)seq * 2 + 0) * maxPagesPerSeq + lp];
        int32_t idV = pageTable[((size_t)seq * 2 + 1) * maxPagesPerSeq + lp];
        /* canonical ids are flat page indices of the [2, numPages] pool: the K
         * plane owns [0, numPages), the V plane [numPages, 2*numPages) */
        if (idK >= 0 && idK < numPages) {
            kDest[t] = ((int64_t)idK * tokensPerPage + inPage) * (int64_t)rowElems;
            const float* cs = tokenAlignedCosSin + (size_t)t * r; /* row t, not row pos */
            for (int hk = 0; hk < Hkv; ++hk)
                rope_head_f16(kDelta + (size_t)t * rowElems + (size_t)hk * D, cs, D, r, style,
                              kOut + (size_t)t * rowElems + (size_t)hk * D);
        }
        if (idV >= numPages && (int64_t)idV < 2 * (int64_t)numPages) {
            vDest[t] = ((int64_t)idV * tokensPerPage + inPage) * (int64_t)rowElems;
            memcpy(vOut + (size_t)t * rowElems, vDelta + (size_t)t * rowElems,
                   sizeof(uint16_t) * rowElems);
        }
    }
    return 0;
}

int ropekv_oracle_paged(const uint16_t* kDelta, const uint16_t* vDelta, uint16_t* kvCache,
                        const float* tokenAlignedCosSin,
                        const int32_t* deltaPositions, const int32_t* deltaTokenToSequence,
                        const int32_t* pageTable,
                        int numDeltaTokens, int batchSize, int Hkv, int D, int r,
                        int numPages, int maxPagesPerSeq, int tokensPerPage, int style)
{
    size_t n = (size_t)(numDeltaTokens > 0 ? numDeltaTokens : 1);
    size_t rowElems = (size_t)(Hkv > 0 ? Hkv : 1) * (size_t)(D > 0 ? D : 1);
    int64_t* kDest = (int64_t*)malloc(sizeof(int64_t) * n);
    int64_t* vDest = (int64_t*)malloc(sizeof(int64_t) * n);
    uint16_t* kOut = (uint16_t*)calloc(n * rowElems, sizeof(uint16_t));
    uint16_t* vOut = (uint16_t*)calloc(n * rowElems, sizeof(uint16_t));
    int rc = ropekv_oracle_paged_rows(kDelta, vDelta, tokenAlignedCosSin, deltaPositions,
                                      deltaTokenToSequence, pageTable, numDeltaTokens,
                                      batchSize, Hkv, D, r, numPages, maxPagesPerSeq,
                                      tokensPerPage, style, kDest, vDest, kOut, vOut);
    if (rc == 0) {
        for (int t = 0; t < numDeltaTokens; ++t) {
            if (kDest[t] >= 0)
                memcpy(kvCache + kDest[t], kOut + (size_t)t * rowElems,
                       sizeof(uint16_t) * rowElems);
            if (vDest[t] >= 0)
                memcpy(kvCache + vDest[t], vOut + (size_t)t * rowElems,
                       sizeof(uint16_t) * rowElems);
        }
    }
    free(vOut);
    free(kOut);
    free(vDest);
    free(kDest);
    return rc;
}

int ropekv_oracle_delta_metadata(const int32_t* oldDraftCacheLengths, const int32_t* deltaLengths,
                                 int deltaWidth, int32_t* deltaPositions,
                                 int32_t* deltaTokenToSequence, int batchSize)
{
    if (deltaWidth < 0 || batchSize < 0)
        return -1;
    for (int b = 0; b < batchSize; ++b) {
        int len = deltaLengths[b]; /* rows past deltaWidth do not exist */
        for (int j = 0; j < deltaWidth; ++j) {
            size_t t = (size_t)b * deltaWidth + j;
            if (j < len) {
                /* the target length after the delta is old + len; the delta's
                 * own tokens sit at old .. old + len - 1 */
                deltaPositions[t] = oldDraftCacheLengths[b] + j;
                deltaTokenToSequence[t] = b;
            } else {
                deltaPositions[t] = -1;
                deltaTokenToSequence[t] = -1;
            }
        }
    }
    return 0;
}

int ropekv_oracle_gather_delta_rope(const float* source, float* output,
                                    const int32_t* deltaPositions,
                                    const int32_t* deltaTokenToSequence,
                                    const int32_t* stateIndices, int numDeltaTokens,
                                    int batchSize, int sourceRows, int cacheCapacity,
                                    int rotaryDim)
{
    if (numDeltaTokens < 0 || batchSize < 0 || sourceRows < 0 || cacheCapacity < 0 ||
        rotaryDim <= 0)
        return -1;
    for (int t = 0; t < numDeltaTokens; ++t) {
        float* out = output + (size_t)t * rotaryDim;
        int32_t pos = deltaPositions[t];
        int32_t seq = deltaTokenToSequence[t];
        int ok = pos >= 0 && seq >= 0 && seq < batchSize && pos < cacheCapacity;
        int32_t state = -1;
        if (ok) {
            if (stateIndices != NULL)
                state = stateIndices[seq];
            else
                state = (sourceRows == 1) ? 0 : seq;
            ok = state >= 0 && state < sourceRows;
        }
        for (int d = 0; d < rotaryDim; ++d)
            out[d] = ok ? source[((size_t)state * cacheCapacity + pos) * rotaryDim + d] : 0.0f;
    }
    return 0;
}

int ropekv_oracle_paged_fused(const uint16_t* kDelta, const uint16_t* vDelta, uint16_t* kvCache,
                              const float* source, const int32_t* oldDraftCacheLengths,
                              const int32_t* deltaLengths, int deltaWidth,
                              const int32_t* stateIndices, const int32_t* pageTable,
                              int batchSize, int Hkv, int D, int r, int numPages,
                              int maxPagesPerSeq, int tokensPerPage, int sourceRows,
                              int cacheCapacity, int style)
{
    if (batchSize < 0 || deltaWidth < 0 || r <= 0)
        return -1;
    size_t n = (size_t)batchSize * (size_t)deltaWidth;
    size_t nn = n > 0 ? n : 1;
    int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * nn);
    int32_t* seq = (int32_t*)malloc(sizeof(int32_t) * nn);
    float* cs = (float*)calloc(nn * (size_t)r, sizeof(float));
    int rc = ropekv_oracle_delta_metadata(oldDraftCacheLengths, deltaLengths, deltaWidth, pos, seq,
                                          batchSize);
    if (rc == 0)
        rc = ropekv_oracle_gather_delta_rope(source, cs, pos, seq, stateIndices, (int)n,
                                             batchSize, sourceRows, cacheCapacity, r);
    if (rc == 0)
        rc = ropekv_oracle_paged(kDelta, vDelta, kvCache, cs, pos, seq, pageTable, (int)n,
                                 batchSize, Hkv, D, r, numPages, maxPagesPerSeq, tokensPerPage,
                                 style);
    free(cs);
    free(seq);
    free(pos);
    return rc;
}

void ropekv_oracle_rms_norm_f64(const double* x, const uint16_t* weight, double eps, int D,
                                double* y)
{
    double ss = 0.0;
    for (int d = 0; d < D; ++d)
        ss += x[d] * x[d];
    double inv = 1.0 / sqrt(ss / D + eps);
    for (int d = 0; d < D; ++d)
        y[d] = x[d] * inv * ropekv_oracle_f16_to_f64(weight[d]);
}

/* Normalize one FP16 head, rotate it and round every dim to FP16. */
static void norm_rope_head_f16(const uint16_t* src, const uint16_t* weight, double eps,
                               const float* cs, int D, int r, int style, uint16_t* dst)
{
    double* x = (double*)calloc((size_t)D, sizeof(double));
    double* n = (double*)calloc((size_t)D, sizeof(double));
    double* y = (double*)calloc((size_t)D, sizeof(double));
    for (int d = 0; d < D; ++d)
        x[d] = ropekv_oracle_f16_to_f64(src[d]);
    ropekv_oracle_rms_norm_f64(x, weight, eps, D, n);
    ropekv_oracle_rope_head_f64(n, cs, D, r, style, y);
    for (int d = 0; d < D; ++d)
        dst[d] = ropekv_oracle_f64_to_f16(y[d]);
    free(y);
    free(n);
    free(x);
}

int ropekv_oracle_continuous_qknorm(const float* cosSin, const int32_t* kvCacheEndLens,
                                    const uint16_t* qkv, uint16_t* kvCache, uint16_t* qOut,
                                    const uint16_t* qNormWeight, const uint16_t* kNormWeight,
                                    float eps, int B, int S, int Hq, int Hkv, int D, int r,
                                    int cap, int csBatch, int csSeq, int style)
{
    if (!dims_ok(B, S, Hq, Hkv, D, r, cap, csBatch, csSeq, style))
        return -1;
    int H = Hq + 2 * Hkv;
    for (int b = 0; b < B; ++b) {
        for (int s = 0; s < S; ++s) {
            /* slot = position = end - S + s, as in the continuous call */
            long long pos = (long long)kvCacheEndLens[b] - S + s;
            long long slot = pos;
            if (slot < 0 || slot >= cap || pos >= csSeq)
                continue;
            const uint16_t* tok = qkv + qkv_at(b, s, 0, S, H, D);
            const float* cs = cs_row_at(cosSin, b, (int)pos, csBatch, csSeq, r);
            for (int hq = 0; hq < Hq; ++hq)
                norm_rope_head_f16(tok + (size_t)hq * D, qNormWeight, (double)eps, cs, D, r,
                                   style, qOut + qout_at(b, s, hq, S, Hq, D));
            for (int hk = 0; hk < Hkv; ++hk)
                norm_rope_head_f16(tok + (size_t)(Hq + hk) * D, kNormWeight, (double)eps, cs, D,
                                   r, style, kvCache + cache_at(b, 0, hk, (int)slot, Hkv, cap, D));
            for (int hv = 0; hv < Hkv; ++hv)
                memcpy(kvCache + cache_at(b, 1, hv, (int)slot, Hkv, cap, D),
                       tok + (size_t)(Hq + Hkv + hv) * D, sizeof(uint16_t) * (size_t)D);
        }
    }
    return 0;
}

int ropekv_oracle_continuous_fp8(const float* cosSin, const int32_t* kvCacheEndLens,
                                 const uint16_t* qkv, uint8_t* kvCache8, uint16_t* qOut,
                                 float kScale, float vScale, int B, int S, int Hq, int Hkv, int D,
                                 int r, int cap, int csBatch, int csSeq, int style)
{
    if (!dims_ok(B, S, Hq, Hkv, D, r, cap, csBatch, csSeq, style) || !(kScale > 0.0f) ||
        !(vScale > 0.0f))
        return -1;
    int H = Hq + 2 * Hkv;
    double* x = (double*)calloc((size_t)D, sizeof(double));
    double* y = (double*)calloc((size_t)D, sizeof(double));
    for (int b = 0; b < B; ++b) {
        for (int s = 0; s < S; ++s) {
            /* slots and positions exactly as the continuous call */
            long long end = kvCacheEndLens[b];
            long long slot = end - S + s;
            if (slot < 0 || slot >= cap || slot >= csSeq)
                continue;
            const uint16_t* tok = qkv + qkv_at(b, s, 0, S, H, D);
            const float* cs = cs_row_at(cosSin, b, (int)slot, csBatch, csSeq, r);
            for (int hq = 0; hq < Hq; ++hq)
                rope_head_f16(tok + (size_t)hq * D, cs, D, r, style,
                              qOut + qout_at(b, s, hq, S, Hq, D));
            for (int hk = 0; hk < Hkv; ++hk) {
                for (int d = 0; d < D; ++d)
                    x[d] = ropekv_oracle_f16_to_f64(tok[(size_t)(Hq + hk) * D + d]);
                ropekv_oracle_rope_head_f64(x, cs, D, r, style, y);
                uint8_t* kc = kvCache8 + cache_at(b, 0, hk, (int)slot, Hkv, cap, D);
                for (int d = 0; d < D; ++d)
                    kc[d] = ropekv_oracle_f64_to_e4m3(y[d] * (1.0 / (double)kScale));
            }
            for (int hv = 0; hv < Hkv; ++hv) {
                const uint16_t* vsrc = tok + (size_t)(Hq + Hkv + hv) * D;
                uint8_t* vc = kvCache8 + cache_at(b, 1, hv, (int)slot, Hkv, cap, D);
                for (int d = 0; d < D; ++d)
                    vc[d] = ropekv_oracle_f64_to_e4m3(ropekv_oracle_f16_to_f64(vsrc[d]) *
                                                      (1.0 / (double)vScale));
            }
        }
    }
    free(y);
    free(x);
    return 0;
}

int ropekv_oracle_slot_mapping(const float* cosSin, const int64_t* positions,
                               const uint16_t* q, int64_t qStride, const uint16_t* k,
                               int64_t kStride, const uint16_t* v, int64_t vStride,
                               const int64_t* slotMapping, uint16_t* keyCache,
                               uint16_t* valueCache, uint16_t* qOut, uint16_t* kOut, int T,
                               int Hq, int Hkv, int D, int r, int cosSinRows, int64_t numBlocks,
                               int blockSize, int style)
{
    if (T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || r <= 0 || r % 2 != 0 ||
        r > D || cosSinRows < 0 || numBlocks < 0 || blockSize <= 0 ||
        (style != STYLE_NEOX && style != STYLE_GPTJ))
        return -1;
    int64_t slots = numBlocks * (int64_t)blockSize;
    for (int t = 0; t < T; ++t) {
        int64_t pos = positions[t];
        if (pos < 0 || pos >= cosSinRows)
            continue; /* no table row: nothing is written for the token */
        const float* cs = cosSin + (size_t)pos * r;
        for (int hq = 0; hq < Hq; ++hq)
            rope_head_f16(q + (size_t)t * qStride + (size_t)hq * D, cs, D, r, style,
                          qOut + ((size_t)t * Hq + hq) * D);
        int64_t slot = slotMapping[t];
        if (slot < 0 || slot >= slots)
            continue; /* the cache write (and kOut) is skipped */
        int64_t block = slot / blockSize;
        int64_t off = slot % blockSize;
        for (int hk = 0; hk < Hkv; ++hk) {
            uint16_t* kc = keyCache + (((size_t)block * blockSize + off) * Hkv + hk) * D;
            rope_head_f16(k + (size_t)t * kStride + (size_t)hk * D, cs, D, r, style, kc);
            if (kOut != NULL)
                memcpy(kOut + ((size_t)t * Hkv + hk) * D, kc, sizeof(uint16_t) * (size_t)D);
            uint16_t* vc = valueCache + (((size_t)block * blockSize + off) * Hkv + hk) * D;
            memcpy(vc, v + (size_t)t * vStride + (size_t)hk * D, sizeof(uint16_t) * (size_t)D);
        }
    }
    return 0;
}

int ropekv_oracle_capacity_rejected(int32_t cosSinSeqLen, int32_t kvCapacity)
{
    /* the RoPE table may be shorter than the page-aligned capacity; only a
     * longer table is rejected */
    return cosSinSeqLen > kvCapacity ? 1 : 0;
}
