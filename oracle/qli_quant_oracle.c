/*
 * CPU oracle for the two steps either side of the indexer's paged gather:
 * the per-head INT8 quantisation of the indexer queries and the write of new
 * index-K rows (INT8 plus FP16 scale) into their PA_BBND page slots.
 *
 * TEST INFRASTRUCTURE, like qli_oracle.c: only the tests, the smoke check and
 * the bench's CPU legs may build and call it. It shares no code, header or
 * constant with the CUDA library. One row at a time, in the order below.
 *
 * Sources (web pages, cited by title and section):
 *  [G]  vllm-ascend developer guide "DeepSeek V4.1 QLI V2 与候选集成",
 *       section "数据流" (data flow): the indexer's projected queries are
 *       quantised per head to INT8, each head with a scale that is
 *       representable in FP16; head weights and K scales are FP16; the
 *       allocator packs the index K and its FP16 scales after the KV inside
 *       the shared page (64-row view, 131072-byte pages for ratio 2; 128-row
 *       view, 147712-byte pages for ratio 1).
 *  [B]  blog "DeepSeek V4.1-Flash 登陆昇腾 · 需求故事（PR 16925）", section 四:
 *       one block ID locates the page that holds both the KV and the index K.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes):
 *  - Inputs are BF16 rows of D values (the projection's output type).
 *  - Symmetric absmax quantisation with 127 levels per side, one scale per
 *    row (a query head, or one index-K position):
 *        amax = max_d |x_d|                       (exact in FP32)
 *        s    = FP16(amax / 127)                  (FP32 quotient, then RN)
 *        q_d  = clamp(rint(x_d / s), -127, 127)   (FP32 quotient, ties to even)
 *    "Representable FP16 scale" is read as: the scale used to divide is the
 *    FP16 value that is stored, so q * s is the dequantised value.
 *  - s is capped at the largest finite FP16 (65504) when amax / 127 rounds
 *    past it; when s rounds to zero (amax < 2^-25 * 127, including an
 *    all-zero row) the row's codes are all 0 with scale +0.
 *  - Non-finite inputs are outside the contract (rejected here).
 *  - The index-K row for slot m (m = page * R + row) goes to the page's
 *    index-K region at k_offset + row * 128 and its scale to
 *    scale_offset + row * 2; a negative slot means "no row" (padding) and
 *    writes nothing; a slot at or past num_pages * R is an error and writes
 *    nothing. Rows are written in input order (the slots of one call are
 *    expected to be distinct).
 *
 * Build with -ffp-contract=off and without -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define QORACLE_OK 0
#define QORACLE_EINVAL (-1)
#define QORACLE_ENONFINITE (-2)
#define QORACLE_ESLOT (-5)

/* BF16 bit pattern -> FP32 (exact: BF16 is the top half of an FP32). */
float oracle_bf16_to_f32(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t f16_bits(_Float16 h) {
    uint16_t b;
    memcpy(&b, &h, sizeof b);
    return b;
}

/* A row's absmax and its FP16 scale s = FP16(amax / levels): FP32 quotient,
 * then RN-even to binary16, capped at the largest finite FP16. Returns 0, or
 * QORACLE_ENONFINITE for a row holding an Inf or NaN. */
static int row_scale(const uint16_t *x, int32_t D, float levels, _Float16 *s_out) {
    float amax = 0.0f;
    for (int32_t d = 0; d < D; ++d) {
        const float v = oracle_bf16_to_f32(x[d]);
        if (!isfinite(v)) return QORACLE_ENONFINITE;
        const float a = fabsf(v);
        if (a > amax) amax = a;
    }
    const float quotient = amax / levels;
    _Float16 s = (_Float16)quotient;                 /* RN-even to binary16 */
    if (isinf((float)s)) s = (_Float16)65504.0f;     /* largest finite FP16 */
    *s_out = s;
    return QORACLE_OK;
}

/* One row: D BF16 values -> D INT8 codes and the FP16 scale bits. Returns 0,
 * or QORACLE_ENONFINITE for a row holding an Inf or NaN. */
int oracle_quant_row(const uint16_t *x, int32_t D, int8_t *q, uint16_t *scale_bits) {
    _Float16 s;
    const int e = row_scale(x, D, 127.0f, &s);
    if (e) return e;
    const float sf = (float)s;
    if (sf == 0.0f) {
        memset(q, 0, (size_t)D);
        *scale_bits = 0;                             /* +0 */
        return QORACLE_OK;
    }
    for (int32_t d = 0; d < D; ++d) {
        float r = rintf(oracle_bf16_to_f32(x[d]) / sf);   /* current mode: to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[d] = (int8_t)r;
    }
    *scale_bits = f16_bits(s);
    return QORACLE_OK;
}

/* Queries: rows = T * N heads of D values, contiguous; codes [rows, D] and
 * scales [rows] (the indexer's TND q and [T, N] q_scale). */
int oracle_quantize_rows(const uint16_t *x, int64_t rows, int32_t D, int8_t *q,
                         uint16_t *scales) {
    if (rows < 0 || D <= 0 || (rows > 0 && (!x || !q || !scales))) return QORACLE_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        const int e = oracle_quant_row(x + r * D, D, q + r * D, scales + r);
        if (e) return e;
    }
    return QORACLE_OK;
}

/* ---- FP8 (E4M3) variant -------------------------------------------------
 * Quant mode 1, which the pages only name (A5 dtype registration). Reading:
 * the same symmetric absmax scheme with E4M3's largest finite value 448 in
 * place of 127:
 *     s   = FP16(amax / 448)            (FP32 quotient, then RN; capped at 65504)
 *     c_d = E4M3(x_d / s)               (FP32 quotient, RN-even, saturated to +-448)
 * s rounding to zero gives codes 0 (+0) and scale +0. */

/* E4M3 code of a finite FP32 value: round to nearest even on the E4M3 grid
 * (quantum 2^-9 below 2^-6, 2^(e-3) in binade [2^e, 2^(e+1))), magnitudes
 * past 448 saturated to 448. */
uint8_t oracle_f32_to_e4m3(float v) {
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    int e;
    (void)frexp(a, &e);                  /* a = f * 2^e, f in [0.5, 1): binade 2^(e-1) */
    int binade = e - 1;
    if (a == 0.0 || binade < -6) binade = -6;    /* subnormal range shares the quantum 2^-9 */
    const double quantum = ldexp(1.0, binade - 3);
    double n = nearbyint(a / quantum);   /* exact division; current mode: to even */
    double r = n * quantum;
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    /* encode r, exactly on the grid */
    int er;
    (void)frexp(r, &er);
    int b = er - 1;
    uint8_t code;
    if (b < -6) {
        code = (uint8_t)(r / ldexp(1.0, -9));                 /* subnormal: m * 2^-9 */
    } else {
        const int m = (int)(r / ldexp(1.0, b - 3)) - 8;       /* (8 + m) * 2^(b-3) */
        code = (uint8_t)(((b + 7) << 3) | m);
    }
    return sign | code;
}

/* One row: D BF16 values -> D E4M3 codes and the FP16 scale bits. Returns 0,
 * or QORACLE_ENONFINITE for a row holding an Inf or NaN. */
int oracle_quant_row_e4m3(const uint16_t *x, int32_t D, uint8_t *c, uint16_t *scale_bits) {
    _Float16 s;
    const int e = row_scale(x, D, 448.0f, &s);
    if (e) return e;
    const float s8 = (float)s;
    if (s8 == 0.0f) {
        memset(c, 0, (size_t)D);
        *scale_bits = 0;
        return QORACLE_OK;
    }
    for (int32_t d = 0; d < D; ++d) c[d] = oracle_f32_to_e4m3(oracle_bf16_to_f32(x[d]) / s8);
    *scale_bits = f16_bits(s);
    return QORACLE_OK;
}

int oracle_quantize_rows_e4m3(const uint16_t *x, int64_t rows, int32_t D, uint8_t *c,
                              uint16_t *scales) {
    if (rows < 0 || D <= 0 || (rows > 0 && (!x || !c || !scales))) return QORACLE_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        const int e = oracle_quant_row_e4m3(x + r * D, D, c + r * D, scales + r);
        if (e) return e;
    }
    return QORACLE_OK;
}

/* Index K: n new rows of D = 128 BF16 values, slot[i] = page * R + row.
 * Writes each row's codes (INT8, or E4M3 when fp8) and scale into the page
 * pool `cache`. Returns 0, or the first error (every valid row is still
 * written). */
static int write_index_k_rows(const uint16_t *k, int64_t n, int32_t D, const int64_t *slot,
                              uint8_t *cache, int64_t num_pages, int64_t page_stride, int32_t R,
                              int64_t k_offset, int64_t scale_offset, int fp8) {
    if (n < 0 || D <= 0 || R <= 0 || num_pages < 0 || (n > 0 && (!k || !slot || !cache)))
        return QORACLE_EINVAL;
    int err = QORACLE_OK;
    int8_t codes[4096];
    if (D > 4096) return QORACLE_EINVAL;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t m = slot[i];
        if (m < 0) continue;
        if (m >= num_pages * (int64_t)R) {
            if (!err) err = QORACLE_ESLOT;
            continue;
        }
        uint16_t s;
        const int e = fp8 ? oracle_quant_row_e4m3(k + i * D, D, (uint8_t *)codes, &s)
                          : oracle_quant_row(k + i * D, D, codes, &s);
        if (e) {
            if (!err) err = e;
            continue;
        }
        const int64_t page = m / R, row = m % R;
        uint8_t *p = cache + page * page_stride;
        memcpy(p + k_offset + row * (int64_t)D, codes, (size_t)D);
        memcpy(p + scale_offset + row * 2, &s, 2);
    }
    return err;
}

int oracle_write_index_k(const uint16_t *k, int64_t n, int32_t D, const int64_t *slot,
                         uint8_t *cache, int64_t num_pages, int64_t page_stride, int32_t R,
                         int64_t k_offset, int64_t scale_offset) {
    return write_index_k_rows(k, n, D, slot, cache, num_pages, page_stride, R, k_offset,
                              scale_offset, 0);
}

/* The FP8 variant: E4M3 codes (oracle_quant_row_e4m3) in the same places. */
int oracle_write_index_k_e4m3(const uint16_t *k, int64_t n, int32_t D, const int64_t *slot,
                              uint8_t *cache, int64_t num_pages, int64_t page_stride, int32_t R,
                              int64_t k_offset, int64_t scale_offset) {
    return write_index_k_rows(k, n, D, slot, cache, num_pages, page_stride, R, k_offset,
                              scale_offset, 1);
}
