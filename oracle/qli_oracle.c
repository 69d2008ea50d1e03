/*
 * CPU oracle for the DeepSeek-V4.1 quantized lightning indexer (QLI).
 *
 * TEST INFRASTRUCTURE. This file is the plain, slow statement of what the
 * indexer computes, used only to check the CUDA path: the tests, the smoke
 * check and the bench's CPU-baseline leg may build and call it; the product
 * path never does. It shares no code, header or constant with the CUDA
 * library. Every number is computed one pair at a time in the order the
 * definition gives; the only parallelism is an OpenMP loop over independent
 * (query, position) pairs, which does not change any result.
 *
 * Sources (web pages, cited by title and section):
 *  [G]  vllm-ascend developer guide "DeepSeek V4.1 QLI V2 与候选集成":
 *       [G/data-flow]  section "数据流" (data flow): paged PA_BBND index K,
 *                      metadata (raw query boundaries, compressed K lengths,
 *                      raw length mod ratio; residual absent for ratio 1),
 *                      the three candidate modes, candidate tensor
 *                      [tokens, 1, blocks] of INT32 block IDs padded with -1,
 *                      8 positions per block, block score = max position
 *                      score, last visible block pinned, chronological
 *                      position order with -1 moved to the end, empty context
 *                      gives empty indices and all-invalid candidates,
 *                      consumer without a source raises.
 *       [G/contract]   section "当前 A3 契约" (current A3 contract): INT8 Q/K,
 *                      FP16 head weights, per-head Q scale, per-token K scale,
 *                      32 or 64 heads, head dim 128, one index-K head, ratio 1
 *                      or 2, causal mask mode 3, TopK in [1, 2048], candidate
 *                      blocks in [64, 2048] and a multiple of 64, block size 8,
 *                      and the numeric golden: INT32 QK / 1024, FP16 ReLU and
 *                      weight * Q_scale, FP32 reduction over heads, then the
 *                      K scale.
 *       [G/coverage]   section "构建与回归覆盖": the candidate tensor size is
 *                      T * N_k * blocks (no extra factor of the batch size).
 *  [B]  blog "DeepSeek V4.1-Flash 登陆昇腾 · 需求故事（PR 16925）", section 四
 *       (implementation), get_layer_tuples: the index K and its FP16 scale sit
 *       after the KV in the same page; one block ID locates the page.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): mode numbers 1/2/3 = none/source/consumer; compressed position j
 * covers raw positions [j*r, (j+1)*r - 1] and becomes visible to a query at
 * raw position pos once complete, so V = floor((pos + 1) / r); the ReLU'd value
 * times FP16(w * q_scale) is an FP16 multiply; heads are summed in ascending
 * order in FP32 starting from +0; ties in TopK (and -0 == +0) go to the lower
 * position, ties between blocks to the lower block ID; a source's position
 * TopK ranges over all visible positions; a consumer uses the given IDs as a
 * set (duplicates, order, -1 and IDs with no visible position are ignored)
 * and does not add the last block itself. Quant mode 1 (FP8, not in the A3
 * contract): E4M3 codes, the exact dot rounded once to FP32, then the same
 * chain (see the FP8 section below).
 *
 * FP16 arithmetic uses the C _Float16 type (IEEE binary16, round to nearest
 * even). Build with -ffp-contract=off and without -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_CONSUMER_WITHOUT_SOURCE (-3)
#define ORACLE_ERR_RESIDUAL_WITH_RATIO1 (-4)

typedef struct oracle_in {
    const int8_t *q;            /* [T, N, D] at q[t*q_stride_t + h*q_stride_h + d] */
    int64_t q_stride_t, q_stride_h;
    int32_t T, N, D;
    const int32_t *cu_seqlens_q; /* [B+1] raw query boundaries */
    int32_t B;
    const int32_t *k_lens;      /* [B] compressed K lengths */
    const int32_t *residual;    /* [B] raw length mod ratio, NULL when ratio == 1 */
    const uint8_t *cache;       /* page pool */
    int64_t page_stride;
    int32_t rows_per_page;
    int64_t k_offset, scale_offset;
    int64_t num_pages;
    const int32_t *block_table; /* [B, bt_stride] */
    int32_t bt_stride;
    const uint16_t *head_weights; /* FP16 bits [T, N] */
    const uint16_t *q_scale;      /* FP16 bits [T, N] */
    int32_t ratio, topk, cand_mode, cand_blocks;
    const int32_t *cand_in;     /* [T, 1, C] consumer input */
    int32_t quant_mode;         /* 2: INT8 Q/K (the A3 contract); 1: FP8 E4M3 codes */
} oracle_in;

/* ---- FP16 helpers (IEEE binary16 through _Float16) ---------------------- */

float oracle_f16_to_f32(uint16_t bits) {
    _Float16 h;
    memcpy(&h, &bits, 2);
    return (float)h;
}

uint16_t oracle_f32_to_f16(float x) {
    _Float16 h = (_Float16)x; /* one rounding, to nearest even */
    uint16_t bits;
    memcpy(&bits, &h, 2);
    return bits;
}

/* FP16 product of two FP16 values: the FP32 product of two binary16 numbers
 * is exact (11 + 11 significant bits), so rounding it once gives the IEEE
 * binary16 product. */
static float f16_mul(float a, float b) {
    return oracle_f16_to_f32(oracle_f32_to_f16(a * b));
}

/* ---- a1: causal visibility, [G/data-flow] metadata + [G/contract] mask 3 - */

/* Number of compressed positions visible to query i (0-based) of a request
 * with q_len queries, compressed length k_len and raw residual res. The
 * queries are the last q_len raw positions of the S = k_len*r + res raw tokens. */
int64_t oracle_visible_count(int64_t k_len, int64_t res, int32_t ratio,
                             int64_t q_len, int64_t i) {
    int64_t S = k_len * ratio + res;
    int64_t pos = S - q_len + i;     /* raw position of the query */
    int64_t seen = pos + 1;          /* raw tokens at or before it */
    if (seen <= 0) return 0;
    int64_t v = seen / ratio;        /* compressed positions fully covered */
    return v < k_len ? v : k_len;
}

/* ---- a2: paged index-K row, [G/data-flow] PA_BBND + [B] page packing ---- */

static const int8_t *k_row(const oracle_in *in, int32_t b, int64_t j) {
    int64_t slot = j / in->rows_per_page;
    int64_t row = j % in->rows_per_page;
    int64_t page = in->block_table[(int64_t)b * in->bt_stride + slot];
    return (const int8_t *)(in->cache + page * in->page_stride + in->k_offset + row * in->D);
}

static uint16_t k_scale(const oracle_in *in, int32_t b, int64_t j) {
    int64_t slot = j / in->rows_per_page;
    int64_t row = j % in->rows_per_page;
    int64_t page = in->block_table[(int64_t)b * in->bt_stride + slot];
    uint16_t bits;
    memcpy(&bits, in->cache + page * in->page_stride + in->scale_offset + row * 2, 2);
    return bits;
}

/* ---- a3 + a4: one pair's score, [G/contract] numeric golden ------------- */

/* INT32 dot product of query head h of token t with a K row. */
int32_t oracle_dot(const int8_t *qh, const int8_t *k, int32_t D) {
    int32_t s = 0;
    for (int32_t d = 0; d < D; ++d) s += (int32_t)qh[d] * (int32_t)k[d];
    return s;
}

/* The chain after the FP16 rounding: fp16(relu(x) * fp16(w * q_scale)). */
static float chain_from_x(float x, uint16_t w_bits, uint16_t qs_bits) {
    float r = x > 0.0f ? x : 0.0f;                                       /* FP16 ReLU */
    float wq = f16_mul(oracle_f16_to_f32(w_bits), oracle_f16_to_f32(qs_bits)); /* FP16 w*qs */
    return f16_mul(r, wq);                                               /* FP16 product */
}

/* One head's FP16 term: fp16(relu(fp16(s / 1024)) * fp16(w * q_scale)). */
float oracle_head_term(int32_t s, uint16_t w_bits, uint16_t qs_bits) {
    float x = oracle_f16_to_f32(oracle_f32_to_f16((float)s / 1024.0f)); /* INT32/1024 -> FP16 */
    return chain_from_x(x, w_bits, qs_bits);
}

/* ---- FP8 variant (quant mode 1) ------------------------------------------
 * [G/compile-scope] lists FP8 as quant mode 1 of the A5 build's dtype
 * registration; the pages print no golden for it. Reading taken: the codes
 * are OCP E4M3 ("fn": bias 7, no infinities, 0x7F / 0xFF are NaN, largest
 * finite 448) in the same byte layout as the INT8 codes, with the same FP16
 * per-head Q scale and per-position K scale, and the A3 chain from the
 * division by 1024 on; the INT32 dot becomes the exact dot of the decoded
 * codes rounded once to FP32. The exact dot needs no accumulation order:
 * every product is a multiple of 2^-18 below 2^18, so any sum of 128 of them
 * is an integer multiple of 2^-18 below 2^43, exact in double. */

/* Value of an E4M3 code (NaN codes decode to NaN). */
double oracle_e4m3_to_f64(uint8_t c) {
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* subnormal: m/8 * 2^-6 */
    else v = ldexp(8.0 + m, e - 10);                 /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* The exact dot of two rows of E4M3 codes, rounded once to FP32. */
float oracle_dot_e4m3(const uint8_t *qh, const uint8_t *k, int32_t D) {
    double s = 0.0;
    for (int32_t d = 0; d < D; ++d) s += oracle_e4m3_to_f64(qh[d]) * oracle_e4m3_to_f64(k[d]);
    return (float)s;
}

/* The FP8 head term: the A3 chain applied to the FP32 dot. */
float oracle_head_term_f8(float s, uint16_t w_bits, uint16_t qs_bits) {
    float x = oracle_f16_to_f32(oracle_f32_to_f16(s / 1024.0f));       /* /1024 exact, -> FP16 */
    return chain_from_x(x, w_bits, qs_bits);
}

/* Score of (token t of request b, compressed position j). */
static float pair_score(const oracle_in *in, int32_t t, int32_t b, int64_t j) {
    const int8_t *k = k_row(in, b, j);
    float acc = 0.0f;                                 /* FP32 head reduction */
    for (int32_t h = 0; h < in->N; ++h) {
        const int8_t *qh = in->q + (int64_t)t * in->q_stride_t + (int64_t)h * in->q_stride_h;
        const uint16_t w = in->head_weights[(int64_t)t * in->N + h];
        const uint16_t qs = in->q_scale[(int64_t)t * in->N + h];
        if (in->quant_mode == 1)
            acc = acc + oracle_head_term_f8(
                            oracle_dot_e4m3((const uint8_t *)qh, (const uint8_t *)k, in->D), w, qs);
        else
            acc = acc + oracle_head_term(oracle_dot(qh, k, in->D), w, qs);
    }
    return acc * oracle_f16_to_f32(k_scale(in, b, j)); /* then the K scale */
}

float oracle_pair_score(const oracle_in *in, int32_t t, int64_t j) {
    int32_t b = 0;
    while (b + 1 < in->B && in->cu_seqlens_q[b + 1] <= t) ++b;
    return pair_score(in, t, b, j);
}

/* ---- a7/a8 ordering helpers -------------------------------------------- */

typedef struct { float s; int64_t id; } scored;

/* Higher score first; equal scores (including -0 vs +0) by lower id. */
static int by_score_then_id(const void *pa, const void *pb) {
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

static int ascending_i64(const void *pa, const void *pb) {
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    return (a > b) - (a < b);
}

/* Take the first `take` entries of the ordered list, write their ids in
 * ascending order, then -1 up to `width` ([G/data-flow]: chronological order,
 * -1 padding at the end). */
static void emit_ascending(const scored *ordered, int64_t take, int32_t *out, int64_t width) {
    int64_t *ids = (int64_t *)malloc(sizeof(int64_t) * (take > 0 ? take : 1));
    for (int64_t i = 0; i < take; ++i) ids[i] = ordered[i].id;
    qsort(ids, (size_t)take, sizeof(int64_t), ascending_i64);
    for (int64_t i = 0; i < width; ++i) out[i] = i < take ? (int32_t)ids[i] : -1;
    free(ids);
}

/* ---- the whole indexer for a list of query tokens ----------------------- */

/*
 * rows[0..nrows) are query token indices. Outputs are per listed row:
 *   idx_out   [nrows, topk]         position TopK (a7, a8)
 *   cand_out  [nrows, cand_blocks]  source candidates (a6), may be NULL otherwise
 *   scores    [nrows, score_stride] optional: FP32 score of every visible j,
 *                                   NaN-free; entries j >= V are left untouched
 *   visible   [nrows]               optional: V of each row
 * Returns ORACLE_OK or a negative error code.
 */
int oracle_qli(const oracle_in *in, const int32_t *rows, int32_t nrows,
               int32_t *idx_out, int32_t *cand_out, float *scores,
               int64_t score_stride, int64_t *visible, int32_t nthreads) {
    if (!in || !rows || !idx_out || in->D <= 0 || in->N <= 0) return ORACLE_ERR_ARG;
    if (in->quant_mode != 1 && in->quant_mode != 2) return ORACLE_ERR_ARG;
    if (in->ratio == 1 && in->residual) return ORACLE_ERR_RESIDUAL_WITH_RATIO1;
    if (in->cand_mode == 3 && !in->cand_in) return ORACLE_ERR_CONSUMER_WITHOUT_SOURCE;
    if (in->cand_mode == 2 && !cand_out) return ORACLE_ERR_ARG;
    const int64_t K = in->topk, C = in->cand_blocks;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

    for (int32_t r = 0; r < nrows; ++r) {
        const int32_t t = rows[r];
        int32_t b = 0;                                  /* request of token t */
        while (b + 1 < in->B && in->cu_seqlens_q[b + 1] <= t) ++b;
        const int64_t q_len = in->cu_seqlens_q[b + 1] - in->cu_seqlens_q[b];
        const int64_t i = t - in->cu_seqlens_q[b];
        const int64_t res = in->residual ? in->residual[b] : 0;
        const int64_t V = oracle_visible_count(in->k_lens[b], res, in->ratio, q_len, i);
        if (visible) visible[r] = V;

        /* a5: eligibility. Consumer: visible and inside a given block. */
        const int64_t nb = (V + 7) / 8;
        unsigned char *in_set = NULL;
        if (in->cand_mode == 3) {
            in_set = (unsigned char *)calloc((size_t)(nb > 0 ? nb : 1), 1);
            const int32_t *cr = in->cand_in + (int64_t)t * C;
            for (int64_t c = 0; c < C; ++c)
                if (cr[c] >= 0 && cr[c] < nb) in_set[cr[c]] = 1;
        }

        /* a2-a4: score every visible position */
        float *sc = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < V; ++j) sc[j] = pair_score(in, t, b, j);
        if (scores)
            for (int64_t j = 0; j < V; ++j) scores[(int64_t)r * score_stride + j] = sc[j];

        /* a7 + a8: position TopK over the eligible positions */
        scored *el = (scored *)malloc(sizeof(scored) * (size_t)(V > 0 ? V : 1));
        int64_t E = 0;
        for (int64_t j = 0; j < V; ++j) {
            if (in_set && !in_set[j / 8]) continue;
            el[E].s = sc[j];
            el[E].id = j;
            ++E;
        }
        qsort(el, (size_t)E, sizeof(scored), by_score_then_id);
        emit_ascending(el, E < K ? E : K, idx_out + (int64_t)r * K, K);

        /* a6: source candidates, block score = max visible position score,
         * last visible block pinned, the rest by block score. */
        if (in->cand_mode == 2) {
            int32_t *co = cand_out + (int64_t)r * C;
            if (nb <= C) {
                for (int64_t c = 0; c < C; ++c) co[c] = c < nb ? (int32_t)c : -1;
            } else {
                scored *bl = (scored *)malloc(sizeof(scored) * (size_t)nb);
                for (int64_t k = 0; k + 1 < nb; ++k) {
                    float m = sc[8 * k];
                    for (int64_t j = 8 * k + 1; j < 8 * k + 8 && j < V; ++j)
                        if (sc[j] > m) m = sc[j];
                    bl[k].s = m;
                    bl[k].id = k;
                }
                qsort(bl, (size_t)(nb - 1), sizeof(scored), by_score_then_id);
                bl[C - 1].id = nb - 1;      /* the pinned last visible block */
                bl[C - 1].s = 0.0f;
                emit_ascending(bl, C, co, C);
                free(bl);
            }
        }
        free(el);
        free(sc);
        free(in_set);
    }
    return ORACLE_OK;
}

int oracle_abi_version(void) { return 1; }
