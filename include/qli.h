/*
 * qli.h — C ABI of the GB300 quantized lightning indexer (QLI).
 *
 * The indexer scores every causally visible compressed position of a paged
 * INT8 index-K cache against per-head INT8 queries and returns, per query
 * token, the chronologically ordered position TopK and, in source mode, the
 * 8-position candidate block IDs. It is the operator the vllm-ascend
 * developer guide "DeepSeek V4.1 QLI V2 与候选集成" documents:
 *   section "数据流" (data flow)      — inputs, page geometry, metadata,
 *                                        the three candidate modes, outputs;
 *   section "当前 A3 契约" (contract)  — dtypes, ranges and the numeric golden;
 *   section "构建与回归覆盖"           — candidate size T * N_k * blocks.
 *
 * Conventions
 *  - Every pointer inside qli_args is a DEVICE pointer (memory of the current
 *    CUDA device, sm_103a) unless stated otherwise. The library never
 *    allocates, frees or synchronises on the run path; the caller owns every
 *    buffer, including the workspace, and keeps it alive until the work
 *    queued on `stream` has finished.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Validation runs on the host before anything is queued; a non-OK status
 *    means nothing was launched. Values that live on the device (lengths,
 *    block-table entries) are checked by the first kernel: out-of-range values
 *    are clamped so that no access leaves its buffer, and a bit is set in the
 *    workspace's error word (qli_read_device_error).
 *  - No state is kept between calls. Candidates produced by a source call
 *    reach a later consumer call only through the caller's buffer.
 *  - Every FP16 value is IEEE binary16 passed as its 16-bit pattern.
 */
#ifndef QLI_H
#define QLI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QLI_ABI_VERSION 1

typedef enum qli_status {
    QLI_OK = 0,
    QLI_ERR_INVALID_ARG = 1,          /* NULL pointer, bad size or extent */
    QLI_ERR_UNSUPPORTED = 2,          /* layout, dtype, quant/mask mode, N, D, ratio,
                                         block size or page geometry outside the contract */
    QLI_ERR_CONSUMER_WITHOUT_SOURCE = 3, /* consumer mode with no candidate input */
    QLI_ERR_RESIDUAL_WITH_RATIO1 = 4, /* a residual tensor was given with ratio 1 */
    QLI_ERR_WORKSPACE_TOO_SMALL = 5,
    QLI_ERR_ALIGNMENT = 6,            /* pointer, stride or offset not 16-byte aligned */
    QLI_ERR_CUDA = 7,                 /* a CUDA runtime call failed */
    QLI_ERR_DEVICE = 8                /* current device is not an sm_103 GPU */
} qli_status;

/* Candidate modes. The guide numbers them 1/2/3 ("候选模式 1/2/3") without
 * naming them in the surviving text; this library reads 1 = none (position
 * TopK only), 2 = source (also emits candidate blocks), 3 = consumer (TopK
 * restricted to given candidate blocks). */
enum { QLI_CAND_NONE = 1, QLI_CAND_SOURCE = 2, QLI_CAND_CONSUMER = 3 };
/* Layouts, quantisation and mask modes the contract compiles. */
enum { QLI_LAYOUT_TND = 1, QLI_LAYOUT_PA_BBND = 2 };
enum { QLI_QUANT_INT8 = 2 };          /* quant mode 2: INT8 Q/K, FP16 weights/scales */
/* Quant mode 1: FP8. The guide's section "编译范围" names FP8 as quant mode 1
 * of the A5 build and prints no FP8 golden; this library reads it as the
 * same layout and chain with E4M3 codes ("fn": bias 7, largest 448, no
 * infinities) in place of the INT8 values: q and the index-K rows hold one
 * code per byte, the dot of the decoded codes (rounded to FP32) takes the
 * INT32 dot's place, and the chain from the division by 1024 on is
 * unchanged. The sums are the tensor core's FP32 ones, so a score can differ
 * from the exactly rounded dot's by the rounding of those sums (a few FP32
 * ulps of each head's dot before its FP16 rounding). */
enum { QLI_QUANT_FP8 = 1 };
enum { QLI_MASK_CAUSAL = 3 };         /* causal mask mode 3 */
/* Stages of one call, for timing them separately (qli_run_stage). */
enum { QLI_STAGE_PLAN = 1, QLI_STAGE_SCORE = 2, QLI_STAGE_SELECT = 3 };
/* Bits of the device error word. */
enum {
    QLI_DEVERR_SEQLENS = 1u << 0,     /* cu_seqlens_q not 0..T non-decreasing */
    QLI_DEVERR_KLEN = 1u << 1,        /* k_lens outside [0, bt_stride*rows_per_page] */
    QLI_DEVERR_RESIDUAL = 1u << 2,    /* residual outside [0, ratio) */
    QLI_DEVERR_PAGE = 1u << 3,        /* block-table entry outside [0, num_pages) */
    QLI_DEVERR_TIMEOUT = 1u << 4      /* an on-chip wait gave up (never expected) */
};

typedef struct qli_args {
    /* Queries, TND: element (t, h, d) at q[t*q_stride_t + h*q_stride_h + d],
     * INT8 (E4M3 codes in quant mode 1), strides in bytes, each a multiple
     * of 16 with q_stride_h >= D. */
    const int8_t *q;
    int64_t q_stride_t, q_stride_h;
    int32_t T;                        /* query tokens (all requests)            */
    int32_t N;                        /* index heads: 32 or 64                  */
    int32_t D;                        /* head dim: 128                          */
    /* Metadata ("数据流"): raw query boundaries, compressed K lengths, raw
     * length mod ratio. Device int32 arrays. */
    const int32_t *cu_seqlens_q;      /* [B+1], 0 = cu[0] <= ... <= cu[B] = T   */
    int32_t B;                        /* requests                               */
    const int32_t *k_lens;            /* [B] compressed positions per request   */
    const int32_t *residual;          /* [B] raw length mod ratio; must be NULL
                                         when ratio == 1, NULL means 0 otherwise */
    /* PA_BBND paged index K: page p starts at cache + p*page_stride; row r of
     * the page holds position (slot*rows_per_page + r) of the request whose
     * block table lists p at `slot`; its 128 INT8 values sit at
     * k_offset + r*128 and its FP16 scale at scale_offset + r*2 inside the page. */
    const uint8_t *cache;
    int64_t page_stride;              /* bytes; 131072 (ratio 2) / 147712 (ratio 1) */
    int32_t rows_per_page;            /* 64 or 128                              */
    int64_t k_offset, scale_offset;   /* bytes inside a page                    */
    int64_t num_pages;                /* pages in the pool (bounds checks)       */
    const int32_t *block_table;       /* [B, bt_stride] page IDs                 */
    int32_t bt_stride;                /* >= pages of the longest request        */
    /* FP16 head weights and per-head Q scales, [T, N] contiguous. */
    const uint16_t *head_weights;
    const uint16_t *q_scale;
    int32_t ratio;                    /* compression ratio: 1 or 2              */
    int32_t mask_mode;                /* QLI_MASK_CAUSAL                        */
    int32_t quant_mode;               /* QLI_QUANT_INT8 or QLI_QUANT_FP8        */
    int32_t layout_q;                 /* QLI_LAYOUT_TND                         */
    int32_t layout_k;                 /* QLI_LAYOUT_PA_BBND                     */
    int32_t topk;                     /* K in [1, 2048]                         */
    int32_t cand_mode;                /* QLI_CAND_*                             */
    int32_t cand_blocks;              /* C in [64, 2048], multiple of 64 (source/consumer) */
    int32_t block_size;               /* positions per candidate block: 8      */
    const int32_t *cand_in;           /* consumer: [T, 1, C] block IDs, -1 pads  */
    int64_t cand_in_numel;            /* must equal T * 1 * C in consumer mode  */
    int32_t *cand_out;                /* source: [T, 1, C] block IDs, -1 padded  */
    int64_t cand_out_numel;           /* must equal T * 1 * C in source mode    */
    int32_t *indices_out;             /* [T, 1, K] positions, ascending, -1 at the end */
    int64_t indices_numel;            /* must equal T * K                       */
} qli_args;

/* Checks `a` against the contract ("当前 A3 契约", "数据流", "构建与回归覆盖")
 * on the host. Touches no device memory. */
qli_status qli_validate(const qli_args *a);

/* Bytes of device workspace qli_run needs for these arguments (an upper bound
 * derived from T, B, N, bt_stride*rows_per_page and C; no device reads). */
qli_status qli_workspace_size(const qli_args *a, size_t *bytes);

/* Queues the whole indexer on `stream`: planning, scoring, selection. Writes
 * indices_out and, in source mode, cand_out. `workspace` must be 256-byte
 * aligned device memory of at least qli_workspace_size bytes; its contents on
 * entry do not matter. Asynchronous: returns once the kernels are queued. */
qli_status qli_run(const qli_args *a, void *workspace, size_t workspace_bytes, void *stream);

/* Queues one stage (QLI_STAGE_*) of qli_run, for timing. Running PLAN, SCORE
 * and SELECT in that order on one stream equals qli_run. Small decode batches
 * (INT8, none or source mode, T <= 64, B <= 64, bt_stride*rows_per_page <=
 * 4096) run planning, scoring and selection in the SCORE stage's one kernel:
 * their PLAN stage only zeroes the error word and per-token counters, and
 * their SELECT stage queues nothing. */
qli_status qli_run_stage(const qli_args *a, void *workspace, size_t workspace_bytes,
                         int32_t stage, void *stream);

/* Kernel launches one call of the given stage queues (0 = all stages). */
qli_status qli_launch_count(const qli_args *a, int32_t stage, int32_t *launches);

/* Where the FP32 scores sit in the workspace after the SCORE stage: row t
 * starts at byte `offset` + t*row_stride*4. In none/source mode entry j of
 * row t is the score of position j (valid for j < V(t)); in consumer mode
 * entry s is the score of the s-th position of the token's sorted candidate
 * blocks. For tests; the values are not part of the operator's outputs. */
qli_status qli_scores_layout(const qli_args *a, size_t *offset, int64_t *row_stride);

/* Copies the device error word (QLI_DEVERR_* bits of the last call that used
 * this workspace) to *host_word and waits for `stream`. Synchronous. */
qli_status qli_read_device_error(const void *workspace, uint32_t *host_word, void *stream);

/* Bytes of the fixed device scratch array qli_run_static uses. */
#define QLI_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Same result as qli_run, for callers that cannot allocate device memory at
 * call time (for example a serving engine whose device memory is all handed
 * to its KV-cache pool at start-up, or a C program with no device allocator).
 * The pages describe no counterpart of this entry point; it is a property of
 * this library only.
 * Instead of a caller workspace it uses one array of QLI_STATIC_SCRATCH_BYTES
 * compiled into the library, held on every GPU that loads the library until
 * the process exits. Nothing is allocated or freed. The array's device
 * address is looked up on the first call made on each device, with that
 * device current; make that first call before any stream capture begins.
 * Calls whose workspace need (qli_workspace_size) exceeds the array return
 * QLI_ERR_WORKSPACE_TOO_SMALL without launching anything. All calls share the
 * array and it keeps the previous call's contents (none of them has to start
 * at zero); calls that overlap on the GPU race on it, so issue them in order
 * on one stream. Inputs, outputs, stream and host-side errors are as for
 * qli_run; the device error word is read with qli_read_static_device_error. */
qli_status qli_run_static(const qli_args *a, void *stream);

/* The device error word (QLI_DEVERR_* bits) of the last qli_run_static call
 * on the current device, copied to *host_word after waiting for `stream`.
 * Synchronous; allocates nothing. The next qli_run_static call on the device
 * resets the word, so read it before issuing another. */
qli_status qli_read_static_device_error(uint32_t *host_word, void *stream);

/* ---- Query quantiser and index-K cache writer -------------------------------
 * The two steps either side of the indexer's paged gather. The guide's
 * section "数据流" (data flow): the indexer's projected queries are quantised
 * per head to INT8, each head with a scale representable in FP16; head
 * weights and K scales are FP16; the page allocator packs the index K and
 * its FP16 scales after the KV inside each page.
 *
 * One row x of D = 128 BF16 values (passed as 16-bit patterns) becomes 128
 * INT8 codes and one FP16 scale:
 *     amax = max_d |x_d|
 *     s    = FP16(amax / 127)   FP32 quotient, then round to nearest even;
 *                               capped at 65504
 *     q_d  = clamp(rint(x_d / s), -127, 127)   FP32 quotient, ties to even
 * A row whose s rounds to zero (amax below 127 * 2^-25, e.g. all zeros)
 * gets codes 0 and scale +0. Inf and NaN inputs are outside the contract
 * (their codes are unspecified; nothing is read or written out of bounds).
 * The pages do not spell the formula out; this is the plain symmetric
 * absmax reading of "INT8 with a representable FP16 scale": the stored FP16
 * value is the one divided by, so q * s is the dequantised value. */

/* Quantises `rows` rows of 128 BF16 values, contiguous at x (16-byte
 * aligned), to codes q_out [rows, 128] (16-byte aligned) and FP16 scales
 * scale_out [rows] (2-byte aligned). For the indexer's queries, rows = T * N
 * and x is [T, N, 128]: q_out is then the TND q (q_stride_t = N * 128,
 * q_stride_h = 128) and scale_out the [T, N] q_scale. Device pointers; one
 * kernel on `stream`; asynchronous. rows = 0 launches nothing. */
qli_status qli_quantize_q(const uint16_t *x, int64_t rows, int8_t *q_out, uint16_t *scale_out,
                          void *stream);

/* Quantises n new index-K rows (k: [n, 128] BF16, 16-byte aligned) and
 * writes row i into the PA_BBND page pool `cache` at slot_mapping[i] =
 * page * rows_per_page + row: codes at cache + page * page_stride +
 * k_offset + row * 128, FP16 scale at cache + page * page_stride +
 * scale_offset + row * 2 (the layout qli_run reads). A negative slot is
 * padding: nothing is written. A slot at or past num_pages * rows_per_page
 * is skipped and, when err_word is not NULL, sets QLI_DEVERR_PAGE in that
 * device word (OR'ed in; the caller clears it). The slots of one call must
 * be distinct. cache, page_stride and k_offset must be multiples of 16 bytes
 * and scale_offset of 2; rows_per_page is 64 or 128 and k_offset +
 * rows_per_page * 128 and scale_offset + rows_per_page * 2 must fit in a
 * page. Device pointers; one kernel on `stream`; asynchronous. */
qli_status qli_write_index_k(const uint16_t *k, int64_t n, const int64_t *slot_mapping,
                             uint8_t *cache, int64_t num_pages, int64_t page_stride,
                             int32_t rows_per_page, int64_t k_offset, int64_t scale_offset,
                             uint32_t *err_word, void *stream);

/* The FP8 variant of the two calls above (quant mode 1, which the guide's
 * section 编译范围 names for the A5 build; the pages give no formula). The
 * same per-row scheme with E4M3's largest finite value 448 in place of 127:
 *     s   = FP16(amax / 448)   FP32 quotient, round to nearest even; capped
 *                              at 65504
 *     c_d = E4M3(x_d / s)      FP32 quotient, rounded to nearest even on the
 *                              E4M3 grid ("fn" encoding: bias 7, no
 *                              infinities), saturated to +-448
 * A row whose s rounds to zero gets codes 0 and scale +0. Codes are E4M3 bit
 * patterns in the bytes the INT8 calls would write, so qli_run with
 * quant_mode = QLI_QUANT_FP8 reads them. Arguments, layouts, alignment and
 * errors as for qli_quantize_q and qli_write_index_k. */
qli_status qli_quantize_q_fp8(const uint16_t *x, int64_t rows, uint8_t *q_out,
                              uint16_t *scale_out, void *stream);
qli_status qli_write_index_k_fp8(const uint16_t *k, int64_t n, const int64_t *slot_mapping,
                                 uint8_t *cache, int64_t num_pages, int64_t page_stride,
                                 int32_t rows_per_page, int64_t k_offset, int64_t scale_offset,
                                 uint32_t *err_word, void *stream);

/* Self-check of the quantisers' divisions, which compute x / s, amax / 127
 * and amax / 448 from the row's reciprocal with one correction step instead
 * of an IEEE divide (Markstein, IBM J. Res. Dev. 34(1), 1990). Both operands
 * come from finite sets (x a BF16 value, s a positive finite FP16 scale), so
 * one kernel on `stream` tries every pair a row can produce: all s with
 * |x| <= 768 s (a row's amax / s stays below 1.5 x 127 or 1.5 x 448 unless
 * s is the 65504 cap) and every finite x for s = 65504; codes are compared
 * for both the INT8 and the E4M3 encoding. It leaves in the device array
 * counts[2] (8-byte aligned; zeroed by the call): counts[0] = pairs whose
 * INT8 code clamp(rint(x / s), -127, 127) or E4M3 code differs from the one
 * an IEEE FP32 division gives, plus the BF16 values amax >= 0 whose scale
 * FP16(amax / 127) or FP16(amax / 448) (computed the same way) differs from
 * the IEEE one; counts[1] = pairs with |x| >= 2^-100 whose FP32 quotient
 * differs from the IEEE one (below that the correction's residual can
 * underflow; those quotients round to code 0 either way). Asynchronous. */
qli_status qli_check_quant_rounding(unsigned long long *counts, void *stream);

/* ---- Sparse attention over the selected positions ---------------------------
 * The stage that consumes the indexer's output: blog "DeepSeek V4.1-Flash
 * 登陆昇腾 · 需求故事（PR 16925）", section 四 (the attention forward passes the
 * compressed indices to the sparse attention, then inverse-rotates the output
 * tail in place); guide "DeepSeek V4.1 QLI V2 与候选集成", section 编译范围
 * (BF16 TND queries over the PA_BBND paged cache, one KV head); section 数据流
 * (each page row holds the KV row first, then the index K and its scale).
 * Readings where the pages are silent: the KV row of a compressed position is
 * 512 BF16 values (1024 bytes) at kv_offset + row * 1024 of its page and is
 * both key and value; the softmax scale is an argument; the sliding-window
 * stage and the sinks are not described on the pages and are not part of
 * this call (the LSE output is what combining with another stage needs).
 * For token t of request b (cu_seqlens_q), head h, and the listed positions
 * J = { indices[t, 0, k] >= 0 } (a position listed twice counts twice):
 *     s_j = scale * sum_d q[t, h, d] * kv_j[d]
 *     out[t, h, :] = BF16( sum_j exp(s_j - m) kv_j / sum_j exp(s_j - m) ),
 *     lse[t, h] = m + ln(sum_j exp(s_j - m)),    m = max_j s_j;
 * an empty J gives out = 0 and lse = -inf. BF16 products are exact; sums are
 * FP32 on the tensor cores, the weights are rounded to BF16 for the value
 * product, so results agree with the exact definition to about 2^-8
 * relative to the largest selected value. */
typedef struct qli_attn_args {
    const uint16_t *q;           /* BF16 [T, H, 512]: (t, h, d) at q[t*q_stride_t + h*q_stride_h + d]
                                    (strides in elements, multiples of 8; d contiguous) */
    int64_t q_stride_t, q_stride_h;
    int32_t T;                   /* query tokens */
    int32_t H;                   /* query heads: 32, 64, 96 or 128 */
    int32_t D;                   /* values per KV row: 512 */
    const int32_t *cu_seqlens_q; /* [B+1] raw query boundaries (token t belongs to the
                                    last request b with cu_seqlens_q[b] <= t) */
    int32_t B;
    const uint8_t *cache;        /* the page pool of the indexer (qli_args.cache) */
    int64_t page_stride;         /* bytes, multiple of 16 */
    int64_t num_pages;
    int32_t rows_per_page;       /* 64 or 128 */
    int64_t kv_offset;           /* bytes from a page's start to row 0's KV values (multiple of 16) */
    const int32_t *block_table;  /* [B, bt_stride] page IDs */
    int32_t bt_stride;
    const int32_t *indices;      /* [T, 1, K] compressed positions (the indexer's output); -1 skipped */
    int32_t K;                   /* entries per token: 1..2048 */
    float scale;                 /* softmax scale (finite) */
    uint16_t *out;               /* BF16 [T, H, 512]: (t, h, d) at out[t*out_stride_t + h*out_stride_h + d] */
    int64_t out_stride_t, out_stride_h;
    float *lse;                  /* [T, H] natural-log LSE, or NULL */
    uint32_t *err_word;          /* device word: QLI_DEVERR_PAGE is OR'ed in when a listed
                                    position lies past the block table or names a page outside
                                    the pool (that entry is skipped), QLI_DEVERR_TIMEOUT when an
                                    on-chip wait gives up; may be NULL; the caller clears it */
} qli_attn_args;

/* Queues the sparse attention on `stream` (one kernel; no workspace: every
 * intermediate stays on chip). Device pointers; asynchronous. Host-side
 * checks as for qli_run (nothing is launched on a non-OK status). */
qli_status qli_sparse_attention(const qli_attn_args *a, void *stream);

/* sizeof(qli_attn_args) the library was built with. */
int64_t qli_attn_args_size(void);

/* Human-readable name of a status. Never NULL. */
const char *qli_status_string(qli_status s);

/* QLI_ABI_VERSION of the loaded library, and sizeof(qli_args) it was built with. */
int32_t qli_abi_version(void);
int64_t qli_args_size(void);

#ifdef __cplusplus
}
#endif
#endif /* QLI_H */
