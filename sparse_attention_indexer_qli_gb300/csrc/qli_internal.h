// Internal declarations shared by the library's translation units: the
// by-value argument block every kernel receives, the workspace layout and the
// stage launchers. Not part of the public ABI (include/qli.h is).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qli.h"

namespace qli {

constexpr int kHeadDim = 128;      // D
constexpr int kTile = 128;         // positions per score tile (MMA M)
constexpr int kBlock = 8;          // positions per candidate block
constexpr int kMaxMmaN = 256;      // token-heads per tile (MMA N)
constexpr int kMaxTopK = 2048;
constexpr int kMaxCand = 2048;
constexpr int kSmemKeys = 44 * 1024;    // keys one selection CTA holds in shared memory
constexpr int kLongChunk = 32768;       // row entries per CTA in the long-row passes
constexpr int kLongChunkCap = 4096;     // candidates kept per chunk
constexpr int kLongCandCap = 16384;     // candidates kept per long row
constexpr int kSmallMaxT = 64;          // single-launch path: tokens,
constexpr int kSmallMaxPositions = 4096;   // and positions a request can hold

// Everything a kernel needs, passed by value (a few hundred bytes).
struct DevArgs {
  // inputs
  const int8_t* q;
  int64_t q_st, q_sh;
  int32_t T, N, B;
  const int32_t* cu;
  const int32_t* k_lens;
  const int32_t* residual;
  const uint8_t* cache;
  int64_t page_stride;
  int32_t R;
  int64_t k_off, s_off, num_pages;
  const int32_t* bt;
  int32_t bt_stride;
  const uint16_t* w;
  const uint16_t* qs;
  int32_t ratio, topk, mode, C;
  int32_t fp8;         // 1: q and the index K hold E4M3 codes (quant mode 1), 0: INT8
  const int32_t* cand_in;
  int32_t* cand_out;
  int32_t* idx_out;
  // workspace views
  uint32_t* err;       // device error word (QLI_DEVERR_*)
  int32_t* tok_V;      // [T] visible compressed positions V(t)
  int32_t* tok_b;      // [T] request of token t, -1 if none
  int32_t* req_lk;     // [B] sanitised compressed length
  int32_t* req_res;    // [B] sanitised residual
  int32_t* req_q0;     // [B] sanitised first token
  int32_t* req_q1;     // [B] sanitised end token
  int32_t* req_g0;     // [B+1] first token group of the request (prefix)
  int32_t* grp_t0;     // [Gmax] first token of a group
  int32_t* grp_cnt;    // [Gmax] tokens in the group (0 = unused)
  int32_t* cand_list;  // [T, C] consumer: sorted distinct usable block IDs
  int32_t* cand_cnt;   // [T] consumer: how many
  int32_t* cand_page;  // [T, C] consumer: the page holding each listed block (checked)
  uint4* cand_sc;      // [T, C] consumer: each listed block's eight FP16 K scales
  int32_t* unit_start; // [T+1] stream path: first score tile of token t; group
                       // path: [Gmax+1] first position tile of group g
  uint32_t* counter;   // consumer: CTAs done in the candidate kernel; group path: rows
                       // listed in flist (reset by plan)
  int32_t* flist;      // group path: [2T] rows (2t + which) left to the general selection
  __half* kf16;        // group path: [B, kstride, 128] widened K
  float* ks32;         // group path: [B, kstride] K scales as FP32
  int64_t kstride;     // group path: rows per request (cap rounded up to 128)
  // long rows (longer than the keys one CTA holds in shared memory): row
  // r = 2t (positions) or 2t+1 (source blocks)
  uint32_t* lext;      // [2T, 4] max key, max complemented key, eligible count, unused
  uint32_t* lhist;     // [2T, 4096] digit histogram below the row's common prefix
  int32_t* lcount;     // [2T, lchunks] candidates found per chunk
  uint32_t* lkey;      // [2T, lchunks, kLongChunkCap] candidate keys, position order
  int32_t* lid;        // [2T, lchunks, kLongChunkCap] candidate ids
  int32_t lchunks;     // chunks per long row (0: no row is long)
  size_t long_zero_bytes;  // bytes from lext that start each call at zero
  uint32_t* fhist;     // stream path: [2T, 4096] counts of the top 12 key bits of
                       // row 2t (positions) and 2t+1 (source blocks), built by the
                       // score stage; nullptr on the group path
  float* scores;       // [T, Lrow]
  float* bscores;      // [T, Brow] source: block maxima
  int64_t Lrow, Brow;
  int32_t Gmax, G;     // token groups (upper bound), tokens per group
  int64_t cap;         // bt_stride * R: most positions a request can hold
  int32_t stream_path; // 1: one token per tile, persistent streaming kernel
  int32_t num_sms;     // SMs of the device (persistent grids)
  int32_t small;       // 1: the single-launch path (planning, scoring, selection in one kernel)
  uint32_t* done;      // single-launch path: [T] CTAs of the token done (zeroed with err)
  int32_t kfused;      // 1: 128-row pages whose FP16 scales follow the index-K rows
                       // (s_off == k_off + 128*128): one copy brings both
};

struct WsLayout {
  size_t err, counter, tok_V, tok_b, req_lk, req_res, req_q0, req_q1, req_g0;
  size_t grp_t0, grp_cnt, unit_start, cand_list, cand_cnt, cand_page, cand_sc, kf16, ks32, scores,
      bscores, flist, total;
  size_t lext, lhist, lcount, lkey, lid, long_bytes;   // long-row selection (zeroed region: lext..lcount)
  size_t fhist;
  int32_t lchunks;
  int64_t Lrow, Brow;
  int32_t Gmax, G;
  int32_t stream_path;
  int32_t small;
  size_t err_bytes;    // err, counter and (single-launch path) the per-token counters
};

// The streaming (decode) kernel takes one token per tile; the group kernel
// shares a tile between up to 256/N tokens of one request (prefill).
bool use_stream_path(const qli_args& a);

// Small decode batches (INT8, none/source, at most kSmallMaxT tokens and 64
// requests, at most kSmallMaxPositions positions per request) run planning,
// scoring and selection in one kernel, after a one-CTA kernel that zeroes the
// first `bytes` of the workspace (the error word and the per-token counters).
bool use_small_path(const qli_args& a);
cudaError_t launch_small_zero(const DevArgs& d, size_t bytes, cudaStream_t s);
cudaError_t launch_small(const DevArgs& d, cudaStream_t s);

// Raises `func`'s dynamic shared-memory limit to `bytes` once per device
// (`done` holds one bit per device ordinal below 64; others always set it).
cudaError_t ensure_smem_limit(const void* func, int bytes, std::atomic<uint64_t>& done);

// Launches `kernel` with programmatic stream serialisation: it may begin
// while the previous kernel on the stream finishes, and must call pdl_wait()
// before reading that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// QLI_OK and the current device's SM count if it is an sm_103 GPU,
// QLI_ERR_DEVICE otherwise (QLI_ERR_CUDA if the runtime fails).
qli_status device_sms(int* sms);

WsLayout workspace_layout(const qli_args& a);
DevArgs make_dev_args(const qli_args& a, void* ws, const WsLayout& L);

// Stage launchers (one .cu file each). Return the first CUDA error.
cudaError_t launch_plan(const DevArgs& d, cudaStream_t s);
cudaError_t launch_score(const DevArgs& d, cudaStream_t s);
cudaError_t launch_select(const DevArgs& d, cudaStream_t s);
cudaError_t launch_prefill(const DevArgs& d, cudaStream_t s);
int prefill_launches(const DevArgs& d);
int plan_launches(const DevArgs& d);
int score_launches(const DevArgs& d);
int select_launches(const DevArgs& d);

}  // namespace qli
