// Host side of the C ABI (include/qli.h): contract validation, workspace
// layout and the sequencing of the three stages. Nothing here allocates,
// frees or synchronises on the run path.
//
// Contract checks follow the guide "DeepSeek V4.1 QLI V2 与候选集成":
//  section 数据流 — TND queries and PA_BBND paged index K only (other layouts
//    are rejected by host validation); residual absent when ratio is 1;
//    a consumer without a source raises;
//  section 当前 A3 契约 — INT8 Q/K with FP16 weights and scales (quant mode 2);
//    section 编译范围 — FP8 (quant mode 1) as the A5 build registers it,
//    32 or 64 heads of dim 128, ratio 1 or 2, causal mask mode 3, TopK in
//    [1, 2048], candidate blocks in [64, 2048] and a multiple of 64, block
//    size exactly 8;
//  section 构建与回归覆盖 — the TND candidate tensor holds T * N_k * blocks
//    elements (T already spans every request; no extra factor of B).
#include <atomic>
#include <cstring>

#include "qli_internal.h"

namespace qli {
namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qli_status validate(const qli_args* a) {
  if (a == nullptr) return QLI_ERR_INVALID_ARG;
  if (a->layout_q != QLI_LAYOUT_TND || a->layout_k != QLI_LAYOUT_PA_BBND) return QLI_ERR_UNSUPPORTED;
  if ((a->quant_mode != QLI_QUANT_INT8 && a->quant_mode != QLI_QUANT_FP8) ||
      a->mask_mode != QLI_MASK_CAUSAL)
    return QLI_ERR_UNSUPPORTED;
  if (a->N != 32 && a->N != 64) return QLI_ERR_UNSUPPORTED;
  if (a->D != kHeadDim) return QLI_ERR_UNSUPPORTED;
  if (a->ratio != 1 && a->ratio != 2) return QLI_ERR_UNSUPPORTED;
  if (a->ratio == 1 && a->residual != nullptr) return QLI_ERR_RESIDUAL_WITH_RATIO1;
  if (a->block_size != kBlock) return QLI_ERR_UNSUPPORTED;
  if (a->rows_per_page != 64 && a->rows_per_page != 128) return QLI_ERR_UNSUPPORTED;
  if (a->cand_mode != QLI_CAND_NONE && a->cand_mode != QLI_CAND_SOURCE &&
      a->cand_mode != QLI_CAND_CONSUMER)
    return QLI_ERR_UNSUPPORTED;
  if (a->topk < 1 || a->topk > kMaxTopK) return QLI_ERR_INVALID_ARG;
  if (a->T < 0 || a->B < 0 || (a->B == 0 && a->T != 0)) return QLI_ERR_INVALID_ARG;
  const int64_t T = a->T, K = a->topk, C = a->cand_blocks;
  if (a->cand_mode != QLI_CAND_NONE) {
    if (C < 64 || C > kMaxCand || C % 64 != 0) return QLI_ERR_INVALID_ARG;
  }
  if (a->cand_mode == QLI_CAND_CONSUMER) {
    if (a->cand_in == nullptr) return QLI_ERR_CONSUMER_WITHOUT_SOURCE;
    if (a->cand_in_numel != T * C) return QLI_ERR_INVALID_ARG;
    if (!aligned(a->cand_in, 4)) return QLI_ERR_ALIGNMENT;
  }
  if (a->cand_mode == QLI_CAND_SOURCE) {
    if (a->cand_out == nullptr || a->cand_out_numel != T * C) return QLI_ERR_INVALID_ARG;
    if (!aligned(a->cand_out, 4)) return QLI_ERR_ALIGNMENT;
  }
  if (a->indices_numel != T * K) return QLI_ERR_INVALID_ARG;
  if (T == 0) return QLI_OK;
  if (a->indices_out == nullptr || a->q == nullptr || a->cu_seqlens_q == nullptr ||
      a->k_lens == nullptr || a->cache == nullptr || a->block_table == nullptr ||
      a->head_weights == nullptr || a->q_scale == nullptr)
    return QLI_ERR_INVALID_ARG;
  if (a->bt_stride < 1 || a->num_pages < 1 || a->page_stride <= 0) return QLI_ERR_INVALID_ARG;
  if (a->q_stride_h < kHeadDim || a->q_stride_t < kHeadDim) return QLI_ERR_INVALID_ARG;
  if (a->k_offset < 0 || a->scale_offset < 0 ||
      a->k_offset + static_cast<int64_t>(a->rows_per_page) * kHeadDim > a->page_stride ||
      a->scale_offset + static_cast<int64_t>(a->rows_per_page) * 2 > a->page_stride)
    return QLI_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || a->q_stride_t % 16 || a->q_stride_h % 16) return QLI_ERR_ALIGNMENT;
  if (!aligned(a->cache, 16) || a->page_stride % 16 || a->k_offset % 16 || a->scale_offset % 16)
    return QLI_ERR_ALIGNMENT;
  if (!aligned(a->cu_seqlens_q, 4) || !aligned(a->k_lens, 4) || !aligned(a->block_table, 4) ||
      !aligned(a->indices_out, 4) || (a->residual && !aligned(a->residual, 4)) ||
      !aligned(a->head_weights, 2) || !aligned(a->q_scale, 2))
    return QLI_ERR_ALIGNMENT;
  return QLI_OK;
}

}  // namespace

// Per device ordinal below 64: 0 = not yet queried, -1 = not an sm_103
// device, otherwise its SM count. Device properties never change within a
// process, so they are queried once.
static std::atomic<int> g_device_sms[64];

qli_status device_sms(int* sms) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QLI_ERR_CUDA;
  int known = (dev >= 0 && dev < 64) ? g_device_sms[dev].load(std::memory_order_relaxed) : 0;
  if (known == 0) {
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&known, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return QLI_ERR_CUDA;
    if (major != 10 || minor != 3) known = -1;
    if (dev >= 0 && dev < 64) g_device_sms[dev].store(known, std::memory_order_relaxed);
  }
  if (known < 0) return QLI_ERR_DEVICE;
  *sms = known;
  return QLI_OK;
}

cudaError_t ensure_smem_limit(const void* func, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}

// Decode-shaped calls (at most two query tokens per request on average) and
// every consumer call take the streaming kernel; prefill-shaped calls take
// the group kernel, which shares each K tile between up to 256/N tokens.
bool use_stream_path(const qli_args& a) {
  return a.cand_mode == QLI_CAND_CONSUMER || static_cast<int64_t>(a.T) <= 2 * static_cast<int64_t>(a.B);
}

WsLayout workspace_layout(const qli_args& a) {
  WsLayout L{};
  const int64_t T = a.T, B = a.B, C = a.cand_blocks;
  const int64_t cap = static_cast<int64_t>(a.bt_stride) * a.rows_per_page;
  L.stream_path = use_stream_path(a) ? 1 : 0;
  L.small = use_small_path(a) ? 1 : 0;
  L.G = L.stream_path ? 1 : kMaxMmaN / (a.N > 0 ? a.N : 64);
  L.Gmax = L.stream_path ? 0 : static_cast<int32_t>((T + L.G - 1) / L.G + B);
  if (a.cand_mode == QLI_CAND_CONSUMER) {
    L.Lrow = C * kBlock;
  } else {
    L.Lrow = static_cast<int64_t>(round_up(static_cast<size_t>(cap), kTile));
  }
  L.Brow = a.cand_mode == QLI_CAND_SOURCE ? L.Lrow / kBlock : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, kAlign);
    return at;
  };
  // err, counter, 8 spare bytes, then (single-launch path) one counter per token
  L.err_bytes = 16 + (L.small ? 4 * static_cast<size_t>(T) : 0);
  L.err = take(L.err_bytes);
  L.counter = L.err + 4;
  L.tok_V = take(4 * T);
  L.tok_b = take(4 * T);
  L.req_lk = take(4 * B);
  L.req_res = take(4 * B);
  L.req_q0 = take(4 * B);
  L.req_q1 = take(4 * B);
  L.req_g0 = take(4 * (B + 1));
  L.grp_t0 = take(4 * static_cast<size_t>(L.Gmax));
  L.grp_cnt = take(4 * static_cast<size_t>(L.Gmax));
  L.unit_start = take(4 * static_cast<size_t>(T + 1));
  const bool cons = a.cand_mode == QLI_CAND_CONSUMER;
  L.cand_list = take(cons ? 4 * T * C : 0);
  L.cand_cnt = take(cons ? 4 * T : 0);
  L.cand_page = take(cons ? 4 * T * C : 0);
  L.cand_sc = take(cons ? 16 * T * C : 0);
  const size_t kstride = round_up(static_cast<size_t>(cap), kTile);
  L.kf16 = take(L.stream_path ? 0 : 2 * kHeadDim * static_cast<size_t>(B) * kstride);
  L.ks32 = take(L.stream_path ? 0 : 4 * static_cast<size_t>(B) * kstride);
  // long-row selection scratch, only when a row can exceed shared memory
  const int64_t longest = L.Lrow > L.Brow ? L.Lrow : L.Brow;
  L.lchunks = longest > kSmemKeys ? static_cast<int32_t>((longest + kLongChunk - 1) / kLongChunk) : 0;
  const size_t rows2 = 2 * static_cast<size_t>(T);
  L.lext = take(L.lchunks ? 16 * rows2 : 0);            // 4 words per row
  L.lhist = take(L.lchunks ? 4 * 4096 * rows2 : 0);
  L.lcount = take(L.lchunks ? 4 * rows2 * L.lchunks : 0);
  L.long_bytes = L.lchunks ? (off - L.lext) : 0;          // zeroed before the passes
  L.lkey = take(L.lchunks ? 4 * rows2 * L.lchunks * kLongChunkCap : 0);
  L.lid = take(L.lchunks ? 4 * rows2 * L.lchunks * kLongChunkCap : 0);
  L.fhist = take(L.stream_path && !L.small ? 4 * 4096 * rows2 : 0);
  L.flist = take(L.stream_path ? 0 : 4 * rows2);
  L.scores = take(4 * static_cast<size_t>(T) * static_cast<size_t>(L.Lrow));
  L.bscores = take(4 * static_cast<size_t>(T) * static_cast<size_t>(L.Brow));
  L.total = off;
  return L;
}

DevArgs make_dev_args(const qli_args& a, void* ws, const WsLayout& L) {
  DevArgs d{};
  uint8_t* w = static_cast<uint8_t*>(ws);
  d.q = a.q;
  d.q_st = a.q_stride_t;
  d.q_sh = a.q_stride_h;
  d.T = a.T;
  d.N = a.N;
  d.B = a.B;
  d.cu = a.cu_seqlens_q;
  d.k_lens = a.k_lens;
  d.residual = a.residual;
  d.cache = a.cache;
  d.page_stride = a.page_stride;
  d.R = a.rows_per_page;
  d.k_off = a.k_offset;
  d.s_off = a.scale_offset;
  d.kfused = a.rows_per_page == kTile && a.scale_offset == a.k_offset + kTile * kHeadDim;
  d.num_pages = a.num_pages;
  d.bt = a.block_table;
  d.bt_stride = a.bt_stride;
  d.w = a.head_weights;
  d.qs = a.q_scale;
  d.ratio = a.ratio;
  d.topk = a.topk;
  d.mode = a.cand_mode;
  d.C = a.cand_blocks;
  d.fp8 = a.quant_mode == QLI_QUANT_FP8 ? 1 : 0;
  d.cand_in = a.cand_in;
  d.cand_out = a.cand_out;
  d.idx_out = a.indices_out;
  d.err = reinterpret_cast<uint32_t*>(w + L.err);
  d.tok_V = reinterpret_cast<int32_t*>(w + L.tok_V);
  d.tok_b = reinterpret_cast<int32_t*>(w + L.tok_b);
  d.req_lk = reinterpret_cast<int32_t*>(w + L.req_lk);
  d.req_res = reinterpret_cast<int32_t*>(w + L.req_res);
  d.req_q0 = reinterpret_cast<int32_t*>(w + L.req_q0);
  d.req_q1 = reinterpret_cast<int32_t*>(w + L.req_q1);
  d.req_g0 = reinterpret_cast<int32_t*>(w + L.req_g0);
  d.grp_t0 = reinterpret_cast<int32_t*>(w + L.grp_t0);
  d.grp_cnt = reinterpret_cast<int32_t*>(w + L.grp_cnt);
  d.unit_start = reinterpret_cast<int32_t*>(w + L.unit_start);
  d.counter = reinterpret_cast<uint32_t*>(w + L.counter);
  d.stream_path = L.stream_path;
  d.lext = reinterpret_cast<uint32_t*>(w + L.lext);
  d.lhist = reinterpret_cast<uint32_t*>(w + L.lhist);
  d.lcount = reinterpret_cast<int32_t*>(w + L.lcount);
  d.lkey = reinterpret_cast<uint32_t*>(w + L.lkey);
  d.lid = reinterpret_cast<int32_t*>(w + L.lid);
  d.lchunks = L.lchunks;
  d.fhist = L.stream_path && !L.small ? reinterpret_cast<uint32_t*>(w + L.fhist) : nullptr;
  d.small = L.small;
  d.done = reinterpret_cast<uint32_t*>(w + L.err + 16);
  d.flist = reinterpret_cast<int32_t*>(w + L.flist);
  d.long_zero_bytes = L.long_bytes;
  d.kf16 = reinterpret_cast<__half*>(w + L.kf16);
  d.ks32 = reinterpret_cast<float*>(w + L.ks32);
  d.kstride = static_cast<int64_t>(round_up(static_cast<size_t>(d.bt_stride) * a.rows_per_page, kTile));
  d.cand_list = reinterpret_cast<int32_t*>(w + L.cand_list);
  d.cand_cnt = reinterpret_cast<int32_t*>(w + L.cand_cnt);
  d.cand_page = reinterpret_cast<int32_t*>(w + L.cand_page);
  d.cand_sc = reinterpret_cast<uint4*>(w + L.cand_sc);
  d.scores = reinterpret_cast<float*>(w + L.scores);
  d.bscores = reinterpret_cast<float*>(w + L.bscores);
  d.Lrow = L.Lrow;
  d.Brow = L.Brow;
  d.Gmax = L.Gmax;
  d.G = L.G;
  d.cap = static_cast<int64_t>(a.bt_stride) * a.rows_per_page;
  return d;
}

namespace {

qli_status run_stages(const qli_args* a, void* ws, size_t bytes, int32_t stage, void* stream) {
  qli_status st = validate(a);
  if (st != QLI_OK) return st;
  if (stage < 0 || stage > QLI_STAGE_SELECT) return QLI_ERR_INVALID_ARG;
  if (a->T == 0) return QLI_OK;
  const WsLayout L = workspace_layout(*a);
  if (ws == nullptr || bytes < L.total) return QLI_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, kAlign)) return QLI_ERR_ALIGNMENT;
  if (L.Gmax > 65535) return QLI_ERR_UNSUPPORTED;
  DevArgs d = make_dev_args(*a, ws, L);
  st = device_sms(&d.num_sms);
  if (st != QLI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (d.small) {
    // planning zeroes the error word and the per-token counters; the score
    // stage's kernel also selects, so the select stage queues nothing
    if (stage == 0 || stage == QLI_STAGE_PLAN) e = launch_small_zero(d, L.err_bytes, s);
    if (e == cudaSuccess && (stage == 0 || stage == QLI_STAGE_SCORE)) e = launch_small(d, s);
    return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
  }
  if (stage == 0 || stage == QLI_STAGE_PLAN) e = launch_plan(d, s);
  if (e == cudaSuccess && (stage == 0 || stage == QLI_STAGE_SCORE)) e = launch_score(d, s);
  if (e == cudaSuccess && (stage == 0 || stage == QLI_STAGE_SELECT)) e = launch_select(d, s);
  return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

}  // namespace
}  // namespace qli

extern "C" {

qli_status qli_validate(const qli_args* a) { return qli::validate(a); }

qli_status qli_workspace_size(const qli_args* a, size_t* bytes) {
  if (bytes == nullptr) return QLI_ERR_INVALID_ARG;
  const qli_status st = qli::validate(a);
  if (st != QLI_OK) return st;
  *bytes = a->T == 0 ? 0 : qli::workspace_layout(*a).total;
  return QLI_OK;
}

qli_status qli_run(const qli_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  return qli::run_stages(a, workspace, workspace_bytes, 0, stream);
}

qli_status qli_run_stage(const qli_args* a, void* workspace, size_t workspace_bytes, int32_t stage,
                         void* stream) {
  if (stage < QLI_STAGE_PLAN || stage > QLI_STAGE_SELECT) return QLI_ERR_INVALID_ARG;
  return qli::run_stages(a, workspace, workspace_bytes, stage, stream);
}

qli_status qli_launch_count(const qli_args* a, int32_t stage, int32_t* launches) {
  if (launches == nullptr) return QLI_ERR_INVALID_ARG;
  const qli_status st = qli::validate(a);
  if (st != QLI_OK) return st;
  if (stage < 0 || stage > QLI_STAGE_SELECT) return QLI_ERR_INVALID_ARG;
  const qli::WsLayout L = qli::workspace_layout(*a);
  const qli::DevArgs d = qli::make_dev_args(*a, nullptr, L);
  int n = 0;
  if (d.small) {
    n = (stage == 0 || stage == QLI_STAGE_PLAN ? 1 : 0) + (stage == 0 || stage == QLI_STAGE_SCORE ? 1 : 0);
  } else {
    if (stage == 0 || stage == QLI_STAGE_PLAN) n += a->T > 0 ? qli::plan_launches(d) : 0;
    if (stage == 0 || stage == QLI_STAGE_SCORE) n += qli::score_launches(d);
    if (stage == 0 || stage == QLI_STAGE_SELECT) n += qli::select_launches(d);
  }
  *launches = n;
  return QLI_OK;
}

qli_status qli_scores_layout(const qli_args* a, size_t* offset, int64_t* row_stride) {
  if (offset == nullptr || row_stride == nullptr) return QLI_ERR_INVALID_ARG;
  const qli_status st = qli::validate(a);
  if (st != QLI_OK) return st;
  const qli::WsLayout L = qli::workspace_layout(*a);
  *offset = L.scores;
  *row_stride = L.Lrow;
  return QLI_OK;
}

qli_status qli_read_device_error(const void* workspace, uint32_t* host_word, void* stream) {
  if (workspace == nullptr || host_word == nullptr) return QLI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_word, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return QLI_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

const char* qli_status_string(qli_status s) {
  switch (s) {
    case QLI_OK: return "ok";
    case QLI_ERR_INVALID_ARG: return "invalid argument";
    case QLI_ERR_UNSUPPORTED: return "unsupported layout, dtype, mode or geometry";
    case QLI_ERR_CONSUMER_WITHOUT_SOURCE: return "consumer mode without source candidates";
    case QLI_ERR_RESIDUAL_WITH_RATIO1: return "residual given with compression ratio 1";
    case QLI_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case QLI_ERR_ALIGNMENT: return "pointer, stride or offset not aligned";
    case QLI_ERR_CUDA: return "CUDA runtime error";
    case QLI_ERR_DEVICE: return "current device is not an sm_103 GPU";
  }
  return "unknown status";
}

int32_t qli_abi_version(void) { return QLI_ABI_VERSION; }

int64_t qli_args_size(void) { return static_cast<int64_t>(sizeof(qli_args)); }

}  // extern "C"
