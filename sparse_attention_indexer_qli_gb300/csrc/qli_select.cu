// Selection stage: per query token, the position TopK and (source mode) the
// candidate blocks, both emitted in ascending order and padded with -1.
//
// Guide "DeepSeek V4.1 QLI V2 与候选集成", section 数据流: candidates are
// [tokens, 1, blocks] INT32 block IDs padded with -1; a block holds 8
// compressed positions and scores as the max of its positions' scores; the
// last visible block is always kept; position indices are put in
// chronological order with the -1 padding at the end; an empty context gives
// empty indices and all-invalid candidates. Section 当前 A3 契约: TopK in
// [1, 2048], candidate blocks in [64, 2048].
//
// Ranking reading: higher score first, equal scores (with -0 == +0) by the
// lower position / block ID. The selected entries are found with an exact
// 4-pass radix select over order-preserving 32-bit keys, then written in
// position order by one ordered pass, so no sort is needed. Rows that fit
// are first copied into shared memory as keys, so the passes never go back
// to L2; longer rows are read from L2 on every pass.
#include <cuda_fp16.h>

#include "qli_internal.h"

namespace qli {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemKeys = 48 * 1024;          // keys cached per row (192 KB)

// Order-preserving map of a finite FP32 score to a non-zero uint32 key
// (larger score -> larger key; -0 and +0 map to the same key). Key 0 is kept
// for "not eligible".
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0) u = 0;   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Shared {
  uint32_t hist[256];
  int warp_cnt[kWarps];
  uint32_t sel[2];
};

// Exclusive count of set flags before this thread over the whole CTA, and
// the CTA total. Every thread must call it.
__device__ __forceinline__ int cta_excl_count(bool f, Shared& sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned m = __ballot_sync(0xffffffffu, f);
  if (lane == 0) sh.warp_cnt[warp] = __popc(m);
  __syncthreads();
  int base = 0;
  total = 0;
#pragma unroll 8
  for (int w = 0; w < kWarps; ++w) {
    const int c = sh.warp_cnt[w];
    base += (w < warp) ? c : 0;
    total += c;
  }
  __syncthreads();
  return base + __popc(m & ((1u << lane) - 1u));
}

__device__ __forceinline__ int cta_sum(int v, Shared& sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sh.warp_cnt[threadIdx.x >> 5] = v;
  __syncthreads();
  int s = 0;
  for (int w = 0; w < kWarps; ++w) s += sh.warp_cnt[w];
  __syncthreads();
  return s;
}

// A row of the selection: entry s has a key (0 = not eligible) and an id.
struct Row {
  const float* vals;      // score row
  const int32_t* blocks;  // consumer: sorted candidate blocks (slot -> position)
  const uint32_t* cached; // keys in shared memory, or nullptr
  int32_t len;            // entries in the row
  int32_t V;              // visible positions of the token
  bool consumer;

  __device__ __forceinline__ uint32_t key_from_global(int32_t s) const {
    if (consumer) {
      const int32_t pos = blocks[s / kBlock] * kBlock + (s & (kBlock - 1));
      if (pos >= V) return 0u;
    }
    return order_key(vals[s]);
  }
  __device__ __forceinline__ uint32_t key(int32_t s) const {
    return cached ? cached[s] : key_from_global(s);
  }
  __device__ __forceinline__ int32_t id(int32_t s) const {
    return consumer ? blocks[s / kBlock] * kBlock + (s & (kBlock - 1)) : s;
  }
};

// Histogram add with one shared atomic per distinct bin within the warp
// (scores concentrate in few bins; plain atomics would serialise).
__device__ __forceinline__ void hist_add(uint32_t* hist, bool valid, uint32_t bin) {
  const uint32_t probe = valid ? bin : 0x10000u + (threadIdx.x & 31);
  const unsigned same = __match_any_sync(0xffffffffu, probe);
  if (valid && (__ffs(same) - 1) == static_cast<int>(threadIdx.x & 31))
    atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(same)));
}

// Writes the ids of the `want` best entries of `r` in ascending id order to
// out[0..), and returns how many were written (min(want, eligible)).
__device__ int select_ascending(const Row& r, int32_t want, int32_t* out, Shared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int local = 0;
  for (int32_t s = tid; s < r.len; s += kThreads) local += r.key(s) != 0u ? 1 : 0;
  const int E = cta_sum(local, sh);

  uint32_t thr = 0u;        // select keys > thr, plus `need_eq` keys == thr
  int32_t need_eq = 0;
  if (E > want) {
    uint32_t prefix = 0u, mask = 0u;
    int32_t k = want;       // rank (1-based) of the threshold among the remaining
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) sh.hist[tid] = 0u;
      __syncthreads();
      const int32_t rounds = (r.len + kThreads - 1) / kThreads;
      for (int32_t i = 0; i < rounds; ++i) {
        const int32_t s = i * kThreads + tid;
        const uint32_t key = s < r.len ? r.key(s) : 0u;
        const bool v = key != 0u && (key & mask) == prefix;
        hist_add(sh.hist, v, (key >> shift) & 255u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255-8l .. 248-8l; find the bin holding rank k
        uint32_t c[8];
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = sh.hist[255 - 8 * lane - j];
          mine += c[j];
        }
        uint32_t incl = mine;
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        uint32_t above = incl - mine;
        if (above < static_cast<uint32_t>(k) && static_cast<uint32_t>(k) <= incl) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (above + c[j] >= static_cast<uint32_t>(k)) {
              sh.sel[0] = 255u - 8u * lane - j;
              sh.sel[1] = static_cast<uint32_t>(k) - above;
              break;
            }
            above += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= sh.sel[0] << shift;
      mask |= 255u << shift;
      k = static_cast<int32_t>(sh.sel[1]);
      __syncthreads();
    }
    thr = prefix;           // the exact key of the want-th best entry
    need_eq = k;            // how many entries equal to it are taken
  }

  // ordered pass: ids with key > thr, and the first need_eq with key == thr
  int32_t written = 0, eq_seen = 0;
  for (int32_t base = 0; base < r.len; base += kThreads) {
    const int32_t s = base + tid;
    const uint32_t key = s < r.len ? r.key(s) : 0u;
    const bool sel_gt = key != 0u && key > thr;
    bool sel = sel_gt;
    if (need_eq > 0) {
      const bool eq = key != 0u && key == thr;
      int eq_total;
      const int eq_rank = cta_excl_count(eq, sh, eq_total);
      sel = sel_gt || (eq && eq_seen + eq_rank < need_eq);
      eq_seen += eq_total;
    }
    int sel_total;
    const int at = cta_excl_count(sel, sh, sel_total);
    if (sel) out[written + at] = r.id(s);
    written += sel_total;
  }
  return written;
}

// Copies the row's keys into shared memory (when it fits) and points the
// row at them.
__device__ void cache_keys(Row& r, uint32_t* keys, int32_t cap) {
  if (r.len > cap) return;
  for (int32_t s = threadIdx.x; s < r.len; s += kThreads) keys[s] = r.key_from_global(s);
  __syncthreads();
  r.cached = keys;
}

// grid.x = token, grid.y = 0: position TopK, 1: source candidate blocks.
__global__ void __launch_bounds__(kThreads) select_kernel(DevArgs a, int32_t key_cap) {
  extern __shared__ uint32_t keys[];
  __shared__ Shared sh;
  const int t = blockIdx.x, which = blockIdx.y, tid = threadIdx.x;
  const bool blocks = which == 1;
  const int32_t width = blocks ? a.C : a.topk;
  int32_t* out = blocks ? a.cand_out + static_cast<int64_t>(t) * a.C
                        : a.idx_out + static_cast<int64_t>(t) * a.topk;
  int32_t written = 0;
  const int32_t V = a.tok_b[t] >= 0 ? a.tok_V[t] : 0;

  Row r;
  r.V = V;
  r.cached = nullptr;
  if (!blocks) {
    r.consumer = a.mode == QLI_CAND_CONSUMER;
    r.vals = a.scores + static_cast<int64_t>(t) * a.Lrow;
    r.blocks = r.consumer ? a.cand_list + static_cast<int64_t>(t) * a.C : nullptr;
    r.len = r.consumer ? (a.tok_b[t] >= 0 ? a.cand_cnt[t] * kBlock : 0) : V;
    cache_keys(r, keys, key_cap);
    written = select_ascending(r, a.topk, out, sh);
  } else {
    const int32_t nb = (V + kBlock - 1) / kBlock;
    if (nb <= a.C) {
      for (int c = tid; c < nb; c += kThreads) out[c] = c;
      written = nb;
    } else {
      // the best C-1 of blocks 0..nb-2, then the pinned last visible block
      r.consumer = false;
      r.vals = a.bscores + static_cast<int64_t>(t) * a.Brow;
      r.blocks = nullptr;
      r.len = nb - 1;
      cache_keys(r, keys, key_cap);
      written = select_ascending(r, a.C - 1, out, sh);
      if (tid == 0) out[written] = nb - 1;
      written += 1;
    }
  }
  for (int k = written + tid; k < width; k += kThreads) out[k] = -1;
}

}  // namespace

cudaError_t launch_select(const DevArgs& d, cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  const int64_t longest = d.Lrow > d.Brow ? d.Lrow : d.Brow;
  const int32_t cap = static_cast<int32_t>(longest < kSmemKeys ? longest : kSmemKeys);
  const int smem = cap * 4;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(d.T), d.mode == QLI_CAND_SOURCE ? 2u : 1u);
  select_kernel<<<grid, kThreads, smem, s>>>(d, cap);
  return cudaGetLastError();
}

int select_launches(const DevArgs& d) { return d.T > 0 ? 1 : 0; }

}  // namespace qli
