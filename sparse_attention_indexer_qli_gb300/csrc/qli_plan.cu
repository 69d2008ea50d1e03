// Planning stage: turns the device-side metadata into per-token and
// per-group work descriptions, and (consumer mode) the sorted set of usable
// candidate blocks per token.
//
// The metadata follows the guide "DeepSeek V4.1 QLI V2 与候选集成", section
// 数据流: raw query boundaries (cu_seqlens_q), compressed K lengths and the raw
// length mod ratio (absent for ratio 1). Causal mask mode 3 is read as: the
// queries of a request are the last q_len of its S = k_len*ratio + residual
// raw tokens, and compressed position j (raw span [j*r, j*r + r - 1]) is
// visible to the query at raw position pos once pos >= j*r + r - 1, i.e.
// V = floor((pos + 1) / r) positions.
#include <climits>

#include "qli_internal.h"
#include "qli_meta.cuh"
#include "qli_ptx.cuh"

namespace qli {
namespace {

// Exclusive prefix sum of f(0..n-1) into out[0..n], by one CTA of NT threads.
template <int NT, class F>
__device__ void cta_scan_store(int32_t n, F f, int32_t* out) {
  __shared__ int32_t warp_tot[NT / 32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int32_t base = 0; base < n; base += NT) {
    const int32_t i = base + tid;
    const int32_t v = i < n ? f(i) : 0;
    int32_t incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int32_t x = lane < NT / 32 ? warp_tot[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane < NT / 32) warp_tot[lane] = x;
    }
    __syncthreads();
    const int32_t excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - v;
    if (i < n) out[i] = excl;
    __syncthreads();
    if (tid == NT - 1) carry = excl + v;
    __syncthreads();
  }
  if (tid == 0) out[n] = carry;
}

constexpr int kZeroChunk = 64 * 1024;
constexpr int kPlanReqCache = 1024;   // requests whose metadata block 0 keeps in shared memory
constexpr int kPlanTokCache = 4096;   // tokens whose tile counts block 0 keeps in shared memory

// Block 0 sanitises the metadata (clamping it so no later kernel can leave
// its buffers, and flagging what was clamped), then writes V(t), the request
// of every token and the token groups that share one score tile. Blocks 1..
// zero the score stage's selection histograms (16 KB per row) in 64 KB
// chunks.

__global__ void __launch_bounds__(1024) plan_kernel(DevArgs a) {
  pdl_trigger();
  if (blockIdx.x > 0) {
    const size_t bytes = sizeof(uint32_t) * kHistBins * 2 * static_cast<size_t>(a.T);
    const size_t lo = static_cast<size_t>(blockIdx.x - 1) * kZeroChunk;
    uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.fhist) + lo);
    const size_t n = (min(bytes, lo + kZeroChunk) - lo) / sizeof(uint4);
    for (size_t i = threadIdx.x; i < n; i += blockDim.x) p[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const int tid = threadIdx.x;
  __shared__ uint32_t s_err;
  // requests' sanitised metadata and tokens' tile counts stay in shared
  // memory when they fit (the global copies are written either way)
  __shared__ int32_t s_q0[kPlanReqCache], s_q1[kPlanReqCache], s_lk[kPlanReqCache],
      s_res[kPlanReqCache];
  __shared__ int32_t s_tiles[kPlanTokCache];
  const bool req_small = a.B <= kPlanReqCache;
  const bool dense_stream = a.stream_path && a.mode != QLI_CAND_CONSUMER;
  const bool tok_small = dense_stream && a.T <= kPlanTokCache;
  if (tid == 0) s_err = 0u;
  if (!a.stream_path)
    for (int g = tid; g < a.Gmax; g += blockDim.x) a.grp_cnt[g] = 0;
  __syncthreads();

  // every request on its own: clamp the query range into [0, T], the
  // compressed length into [0, cap] and the residual into [0, ratio)
  uint32_t e = 0u;
  for (int b = tid; b < a.B; b += blockDim.x) {
    int32_t q0, q1, lk, res;
    e |= sanitize_request(a, b, q0, q1, lk, res);
    a.req_q0[b] = q0;
    a.req_q1[b] = q1;
    a.req_lk[b] = lk;
    a.req_res[b] = res;
    if (req_small) {
      s_q0[b] = q0;
      s_q1[b] = q1;
      s_lk[b] = lk;
      s_res[b] = res;
    }
  }
  if (e) atomicOr(&s_err, e);
  __syncthreads();
  const int32_t* q0s = req_small ? s_q0 : a.req_q0;
  const int32_t* q1s = req_small ? s_q1 : a.req_q1;
  const int32_t* lks = req_small ? s_lk : a.req_lk;
  const int32_t* ress = req_small ? s_res : a.req_res;
  if (!a.stream_path) {
    // first token group of every request (groups never span two requests)
    cta_scan_store<1024>(a.B, [&](int32_t b) { return (q1s[b] - q0s[b] + a.G - 1) / a.G; },
                         a.req_g0);
  }
  if (tid == 0) {
    *a.err = s_err;   // first writer of this call: resets the word
    *a.counter = 0u;
  }

  // every token: its request is the last one starting at or before it (the
  // sanitised starts never decrease for valid metadata; a token no request
  // covers keeps V = 0 and request -1)
  for (int t = tid; t < a.T; t += blockDim.x) {
    int32_t owner;
    const int32_t V = token_owner(a, q0s, q1s, lks, ress, t, owner);
    a.tok_V[t] = V;
    a.tok_b[t] = owner;
    if (tok_small) s_tiles[t] = (V + kTile - 1) / kTile;
  }
  __syncthreads();

  if (dense_stream) {
    // stream path, dense modes: token t owns ceil(V(t)/128) score tiles
    cta_scan_store<1024>(
        a.T, [&](int32_t t) { return tok_small ? s_tiles[t] : (a.tok_V[t] + kTile - 1) / kTile; },
        a.unit_start);
  } else if (!a.stream_path) {
    // group path: one warp per request, lanes over its groups
    const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    for (int b = warp; b < a.B; b += nwarps) {
      const int32_t q0 = q0s[b], qlen = q1s[b] - q0;
      const int32_t ng = (qlen + a.G - 1) / a.G;
      for (int gi = lane; gi < ng; gi += 32) {
        const int32_t g = a.req_g0[b] + gi;
        if (g < a.Gmax) {
          a.grp_t0[g] = q0 + gi * a.G;
          a.grp_cnt[g] = min(a.G, qlen - gi * a.G);
        }
      }
    }
    __syncthreads();
    // group g owns ceil(V/128) position tiles, V of its last (most
    // advanced) token: unit_start is the tile prefix over the groups
    cta_scan_store<1024>(
        a.Gmax,
        [&](int32_t g) {
          const int32_t c = a.grp_cnt[g];
          if (c == 0) return 0;
          return (a.tok_V[a.grp_t0[g] + c - 1] + kTile - 1) / kTile;
        },
        a.unit_start);
  }
}

// Consumer mode: the last CTA to finish turns the per-token candidate counts
// into the stream path's tile prefix (token t owns ceil(count/16) tiles of
// 128 candidate positions).
template <int NT>
__device__ void consumer_units(const DevArgs& a) {
  __shared__ bool s_last;
  __threadfence();
  if (threadIdx.x == 0) s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (s_last && a.stream_path) {
    __threadfence();
    cta_scan_store<NT>(
        a.T, [&](int32_t i) { return (__ldcg(&a.cand_cnt[i]) + kTile / kBlock - 1) / (kTile / kBlock); },
        a.unit_start);
  }
}

// The page of each of token t's n listed candidate blocks (its request's
// block table at the block's first position) and the block's eight FP16 K
// scales (16 bytes after the page's K rows), one coalesced pass after the
// list is written; an entry outside the pool sets QLI_DEVERR_PAGE and reads
// page 0 instead. The score kernel then needs one round trip per tile and
// one copy per block.
template <int NT>
__device__ void cand_pages(const DevArgs& a, int t, int32_t n, const int32_t* list) {
  __syncthreads();                       // the CTA's list writes are visible
  const int32_t b = a.tok_b[t];
  int32_t* pages = a.cand_page + static_cast<int64_t>(t) * a.C;
  const int64_t bt_row = static_cast<int64_t>(b < 0 ? 0 : b) * a.bt_stride;
  bool bad = false;
  for (int32_t i = threadIdx.x; i < n; i += NT) {
    const int64_t pos0 = static_cast<int64_t>(list[i]) * kBlock;
    int32_t page = a.bt[bt_row + pos0 / a.R];
    if (page < 0 || page >= a.num_pages) {
      bad = true;
      page = 0;
    }
    pages[i] = page;
    a.cand_sc[static_cast<int64_t>(t) * a.C + i] = *reinterpret_cast<const uint4*>(
        a.cache + static_cast<int64_t>(page) * a.page_stride + a.s_off + (pos0 % a.R) * 2);
  }
  if (bad) atomicOr(a.err, QLI_DEVERR_PAGE);
}

// Consumer mode, one CTA per token: keep the candidate IDs that name a block
// with at least one visible position (0 <= id < ceil(V/8)), sort them
// ascending and drop duplicates. The guide gives candidates as a padded list
// of block IDs; they are used as a set.
constexpr int kPrepThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) cand_prep_kernel(DevArgs a, int32_t pow2) {
  __shared__ int32_t keys[kMaxCand];
  __shared__ int32_t warp_sum[kPrepThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();                            // V(t) and the zeroed counter
  const int32_t V = a.tok_V[t];
  const int32_t nb = (V + kBlock - 1) / kBlock;
  const int32_t* row = a.cand_in + static_cast<int64_t>(t) * a.C;
  for (int k = tid; k < pow2; k += kPrepThreads) {
    int32_t v = k < a.C ? row[k] : INT_MAX;
    if (v < 0 || v >= nb) v = INT_MAX;
    keys[k] = v;
  }
  __syncthreads();
  // bitonic sort, ascending
  for (int size = 2; size <= pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int k = tid; k < pow2; k += kPrepThreads) {
        const int partner = k ^ stride;
        if (partner > k) {
          const bool up = (k & size) == 0;
          const int32_t x = keys[k], y = keys[partner];
          if ((x > y) == up) {
            keys[k] = y;
            keys[partner] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  // keep first occurrences of real IDs; each thread owns a contiguous run
  const int per = pow2 / kPrepThreads > 0 ? pow2 / kPrepThreads : 1;
  const int lo = tid * per;
  int cnt = 0;
  for (int k = lo; k < lo + per && k < pow2; ++k)
    cnt += (keys[k] != INT_MAX && (k == 0 || keys[k] != keys[k - 1])) ? 1 : 0;
  // block exclusive scan of cnt
  const int lane = tid & 31, warp = tid >> 5;
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < kPrepThreads / 32; ++w) {
    if (w < warp) base += warp_sum[w];
    total += warp_sum[w];
  }
  int pos = base + incl - cnt;
  int32_t* out = a.cand_list + static_cast<int64_t>(t) * a.C;
  for (int k = lo; k < lo + per && k < pow2; ++k)
    if (keys[k] != INT_MAX && (k == 0 || keys[k] != keys[k - 1])) out[pos++] = keys[k];
  if (tid == 0) a.cand_cnt[t] = total;
  cand_pages<kPrepThreads>(a, t, total, a.cand_list + static_cast<int64_t>(t) * a.C);

  consumer_units<kPrepThreads>(a);
}

// Consumer mode, the same result for contexts of up to kBitmapWords * 32
// candidate blocks: one CTA per token marks the valid IDs in a bitmap of the
// token's visible blocks (shared memory), then writes the set bits in
// ascending order (one block scan of the per-thread bit counts): sorted,
// without duplicates, in a few barriers.
constexpr int kBitmapThreads = 512;
constexpr int kBitmapWords = 16384;                  // 64 KB: 524288 blocks

__global__ void __launch_bounds__(kBitmapThreads) cand_bitmap_kernel(DevArgs a, int32_t words) {
  extern __shared__ uint32_t bm[];
  __shared__ int32_t warp_sum[kBitmapThreads / 32];
  __shared__ int32_t s_list[kMaxCand];    // the list again, for the page lookups
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the score kernel may start its set-up now; V(t) and the zeroed counter
  // come from the planning kernel
  pdl_trigger();
  pdl_wait();
  const int32_t V = a.tok_V[t];
  const int32_t nb = (V + kBlock - 1) / kBlock;
  const int32_t nw = min((nb + 31) >> 5, words);
  for (int i = tid; i < nw; i += kBitmapThreads) bm[i] = 0u;
  __syncthreads();
  const int32_t* row = a.cand_in + static_cast<int64_t>(t) * a.C;
  for (int k = tid; k < a.C; k += kBitmapThreads) {
    const int32_t id = row[k];
    if (id >= 0 && id < nb && (id >> 5) < nw) atomicOr(&bm[id >> 5], 1u << (id & 31));
  }
  __syncthreads();
  // thread i owns words [i * per, (i + 1) * per)
  const int32_t per = (nw + kBitmapThreads - 1) / kBitmapThreads;
  const int32_t w0 = tid * per, w1 = min(nw, w0 + per);
  int cnt = 0;
  for (int32_t w = w0; w < w1; ++w) cnt += __popc(bm[w]);
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < kBitmapThreads / 32; ++w) {
    if (w < warp) base += warp_sum[w];
    total += warp_sum[w];
  }
  int pos = base + incl - cnt;
  int32_t* out = a.cand_list + static_cast<int64_t>(t) * a.C;
  for (int32_t w = w0; w < w1; ++w) {
    uint32_t bits = bm[w];
    while (bits) {
      const int32_t id = (w << 5) + (__ffs(bits) - 1);
      out[pos] = id;
      s_list[pos++] = id;
      bits &= bits - 1u;
    }
  }
  if (tid == 0) a.cand_cnt[t] = total;
  cand_pages<kBitmapThreads>(a, t, total, s_list);
  consumer_units<kBitmapThreads>(a);
}

std::atomic<uint64_t> g_smem_cand_bitmap{0};

}  // namespace

cudaError_t launch_plan(const DevArgs& d, cudaStream_t s) {
  const size_t hist_bytes =
      d.fhist ? sizeof(uint32_t) * kHistBins * 2 * static_cast<size_t>(d.T) : 0;
  const unsigned zero_blocks = static_cast<unsigned>((hist_bytes + kZeroChunk - 1) / kZeroChunk);
  plan_kernel<<<1 + zero_blocks, 1024, 0, s>>>(d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (d.mode == QLI_CAND_CONSUMER && d.T > 0) {
    // the bitmap covers every block a token can see: ceil(cap / 8) bits
    const int64_t words = (static_cast<int64_t>(d.cap) / kBlock + 1 + 31) / 32;
    if (words <= kBitmapWords) {
      const int w = static_cast<int>(words);
      if (4 * w > 48 * 1024) {
        e = ensure_smem_limit(reinterpret_cast<const void*>(cand_bitmap_kernel), 4 * kBitmapWords,
                              g_smem_cand_bitmap);
        if (e != cudaSuccess) return e;
      }
      e = launch_pdl(cand_bitmap_kernel, dim3(static_cast<unsigned>(d.T)), dim3(kBitmapThreads),
                     static_cast<size_t>(4 * w), s, d, w);
      if (e != cudaSuccess) return e;
    } else {
      int32_t pow2 = 1;
      while (pow2 < d.C) pow2 <<= 1;
      if (pow2 < kPrepThreads) pow2 = kPrepThreads;
      e = launch_pdl(cand_prep_kernel, dim3(static_cast<unsigned>(d.T)), dim3(kPrepThreads), 0, s,
                     d, pow2);
      if (e != cudaSuccess) return e;
    }
    e = cudaGetLastError();
  }
  return e;
}

int plan_launches(const DevArgs& d) {
  return 1 + ((d.mode == QLI_CAND_CONSUMER && d.T > 0) ? 1 : 0);
}

}  // namespace qli
