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
// lower position / block ID. Scores are compared as order-preserving 32-bit
// keys. A row's threshold bin comes from a 4096-bin histogram of the keys'
// top 12 bits (built by the decode score stage, or counted here in shared
// memory for prefill rows); one pass compacts the entries at or above that
// bin in row order, an exact refine on the remaining 20 bits (10-bit digits)
// finds the want-th key, and two warp-segmented sweeps write the IDs in
// position order, so no sort is needed. Rows longer than one CTA's shared
// memory are compacted chunk by chunk by lcompact_kernel first. When a bin
// holds more candidates than the scratch space, the whole row is ranked by a
// digit-by-digit radix select below the bits its eligible keys share.
#include <cuda_fp16.h>

#include "qli_fast_select.cuh"
#include "qli_internal.h"
#include "qli_ptx.cuh"

namespace qli {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSampleKeys = 1024;      // sample size of the sample path
constexpr int kHeadWords = 4096;       // scratch head: the sample or a row's histogram
constexpr int kCandCap = 8192;         // candidates the sample / histogram paths keep

struct Shared {
  uint32_t hist[256];
  int warp_a[kWarps], warp_b[kWarps];
  int chunk_w[2][kWarps];
  uint32_t red[kWarps][3];
  uint32_t sel[3];
};

static_assert(kWarps == 32, "per-warp tables are read one entry per lane");

// Sum of per_warp[] over the warps before this one, and the block total:
// one shared-memory read per lane and a warp scan.
__device__ __forceinline__ int warps_before(const int* per_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int x = per_warp[lane];
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(0xffffffffu, incl, 31);
  return __shfl_sync(0xffffffffu, incl - x, warp);
}

// Adds the warp's live digits to `hist` with one shared atomic per distinct
// digit: lanes holding the same digit are found by one ballot per digit bit.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool live, uint32_t digit, int width) {
  const unsigned live_mask = __ballot_sync(0xffffffffu, live);
  if (live_mask == 0u) return;
  unsigned peers = live_mask;
  for (int b = 0; b < width; ++b) {
    const bool bit = (digit >> b) & 1u;
    const unsigned m = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? m : ~m;
  }
  const int lane = threadIdx.x & 31;
  if (live && (__ffs(peers) - 1) == lane) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
}

// Eligible count and the extreme eligible keys of a row.
struct Stats {
  uint32_t E, kmax, kmin;
};

// Block totals of the per-warp statistics in sh.red (every thread gets them).
__device__ __forceinline__ Stats block_stats_from(const Shared& sh) {
  const int lane = threadIdx.x & 31;
  Stats st{sh.red[lane][0], sh.red[lane][1], sh.red[lane][2]};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    st.E += __shfl_xor_sync(0xffffffffu, st.E, o);
    st.kmax = max(st.kmax, __shfl_xor_sync(0xffffffffu, st.kmax, o));
    st.kmin = min(st.kmin, __shfl_xor_sync(0xffffffffu, st.kmin, o));
  }
  return st;
}

__device__ Stats row_stats(const Row& r, Shared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t cnt = 0u, kmax = 0u, kmin = 0xffffffffu;
  for (int32_t s = tid; s < r.len; s += kThreads) {
    const uint32_t k = r.key(s);
    if (k != 0u) {
      ++cnt;
      kmax = max(kmax, k);
      kmin = min(kmin, k);
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
  }
  __syncthreads();
  if (lane == 0) {
    sh.red[warp][0] = cnt;
    sh.red[warp][1] = kmax;
    sh.red[warp][2] = kmin;
  }
  __syncthreads();
  Stats st = block_stats_from(sh);
  return st;
}

// The key of the k-th best eligible entry (k <= E) and how many entries
// equal to it rank within the best k: take keys > thr plus the first
// need_eq keys == thr. Exact radix select, 8-bit digits below the bits
// every eligible key shares.
__device__ void radix_threshold(const Row& r, int32_t k, const Stats& st, uint32_t& thr,
                                int32_t& need_eq, Shared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t diff = st.kmax ^ st.kmin;
  if (diff == 0u) {
    thr = st.kmax;          // every eligible key is equal: take the first k
    need_eq = k;
    return;
  }
  int hi = 31 - __clz(diff);               // highest bit still undecided
  uint32_t mask = hi == 31 ? 0u : ~((2u << hi) - 1u);
  uint32_t prefix = st.kmax & mask;
  while (hi >= 0) {
    const int width = hi + 1 < 8 ? hi + 1 : 8;
    const int shift = hi + 1 - width;
    if (tid < 256) sh.hist[tid] = 0u;
    __syncthreads();
    const int32_t rounds = (r.len + kThreads - 1) / kThreads;
    for (int32_t i = 0; i < rounds; ++i) {
      const int32_t s = i * kThreads + tid;
      const uint32_t key = s < r.len ? r.key(s) : 0u;
      const bool live = key != 0u && (key & mask) == prefix;
      hist_add(sh.hist, live, (key >> shift) & ((1u << width) - 1u), width);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns 8 bins from the top; find the bin holding rank k
      const int nb = 1 << width;
      uint32_t c[8];
      uint32_t mine = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int bin = nb - 1 - 8 * lane - j;
        c[j] = bin >= 0 ? sh.hist[bin] : 0u;
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
            sh.sel[0] = static_cast<uint32_t>(nb - 1 - 8 * lane - j);
            sh.sel[1] = static_cast<uint32_t>(k) - above;
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= sh.sel[0] << shift;
    mask |= ((1u << width) - 1u) << shift;
    k = static_cast<int32_t>(sh.sel[1]);
    __syncthreads();
    hi = shift - 1;
  }
  thr = prefix;
  need_eq = k;
}

// Writes, in row order, the ids of the entries with key > thr and of the
// first need_eq entries with key == thr; returns how many. Warp w owns a
// contiguous segment: one sweep counts, one block prefix places the warps,
// a second sweep writes. At most `cap` ids are written (the room the caller
// has): the threshold always admits at most that many when it was derived
// from the row itself, and the bound keeps a row whose score-stage
// histogram disagrees with its scores (a score stage that gave up a wait)
// inside its output.
__device__ int ordered_output(const Row& r, uint32_t thr, int32_t need_eq, int32_t* out,
                              int32_t cap, Shared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t seg = ((r.len + kWarps - 1) / kWarps + 31) & ~31;
  const int32_t lo = warp * seg, hi = min(r.len, lo + seg);
  const unsigned below = (1u << lane) - 1u;
  int gt_cnt = 0, eq_cnt = 0;
  for (int32_t base = lo; base < hi; base += 32) {
    const int32_t s = base + lane;
    const uint32_t key = s < hi ? r.key(s) : 0u;
    gt_cnt += __popc(__ballot_sync(0xffffffffu, key != 0u && key > thr));
    eq_cnt += __popc(__ballot_sync(0xffffffffu, key != 0u && key == thr && need_eq > 0));
  }
  __syncthreads();
  if (lane == 0) {
    sh.warp_a[warp] = gt_cnt;
    sh.warp_b[warp] = eq_cnt;
  }
  __syncthreads();
  int total_gt, total_eq;
  const int gt_before = warps_before(sh.warp_a, total_gt);
  const int eq_before = warps_before(sh.warp_b, total_eq);
  int at = gt_before + min(need_eq, eq_before);
  int eq_seen = eq_before;
  for (int32_t base = lo; base < hi; base += 32) {
    const int32_t s = base + lane;
    const uint32_t key = s < hi ? r.key(s) : 0u;
    const bool gt = key != 0u && key > thr;
    const bool eq = key != 0u && key == thr && need_eq > 0;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_seen + __popc(eqm & below) < need_eq);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    const int o = at + __popc(tm & below);
    if (take && o < cap) out[o] = r.id(s);
    at += __popc(tm);
    eq_seen += __popc(eqm);
  }
  __syncthreads();
  return min(total_gt + min(need_eq, total_eq), cap);
}

// Indices s (in row order) of the entries with key >= t_lo, into idx[];
// returns how many (idx is written only while the count stays <= cap).
__device__ int compact_at_least(const Row& r, uint32_t t_lo, int32_t* idx, int cap, Shared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t seg = ((r.len + kWarps - 1) / kWarps + 31) & ~31;
  const int32_t lo = warp * seg, hi = min(r.len, lo + seg);
  const unsigned below = (1u << lane) - 1u;
  int cnt = 0;
  for (int32_t base = lo; base < hi; base += 32) {
    const int32_t s = base + lane;
    const uint32_t key = s < hi ? r.key(s) : 0u;
    cnt += __popc(__ballot_sync(0xffffffffu, key != 0u && key >= t_lo));
  }
  __syncthreads();
  if (lane == 0) sh.warp_a[warp] = cnt;
  __syncthreads();
  int total;
  int at = warps_before(sh.warp_a, total);
  if (total <= cap) {
    for (int32_t base = lo; base < hi; base += 32) {
      const int32_t s = base + lane;
      const uint32_t key = s < hi ? r.key(s) : 0u;
      const bool keep = key != 0u && key >= t_lo;
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      if (keep) idx[at + __popc(m & below)] = s;
      at += __popc(m);
    }
  }
  __syncthreads();
  return total;
}

// Block-wide inclusive scan of one value per thread (thread order); returns
// the thread's inclusive sum and the block total. Two barriers.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t& total, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();                       // the previous scan's readers are done
  if (lane == 31) sh.warp_a[warp] = static_cast<int>(incl);
  __syncthreads();
  uint32_t w = static_cast<uint32_t>(sh.warp_a[lane]), wincl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += y;
  }
  total = __shfl_sync(0xffffffffu, wincl, 31);
  return incl + __shfl_sync(0xffffffffu, wincl - w, warp);
}

// Where the want-th best entry of a row sits in its 4096-bin histogram of
// the top 12 key bits (built by the score stage): bin `sel`, `above` entries
// in higher bins, `cbin` in bin sel itself; E = the row's eligible count.
// `pinned` (-1: none) is the bin of the pinned last block, which the block
// row does not rank. Thread i holds bins 4095-4i .. 4092-4i (one 16-byte
// load).
struct HistSel {
  uint32_t sel, above, cbin, E;
};
static_assert(kHistBins == 4 * kThreads, "one 16-byte histogram load per thread");

// This thread's 16-byte word of a row's histogram (see hist_select).
__device__ __forceinline__ uint4 hist_word(const uint32_t* g) {
  return __ldcg(reinterpret_cast<const uint4*>(g) + (kHistBins / 4 - 1 - static_cast<int>(threadIdx.x)));
}

__device__ HistSel hist_select_word(const uint4 v, int32_t pinned, int32_t want, Shared& sh) {
  const int tid = threadIdx.x;
  const int q = kHistBins / 4 - 1 - tid;
  uint32_t c[4] = {v.w, v.z, v.y, v.x};                     // bins 4q+3 .. 4q
  if (pinned >= 0 && (pinned >> 2) == q) c[3 - (pinned & 3)] -= 1u;
  const uint32_t mine = c[0] + c[1] + c[2] + c[3];
  uint32_t E;
  const uint32_t incl = block_scan(mine, E, sh);
  const uint32_t k = static_cast<uint32_t>(want);
  uint32_t above = incl - mine;
  if (E > k && above < k && k <= incl) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (above + c[j] >= k) {
        sh.sel[0] = static_cast<uint32_t>(4 * q + 3 - j);
        sh.sel[1] = above;
        sh.sel[2] = c[j];
        break;
      }
      above += c[j];
    }
  }
  __syncthreads();
  HistSel h{sh.sel[0], sh.sel[1], sh.sel[2], E};
  __syncthreads();
  return h;
}

__device__ __forceinline__ HistSel hist_select(const uint32_t* g, int32_t pinned, int32_t want,
                                               Shared& sh) {
  return hist_select_word(hist_word(g), pinned, want, sh);
}

// One pass over entries [begin, end) of a row in global memory keeping, in
// row order, every eligible entry whose key passes keep(): its key to
// ckeys[] and its id (position) to cid[] (shared or global memory); returns
// how many (written only while below cap). Chunks of 4096 entries, thread i
// taking entries 4i..4i+3 of a chunk with one 16-byte load (begin is a
// multiple of 4); the loads of up to kBatch chunks are issued before the
// first is used. One barrier per chunk.
template <bool kConsumer, class Keep>
__device__ int compact_range(const Row& r, int32_t begin, int32_t end, Keep keep_key,
                             uint32_t* ckeys, int32_t* cid, int cap, Shared& sh) {
  constexpr int kBatch = 6;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned below = (1u << lane) - 1u;
  const int32_t nchunks = (end - begin + 4 * kThreads - 1) / (4 * kThreads);
  const float4* v4 = reinterpret_cast<const float4*>(r.vals);
  int base = 0;
  for (int32_t c0 = 0; c0 < nchunks; c0 += kBatch) {
    float4 f[kBatch];
    int32_t blk[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int32_t s0 = begin + (c0 + u) * 4 * kThreads + 4 * tid;
      f[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      blk[u] = 0;
      if (s0 < end) {
        f[u] = __ldcg(v4 + (s0 >> 2));
        if (kConsumer) blk[u] = __ldcg(r.blocks + (s0 >> 3));
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (c0 + u >= nchunks) break;                         // block-uniform
      const int32_t s0 = begin + (c0 + u) * 4 * kThreads + 4 * tid;
      const int32_t id0 = kConsumer ? blk[u] * kBlock + (s0 & (kBlock - 1)) : s0;
      const uint32_t k[4] = {order_key(f[u].x), order_key(f[u].y), order_key(f[u].z),
                             order_key(f[u].w)};
      unsigned keep = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool ok = s0 + j < end && (!kConsumer || id0 + j < r.V) && k[j] != 0u && keep_key(k[j]);
        keep |= ok ? (1u << j) : 0u;
      }
      const int cnt = __popc(keep);
      const unsigned b0 = __ballot_sync(0xffffffffu, cnt & 1), b1 = __ballot_sync(0xffffffffu, cnt & 2),
                     b2 = __ballot_sync(0xffffffffu, cnt & 4);
      const int pre = __popc(b0 & below) + 2 * __popc(b1 & below) + 4 * __popc(b2 & below);
      const int wsum = __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
      const int par = (c0 + u) & 1;                         // two buffers: one barrier per chunk
      if (lane == 0) sh.chunk_w[par][warp] = wsum;
      __syncthreads();
      const int w = sh.chunk_w[par][lane];
      int wincl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += y;
      }
      int at = base + __shfl_sync(0xffffffffu, wincl - w, warp) + pre;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if ((keep >> j) & 1u) {
          if (at < cap) {
            ckeys[at] = k[j];
            cid[at] = id0 + j;
          }
          ++at;
        }
      }
      base += __shfl_sync(0xffffffffu, wincl, 31);
    }
  }
  __syncthreads();
  return base;
}

// Ordered compaction of a row of at most kShortChunks * 4096 entries whose
// threshold bin is known (t_lo: the bin's lowest key). The row is read in
// chunks of 4096 entries, thread i taking entries 4i..4i+3 of each chunk
// with one 16-byte load (all issued together); the raw values go to
// `cache` (shared memory, the row's length), a keep bit per entry stays in a
// register, and only kept entries are turned into keys. The row-order offset of thread i's kept entries in chunk c is
// (kept entries of chunks before c) + (kept entries of chunk c in threads
// before i): packed warp scans give all chunks' offsets at once (8-bit
// fields within a warp, 16-bit fields across warps) with one block barrier.
// Kept keys go to ckeys[], their ids to cid[] (shared or global memory,
// written only while below cap); a dense row's ids are id_base + entry.
// Returns how many there are.
constexpr int kShortChunks = 8;
constexpr int kCandHalf = (kHeadWords + kCandCap - 1024) / 2;   // 5632

// The row's entries as float4 chunks (thread i: entries 4i..4i+3 of each
// chunk of 4096) and, for a consumer row, the block of each chunk's group of
// eight; issued together, so one round trip covers the row.
template <bool kConsumer>
__device__ __forceinline__ void short_load(const Row& r, float4 (&f)[kShortChunks],
                                           int32_t (&blk)[kShortChunks]) {
  const int tid = threadIdx.x;
  const int32_t nch = (r.len + 4 * kThreads - 1) / (4 * kThreads);
  const float4* v4 = reinterpret_cast<const float4*>(r.vals);
#pragma unroll
  for (int c = 0; c < kShortChunks; ++c) {
    const int32_t s0 = c * 4 * kThreads + 4 * tid;
    f[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    blk[c] = 0;
    if (c < nch && s0 < r.len) {
      f[c] = __ldcg(v4 + (s0 >> 2));
      if (kConsumer) blk[c] = __ldcg(r.blocks + (s0 >> 3));
    }
  }
}

// order_key(x) >= t_lo as one unsigned range test on the raw FP32 bits u:
// (u - lo) <= span. A threshold at or above 2^31 (non-negative values) keeps
// lo' <= u <= 0x7fffffff with lo' = t_lo - 2^31, and also u = 0x80000000
// (-0, whose key is +0's) when lo' = 0; a lower threshold keeps every u <=
// ~t_lo (all non-negative values, -0, and the negative ones down to it).
struct KeepRange {
  uint32_t lo, span;
  __device__ __forceinline__ explicit KeepRange(uint32_t t_lo) {
    if (t_lo >= 0x80000000u) {
      lo = t_lo - 0x80000000u;
      span = lo == 0u ? 0x80000000u : 0x7fffffffu - lo;
    } else {
      lo = 0u;
      span = ~t_lo;
    }
  }
  __device__ __forceinline__ bool operator()(uint32_t u) const { return u - lo <= span; }
};

// Compacts a row of up to kShortChunks chunks already loaded by short_load:
// raw values to `cache` (shared memory), then, in row order, the key and id
// of every entry whose key is >= t_lo to ckeys / cid (written while below
// cap). Per-chunk counts travel as packed 8-bit fields through one warp scan
// and (widened to 16 bits) one cross-warp scan, so the whole compaction
// takes one barrier pair. Returns how many entries passed.
template <bool kConsumer>
__device__ int compact_short_from(const Row& r, uint32_t t_lo, const float4 (&f)[kShortChunks],
                                  const int32_t (&blk)[kShortChunks], uint32_t* cache,
                                  uint32_t* ckeys, int32_t* cid, int cap, Shared& sh,
                                  int32_t id_base = 0) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t nch = (r.len + 4 * kThreads - 1) / (4 * kThreads);
  const KeepRange pass(t_lo);
  const auto id_of = [&](int c, int j) {
    const int32_t s = c * 4 * kThreads + 4 * tid + j;
    return kConsumer ? blk[c] * kBlock + (s & (kBlock - 1)) : id_base + s;
  };
  // raw values to the cache, keep bits to `keep` (bit 4c + j), counts per
  // chunk as 8-bit fields (chunks 0-3 in mine[0], 4-7 in mine[1])
  uint32_t keep = 0u, mine[2] = {0u, 0u};
#pragma unroll
  for (int c = 0; c < kShortChunks; ++c) {
    const int32_t s0 = c * 4 * kThreads + 4 * tid;
    if (c < nch && s0 < r.len) {
      const uint4 u4 = make_uint4(__float_as_uint(f[c].x), __float_as_uint(f[c].y),
                                  __float_as_uint(f[c].z), __float_as_uint(f[c].w));
      uint32_t m = (pass(u4.x) ? 1u : 0u) | (pass(u4.y) ? 2u : 0u) | (pass(u4.z) ? 4u : 0u) |
                   (pass(u4.w) ? 8u : 0u);
      const int32_t left = r.len - s0;
      if (left < 4) m &= (1u << left) - 1u;
      if (kConsumer) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (id_of(c, j) >= r.V) m &= ~(1u << j);
      }
      keep |= m << (4 * c);
      *reinterpret_cast<uint4*>(cache + s0) = u4;      // s0 + 3 < the row's padded length
      mine[c >> 2] |= static_cast<uint32_t>(__popc(m)) << (8 * (c & 3));
    }
  }
  // within the warp: at most 32 x 4 per field
  uint32_t incl[2] = {mine[0], mine[1]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl[h], o);
      if (lane >= o) incl[h] += y;
    }
  }
  __syncthreads();                       // earlier users of chunk_w are done
  if (lane == 31) {
    sh.chunk_w[0][warp] = static_cast<int>(incl[0]);
    sh.chunk_w[1][warp] = static_cast<int>(incl[1]);
  }
  __syncthreads();
  // across warps: lane l holds warp l's totals, widened to 16-bit fields
  uint32_t wide[4];
  {
    const uint32_t lo = static_cast<uint32_t>(sh.chunk_w[0][lane]);
    const uint32_t hi = static_cast<uint32_t>(sh.chunk_w[1][lane]);
    wide[0] = (lo & 0xffu) | (((lo >> 8) & 0xffu) << 16);
    wide[1] = ((lo >> 16) & 0xffu) | ((lo >> 24) << 16);
    wide[2] = (hi & 0xffu) | (((hi >> 8) & 0xffu) << 16);
    wide[3] = ((hi >> 16) & 0xffu) | ((hi >> 24) << 16);
  }
  uint32_t wincl[4] = {wide[0], wide[1], wide[2], wide[3]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wincl[h], o);
      if (lane >= o) wincl[h] += y;
    }
  }
  int total = 0;
#pragma unroll
  for (int c = 0; c < kShortChunks; ++c) {
    const uint32_t shift = 16 * (c & 1);
    const int tot_c = static_cast<int>((__shfl_sync(0xffffffffu, wincl[c >> 1], 31) >> shift) & 0xffffu);
    const int bw = static_cast<int>(
        ((__shfl_sync(0xffffffffu, wincl[c >> 1] - wide[c >> 1], warp) >> shift) & 0xffffu));
    const int bt = static_cast<int>((((incl[c >> 2] - mine[c >> 2]) >> (8 * (c & 3))) & 0xffu));
    int at = total + bw + bt;
    total += tot_c;
    const uint32_t bits = (keep >> (4 * c)) & 0xfu;
    if (bits) {
      const int32_t s0 = c * 4 * kThreads + 4 * tid;
      const uint4 u4 = *reinterpret_cast<const uint4*>(cache + s0);
      const uint32_t uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if ((bits >> j) & 1u) {
          if (at < cap) {
            ckeys[at] = order_key(__uint_as_float(uu[j]));
            cid[at] = id_of(c, j);
          }
          ++at;
        }
      }
    }
  }
  __syncthreads();
  return total;
}

// short_load + compact_short_from.
template <bool kConsumer>
__device__ int compact_short(const Row& r, uint32_t t_lo, uint32_t* cache, uint32_t* ckeys,
                             int32_t* cid, int cap, Shared& sh, int32_t id_base = 0) {
  float4 f[kShortChunks];
  int32_t blk[kShortChunks];
  short_load<kConsumer>(r, f, blk);
  return compact_short_from<kConsumer>(r, t_lo, f, blk, cache, ckeys, cid, cap, sh, id_base);
}

// For a dense row of up to 32K entries without a score-stage histogram: one
// coalesced pass (chunks of 4096 entries, thread i taking entries 4i..4i+3
// of each) caches the keys in `cache` (shared memory) and counts their top
// 12 bits in `hist` (4096 words of shared memory, zeroed here).
__device__ void cache_and_count(const Row& r, uint32_t* cache, uint32_t* hist, Shared& sh) {
  const int tid = threadIdx.x;
  reinterpret_cast<uint4*>(hist)[tid] = make_uint4(0u, 0u, 0u, 0u);    // 4096 = 4 x kThreads
  const int32_t nch = (r.len + 4 * kThreads - 1) / (4 * kThreads);
  const float4* v4 = reinterpret_cast<const float4*>(r.vals);
  float4 f[kShortChunks];
#pragma unroll
  for (int c = 0; c < kShortChunks; ++c) {
    const int32_t s0 = c * 4 * kThreads + 4 * tid;
    f[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nch && s0 < r.len) f[c] = __ldcg(v4 + (s0 >> 2));
  }
  __syncthreads();                       // the histogram is zero
#pragma unroll
  for (int c = 0; c < kShortChunks; ++c) {
    const int32_t s0 = c * 4 * kThreads + 4 * tid;
    if (c < nch && s0 < r.len) {
      const uint4 k4 = make_uint4(order_key(f[c].x), order_key(f[c].y), order_key(f[c].z),
                                  order_key(f[c].w));
      *reinterpret_cast<uint4*>(cache + s0) = k4;     // s0 + 3 < the row's padded length
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (s0 + j < r.len) atomicAdd(&hist[hist_bin(kk[j])], 1u);
    }
  }
  __syncthreads();
  (void)sh;
}

// Ordered compaction of a dense row whose keys sit in `cache` (see
// cache_and_count): the entries with key >= t_lo, in row order, keys to
// ckeys[] and positions to cid[] (written only while below cap), placed by
// packed warp scans with one block barrier. Returns how many there are.
__device__ int compact_cached(const Row& r, uint32_t t_lo, const uint32_t* cache, uint32_t* ckeys,
                              int32_t* cid, int cap, Shared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t nch = (r.len + 4 * kThreads - 1) / (4 * kThreads);
  uint32_t keep = 0u, mine[2] = {0u, 0u};
#pragma unroll
  for (int c = 0; c < kShortChunks; ++c) {
    const int32_t s0 = c * 4 * kThreads + 4 * tid;
    if (c < nch && s0 < r.len) {
      const uint4 k4 = *reinterpret_cast<const uint4*>(cache + s0);
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
      uint32_t n = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool ok = s0 + j < r.len && kk[j] >= t_lo;
        keep |= ok ? (1u << (4 * c + j)) : 0u;
        n += ok ? 1u : 0u;
      }
      mine[c >> 2] |= n << (8 * (c & 3));
    }
  }
  uint32_t incl[2] = {mine[0], mine[1]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl[h], o);
      if (lane >= o) incl[h] += y;
    }
  }
  __syncthreads();
  if (lane == 31) {
    sh.chunk_w[0][warp] = static_cast<int>(incl[0]);
    sh.chunk_w[1][warp] = static_cast<int>(incl[1]);
  }
  __syncthreads();
  uint32_t wide[4];
  {
    const uint32_t lo = static_cast<uint32_t>(sh.chunk_w[0][lane]);
    const uint32_t hi = static_cast<uint32_t>(sh.chunk_w[1][lane]);
    wide[0] = (lo & 0xffu) | (((lo >> 8) & 0xffu) << 16);
    wide[1] = ((lo >> 16) & 0xffu) | ((lo >> 24) << 16);
    wide[2] = (hi & 0xffu) | (((hi >> 8) & 0xffu) << 16);
    wide[3] = ((hi >> 16) & 0xffu) | ((hi >> 24) << 16);
  }
  uint32_t wincl[4] = {wide[0], wide[1], wide[2], wide[3]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wincl[h], o);
      if (lane >= o) wincl[h] += y;
    }
  }
  int total = 0;
#pragma unroll
  for (int c = 0; c < kShortChunks; ++c) {
    const uint32_t shift = 16 * (c & 1);
    const int tot_c = static_cast<int>((__shfl_sync(0xffffffffu, wincl[c >> 1], 31) >> shift) & 0xffffu);
    const int bw = static_cast<int>(
        ((__shfl_sync(0xffffffffu, wincl[c >> 1] - wide[c >> 1], warp) >> shift) & 0xffffu));
    const int bt = static_cast<int>((((incl[c >> 2] - mine[c >> 2]) >> (8 * (c & 3))) & 0xffu));
    int at = total + bw + bt;
    total += tot_c;
    const uint32_t bits = (keep >> (4 * c)) & 0xfu;
    if (bits) {
      const int32_t s0 = c * 4 * kThreads + 4 * tid;
      const uint4 k4 = *reinterpret_cast<const uint4*>(cache + s0);
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if ((bits >> j) & 1u) {
          if (at < cap) {
            ckeys[at] = kk[j];
            cid[at] = s0 + j;
          }
          ++at;
        }
      }
    }
  }
  __syncthreads();
  return total;
}

// Exact threshold among n candidate keys (any order) whose top 12 bits
// already single out bin `sel`: the k-th largest key of that bin (k >= 1),
// in the convention of ordered_output (take keys > thr and the first
// need_eq keys == thr). 10-bit digits on the remaining 20 bits, histogram
// in `hist` (1024 words of shared memory); stops as soon as the chosen
// digit's entries are exactly the ones still needed.
__device__ void refine_threshold(const uint32_t* ckeys, int n, uint32_t sel, int32_t k,
                                 uint32_t* hist, Shared& sh, uint32_t& thr, int32_t& need_eq) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t prefix = sel << (32 - kHistBits), mask = ~0u << (32 - kHistBits);
  int hi = 31 - kHistBits;
  while (hi >= 0) {
    const int width = hi + 1 < 10 ? hi + 1 : 10;
    const int shift = hi + 1 - width;
    const int nb = 1 << width;
    hist[tid] = 0u;
    __syncthreads();
    for (int b = 0; b < n; b += kThreads) {
      const int s = b + tid;
      const uint32_t key = s < n ? ckeys[s] : 0u;
      const bool live = s < n && (key & mask) == prefix;
      const uint32_t d = live ? (key >> shift) & static_cast<uint32_t>(nb - 1) : 0xffffffffu;
      const unsigned peers = __match_any_sync(0xffffffffu, d);
      if (live && (__ffs(peers) - 1) == lane) atomicAdd(&hist[d], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    // thread i holds digit nb-1-i (top down)
    const uint32_t c = tid < nb ? hist[nb - 1 - tid] : 0u;
    uint32_t total;
    const uint32_t incl = block_scan(c, total, sh);
    if (tid < nb && incl - c < static_cast<uint32_t>(k) && static_cast<uint32_t>(k) <= incl) {
      sh.sel[0] = static_cast<uint32_t>(nb - 1 - tid);
      sh.sel[1] = static_cast<uint32_t>(k) - (incl - c);
      sh.sel[2] = c;
    }
    __syncthreads();
    prefix |= sh.sel[0] << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    k = static_cast<int32_t>(sh.sel[1]);
    const uint32_t in_digit = sh.sel[2];
    __syncthreads();
    if (in_digit == static_cast<uint32_t>(k)) {
      // every key of this digit is needed: take all keys >= its lowest key
      thr = prefix == 0u ? 0u : prefix - 1u;
      need_eq = 0;
      return;
    }
    hi = shift - 1;
  }
  thr = prefix;
  need_eq = k;
}

// Writes the ids of the `want` best entries of `r` in ascending id order to
// out[0..), and returns how many were written (min(want, eligible)).
// `scratch` (shared memory, kHeadWords + kCandCap words) enables the sample
// path for long cached rows: a threshold taken a little below the want-th
// key of an evenly spaced sample keeps a few thousand candidates, compacted
// in row order, on which the exact selection runs. If the sample misjudges
// (fewer than `want` or more than kCandCap candidates) the exact selection
// runs on the whole row; the result is the same either way.
__device__ __noinline__ int select_ascending(const Row& r, int32_t want, int32_t* out, Shared& sh,
                                         uint32_t* scratch, const Stats* known = nullptr) {
  const Stats st = known ? *known : row_stats(r, sh);
  if (st.E <= static_cast<uint32_t>(want)) return ordered_output(r, 0u, 0, out, want, sh);
  if (scratch != nullptr && r.cached != nullptr && r.idx == nullptr && r.ids == nullptr &&
      r.len >= 4 * want && r.len > 2 * kSampleKeys) {
    // sample of kSampleKeys evenly spaced keys (one per thread)
    uint32_t* sample = scratch;
    int32_t* cand = reinterpret_cast<int32_t*>(scratch + kHeadWords);
    for (int i = threadIdx.x; i < kSampleKeys; i += kThreads)
      sample[i] = r.key(static_cast<int32_t>((static_cast<int64_t>(i) * r.len) / kSampleKeys));
    __syncthreads();
    Row sr = r;
    sr.cached = sample;
    sr.ids = nullptr;
    sr.idx = nullptr;
    sr.len = kSampleKeys;
    sr.consumer = false;
    const Stats ss = row_stats(sr, sh);
    // aim 20% + 16 sample ranks past the expected rank of the want-th key
    int32_t j = static_cast<int32_t>((static_cast<int64_t>(want) * kSampleKeys * 6) / (5 * r.len)) + 16;
    if (ss.E > static_cast<uint32_t>(j)) {
      uint32_t t_lo;
      int32_t eq_unused;
      radix_threshold(sr, j, ss, t_lo, eq_unused, sh);
      const int n = compact_at_least(r, t_lo, cand, kCandCap, sh);
      if (n >= want && n <= kCandCap) {
        Row cr = r;
        cr.idx = cand;
        cr.len = n;
        const Stats cs = row_stats(cr, sh);
        uint32_t thr;
        int32_t need_eq;
        radix_threshold(cr, want, cs, thr, need_eq, sh);
        return ordered_output(cr, thr, need_eq, out, want, sh);
      }
    }
  }
  uint32_t thr;
  int32_t need_eq;
  radix_threshold(r, want, st, thr, need_eq, sh);
  return ordered_output(r, thr, need_eq, out, want, sh);
}

// ---------------------------------------------------------------------------
// Long rows (more entries than one CTA holds in shared memory). Three passes,
// each spread over many CTAs (grid: chunk of 16384 entries x token x which):
//   lstat    eligible count, max key and min key of the row;
//   lhist    histogram of the 12 key bits just below the bits every eligible
//            key shares (the common prefix of max and min);
//   lcompact each CTA finds the digit holding the want-th best entry and keeps
//            its chunk's entries at or above it, in position order, in the
//            chunk's candidate segment.
// The select kernel then ranks the (few thousand) candidates exactly in
// shared memory; segments read in chunk order keep position order, so ties
// and the ascending output need no sort. A segment or a row that overflows
// its capacity falls back to ranking the row from L2.

__device__ __forceinline__ bool long_row(const DevArgs& a, int t, int which, Row& r, int32_t& want,
                                         int32_t& lo, int32_t& hi) {
  r = row_of(a, t, which, want);
  if (r.len <= kSmemKeys) return false;
  lo = blockIdx.x * kLongChunk;
  hi = min(r.len, lo + kLongChunk);
  return lo < hi;
}

__global__ void __launch_bounds__(kThreads) lstat_kernel(DevArgs a) {
  Row r;
  int32_t want, lo, hi;
  const int t = blockIdx.y, which = blockIdx.z;
  if (!long_row(a, t, which, r, want, lo, hi)) return;
  uint32_t cnt = 0u, kmax = 0u, nmin = 0u;
  for (int32_t s = lo + threadIdx.x; s < hi; s += kThreads) {
    const uint32_t k = r.key(s);
    if (k != 0u) {
      ++cnt;
      kmax = max(kmax, k);
      nmin = max(nmin, ~k);
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    nmin = max(nmin, __shfl_xor_sync(0xffffffffu, nmin, o));
  }
  if ((threadIdx.x & 31) == 0 && cnt) {
    uint32_t* e = a.lext + 4 * (2 * static_cast<int64_t>(t) + which);
    atomicMax(&e[0], kmax);
    atomicMax(&e[1], nmin);
    atomicAdd(&e[2], cnt);
  }
}

// Digit of `key` in the long-row histogram: the (up to) 12 bits below the
// row's common prefix.
struct LongDigit {
  int shift, width;
  __device__ LongDigit(uint32_t kmax, uint32_t kmin) {
    const uint32_t diff = kmax ^ kmin;
    const int hi = diff ? 31 - __clz(diff) : -1;
    width = hi + 1 < 12 ? hi + 1 : 12;
    shift = hi + 1 - width;
  }
  __device__ LongDigit() : shift(32 - kHistBits), width(kHistBits) {}  // top 12 bits
  __device__ __forceinline__ uint32_t of(uint32_t key) const {
    return width ? (key >> shift) & ((1u << width) - 1u) : 0u;
  }
};

__global__ void __launch_bounds__(kThreads) lhist_kernel(DevArgs a) {
  __shared__ uint32_t hist[4096];
  Row r;
  int32_t want, lo, hi;
  const int t = blockIdx.y, which = blockIdx.z;
  if (!long_row(a, t, which, r, want, lo, hi)) return;
  const int64_t row = 2 * static_cast<int64_t>(t) + which;
  const uint32_t* e = a.lext + 4 * row;
  const LongDigit dg(e[0], ~e[1]);
  if (e[2] <= static_cast<uint32_t>(want) || dg.width == 0) return;   // no histogram needed
  for (int i = threadIdx.x; i < 4096; i += kThreads) hist[i] = 0u;
  __syncthreads();
  const int32_t rounds = (hi - lo + kThreads - 1) / kThreads;
  for (int32_t i = 0; i < rounds; ++i) {
    const int32_t s = lo + i * kThreads + threadIdx.x;
    const uint32_t key = s < hi ? r.key(s) : 0u;
    hist_add(hist, key != 0u, dg.of(key), dg.width);
  }
  __syncthreads();
  uint32_t* g = a.lhist + 4096 * row;
  for (int i = threadIdx.x; i < 4096; i += kThreads)
    if (hist[i]) atomicAdd(&g[i], hist[i]);
}

// Dynamic shared memory: kLongChunk words caching the chunk's keys.
static_assert(kLongChunk <= kShortChunks * 4 * kThreads, "a long-row chunk fits one ordered compaction");
__global__ void __launch_bounds__(kThreads) lcompact_kernel(DevArgs a) {
  extern __shared__ uint32_t lcache[];
  pdl_trigger();
  pdl_wait();
  __shared__ Shared sh;
  Row r;
  int32_t want, lo, hi;
  const int t = blockIdx.y, which = blockIdx.z;
  if (!long_row(a, t, which, r, want, lo, hi)) return;
  const int tid = threadIdx.x;
  const int64_t row = 2 * static_cast<int64_t>(t) + which;
  const int64_t segbase = (row * a.lchunks + blockIdx.x) * static_cast<int64_t>(kLongChunkCap);
  uint32_t* okey = a.lkey + segbase;
  int32_t* oid = a.lid + segbase;
  int total;
  if (a.fhist != nullptr) {
    // the score stage's top-12-bit histogram: keep the bin holding the
    // want-th best entry and everything above it (every eligible entry when
    // the row has no more than `want`); the pinned last block is counted in
    // the block histogram but not ranked
    int32_t pinned = -1;
    if (which == 1) {
      const int32_t last = (r.V + kBlock - 1) / kBlock - 1;
      pinned = static_cast<int32_t>(
          hist_bin(order_key(a.bscores[static_cast<int64_t>(t) * a.Brow + last])));
    }
    const HistSel hs = hist_select(a.fhist + row * kHistBins, pinned, want, sh);
    const uint32_t t_lo = hs.E > static_cast<uint32_t>(want) ? hs.sel << (32 - kHistBits) : 1u;
    // the chunk as a row of its own (ids offset by its start): one ordered
    // compaction with a single barrier, keys cached in shared memory
    Row rc = r;
    rc.vals = r.vals + lo;
    if (r.consumer) rc.blocks = r.blocks + lo / kBlock;
    rc.len = hi - lo;
    total = r.consumer ? compact_short<true>(rc, t_lo, lcache, okey, oid, kLongChunkCap, sh)
                       : compact_short<false>(rc, t_lo, lcache, okey, oid, kLongChunkCap, sh, lo);
  } else {
    // the 12 bits below the row's common prefix (lstat / lhist): the digit
    // holding the want-th best entry (0: keep every eligible entry)
    const uint32_t* e = a.lext + 4 * row;
    const LongDigit dg(e[0], ~e[1]);
    const uint32_t* g = a.lhist + 4096 * row;
    if (tid == 0) sh.sel[0] = 0u;
    __syncthreads();
    if (dg.width > 0) {
      const int nb = 1 << dg.width;
      // thread i holds digits nb-1-4i .. nb-4-4i (top down)
      uint32_t c[4], mine = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int bin = nb - 1 - 4 * tid - j;
        c[j] = bin >= 0 ? g[bin] : 0u;
        mine += c[j];
      }
      uint32_t E;
      const uint32_t incl = block_scan(mine, E, sh);
      uint32_t above = incl - mine;
      const uint32_t k = static_cast<uint32_t>(want);
      if (E > k && above < k && k <= incl) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (above + c[j] >= k) {
            sh.sel[0] = static_cast<uint32_t>(nb - 1 - 4 * tid - j);
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t dmin = sh.sel[0];
    const auto keep = [dg, dmin](uint32_t k) { return dg.of(k) >= dmin; };
    total = r.consumer ? compact_range<true>(r, lo, hi, keep, okey, oid, kLongChunkCap, sh)
                       : compact_range<false>(r, lo, hi, keep, okey, oid, kLongChunkCap, sh);
  }
  if (tid == 0) a.lcount[row * a.lchunks + blockIdx.x] = total;
}

// Replaces a long row by its candidates (keys and ids in shared memory, in
// position order) when every segment fits; returns false to rank from L2.
// Thread c reads chunk c's count; a block scan places the segments; then
// every thread copies entries, four loads in flight. `offs` is shared
// scratch of at least kThreads + 1 words.
__device__ bool load_candidates(const DevArgs& a, int t, int which, Row& r, uint32_t* keys,
                                int32_t* ids, int32_t* offs, Shared& sh) {
  const int tid = threadIdx.x;
  const int64_t row = 2 * static_cast<int64_t>(t) + which;
  const int32_t nch = (r.len + kLongChunk - 1) / kLongChunk;
  if (nch > kThreads) return false;                          // block-uniform
  const int n = tid < nch ? a.lcount[row * a.lchunks + tid] : 0;
  const int over = __syncthreads_or(n > kLongChunkCap);
  uint32_t total_u;
  const uint32_t incl = block_scan(static_cast<uint32_t>(n), total_u, sh);
  const int total = static_cast<int>(total_u);
  if (over || total > kLongCandCap) return false;
  if (tid < nch) offs[tid] = static_cast<int32_t>(incl) - n;
  if (tid == 0) offs[nch] = total;
  __syncthreads();
  const int64_t seg0 = row * a.lchunks * static_cast<int64_t>(kLongChunkCap);
  for (int base = 0; base < total; base += 4 * kThreads) {
    uint32_t kk[4];
    int32_t ii[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * kThreads + tid;
      kk[u] = 0u;
      ii[u] = 0;
      if (i < total) {
        int lo = 0, hi = nch - 1;           // the chunk whose segment holds entry i
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (offs[mid] <= i) lo = mid; else hi = mid - 1;
        }
        const int64_t at = seg0 + static_cast<int64_t>(lo) * kLongChunkCap + (i - offs[lo]);
        kk[u] = __ldcg(a.lkey + at);
        ii[u] = __ldcg(a.lid + at);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * kThreads + tid;
      if (i < total) {
        keys[i] = kk[u];
        ids[i] = ii[u];
      }
    }
  }
  __syncthreads();
  r.cached = keys;
  r.ids = ids;
  r.idx = nullptr;
  r.len = total;
  r.consumer = false;
  return true;
}

// Copies the row's keys into shared memory (when it fits), points the row at
// them, and returns the row's statistics gathered on the way. Dense rows are
// read as float4, two loads in flight per thread.
__device__ __noinline__ Stats cache_keys(Row& r, uint32_t* keys, int32_t cap, Shared& sh,
                                       bool& cached) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  cached = r.len <= cap;
  uint32_t cnt = 0u, kmax = 0u, kmin = 0xffffffffu;
  auto take = [&](int32_t s, uint32_t k) {
    if (cached) keys[s] = k;
    if (k != 0u) {
      ++cnt;
      kmax = max(kmax, k);
      kmin = min(kmin, k);
    }
  };
  if (!r.consumer) {
    const int32_t nv = r.len >> 2;
    const float4* v4 = reinterpret_cast<const float4*>(r.vals);
    for (int32_t base = 0; base < nv; base += 2 * kThreads) {
      float4 f[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int32_t i = base + u * kThreads + tid;
        if (i < nv) f[u] = v4[i];
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int32_t i = base + u * kThreads + tid;
        if (i < nv) {
          take(4 * i, order_key(f[u].x));
          take(4 * i + 1, order_key(f[u].y));
          take(4 * i + 2, order_key(f[u].z));
          take(4 * i + 3, order_key(f[u].w));
        }
      }
    }
    for (int32_t s = 4 * nv + tid; s < r.len; s += kThreads) take(s, order_key(r.vals[s]));
  } else {
#pragma unroll 4
    for (int32_t s = tid; s < r.len; s += kThreads) take(s, r.key_from_global(s));
  }
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
  }
  __syncthreads();
  if (lane == 0) {
    sh.red[warp][0] = cnt;
    sh.red[warp][1] = kmax;
    sh.red[warp][2] = kmin;
  }
  __syncthreads();
  Stats st = block_stats_from(sh);
  if (cached) r.cached = keys;
  return st;
}

// A row longer than the key region: its candidates (every entry in or above
// the threshold bin or digit) were compacted by lcompact_kernel; they are
// ranked here, or the row is ranked from L2 when they overflowed.
__device__ __noinline__ int select_long_row(const DevArgs& a, int t, int which, Row r,
                                            int32_t want, uint32_t* keys, uint32_t* scratch,
                                            int32_t* out, Shared& sh) {
  const bool blocks = which == 1;
  int32_t written = 0;
  // long row: its candidates (every entry in or above the threshold bin
  // or digit) were compacted by lcompact_kernel
  int32_t* cid = reinterpret_cast<int32_t*>(keys) + kLongCandCap;
  int32_t* offs = reinterpret_cast<int32_t*>(scratch);
  bool done = false;
  if (a.lchunks > 0 && a.fhist != nullptr) {
    int32_t pinned = -1;
    if (blocks) {
      const int32_t last = (r.V + kBlock - 1) / kBlock - 1;
      pinned = static_cast<int32_t>(
          hist_bin(order_key(a.bscores[static_cast<int64_t>(t) * a.Brow + last])));
    }
    const HistSel hs = hist_select(
        a.fhist + (2 * static_cast<int64_t>(t) + which) * kHistBins, pinned, want, sh);
    if (hs.E > static_cast<uint32_t>(want) &&
        load_candidates(a, t, which, r, keys, cid, offs, sh)) {
      if (static_cast<uint32_t>(r.len) == hs.above + hs.cbin) {
        uint32_t thr;
        int32_t need_eq;
        refine_threshold(keys, r.len, hs.sel, want - static_cast<int32_t>(hs.above),
                         scratch + kHeadWords + kCandCap - 1024, sh, thr, need_eq);
        written = ordered_output(r, thr, need_eq, out, want, sh);
      } else {
        written = select_ascending(r, want, out, sh, nullptr);
      }
      done = true;
    }
  } else if (a.lchunks > 0) {
    (void)load_candidates(a, t, which, r, keys, cid, offs, sh);
  }
  if (!done) written = select_ascending(r, want, out, sh, nullptr);
  return written;
}

// Dynamic shared memory: `region` words for the row's keys (or a long row's
// candidates), then kHeadWords + kCandCap words for the sample and
// histogram paths. One instance per launch mode (score-stage histogram or
// not, consumer rows or not), so each holds only the code its rows can take.
template <bool kFused, bool kConsumerMode>
__device__ __forceinline__ void select_one(const DevArgs& a, int t, int which, int32_t key_cap,
                                           int32_t region, uint32_t* keys, Shared& sh) {
  uint32_t* scratch = keys + region;
  const int tid = threadIdx.x;
  const bool blocks = which == 1;
  const int32_t width = blocks ? a.C : a.topk;
  int32_t* out = blocks ? a.cand_out + static_cast<int64_t>(t) * a.C
                        : a.idx_out + static_cast<int64_t>(t) * a.topk;
  // the row's histogram word is requested before the row's metadata, so the
  // two round trips overlap
  const uint4 fh_word = kFused
                            ? hist_word(a.fhist + (2 * static_cast<int64_t>(t) + which) * kHistBins)
                            : make_uint4(0u, 0u, 0u, 0u);
  int32_t want;
  Row r = row_of(a, t, which, want);
  r.consumer = kConsumerMode;      // a consumer launch has only consumer rows
  int32_t written = 0;
  if (blocks && r.len == 0) {
    // at most C visible blocks: all of them, in order
    const int32_t nb = (r.V + kBlock - 1) / kBlock;
    for (int c = tid; c < nb; c += kThreads) out[c] = c;
    written = nb;
  } else {
    if (r.len > key_cap) {
      written = select_long_row(a, t, which, r, want, keys, scratch, out, sh);
    } else if (kFused) {
      // the score stage's histogram gives the threshold bin up front: the
      // entries at or above it are compacted in row order in one pass over
      // the row and ranked exactly
      int32_t pinned = -1;
      if (blocks) {
        const int32_t last = (r.V + kBlock - 1) / kBlock - 1;
        pinned = static_cast<int32_t>(
            hist_bin(order_key(a.bscores[static_cast<int64_t>(t) * a.Brow + last])));
      }
      // candidates: a row of 2 to kShortChunks chunks of 4096 entries caches
      // its values in the key region and puts the candidates' keys and ids
      // in the scratch area (kCandHalf words each); a one-chunk or a longer
      // row puts keys in the key region and ids in the scratch area (one
      // chunk needs a single barrier that way). The scratch area's last 1024
      // words hold the refine's digit histogram. A short row's loads are in
      // flight while the histogram picks the threshold bin.
      const bool short_row = r.len > 4 * kThreads && r.len <= kShortChunks * 4 * kThreads;
      float4 f[kShortChunks];
      int32_t blk[kShortChunks];
      if (short_row) short_load<kConsumerMode>(r, f, blk);
      const HistSel hs = hist_select_word(fh_word, pinned, want, sh);
      uint32_t* ckeys = short_row ? scratch : keys;
      int32_t* cid = reinterpret_cast<int32_t*>(short_row ? scratch + kCandHalf : scratch);
      const int cap = short_row ? kCandHalf : min(region, kHeadWords + kCandCap - 1024);
      const uint32_t n = hs.above + hs.cbin;
      bool done = false;
      if (hs.E <= static_cast<uint32_t>(want)) {
        written = ordered_output(r, 0u, 0, out, want, sh);        // every eligible entry, in order
        done = true;
      } else if (n <= static_cast<uint32_t>(cap)) {
        const uint32_t t_lo = hs.sel << (32 - kHistBits);
        int got;
        if (short_row) {
          got = compact_short_from<kConsumerMode>(r, t_lo, f, blk, keys, ckeys, cid, cap, sh);
        } else {
          const auto keep = [t_lo](uint32_t k) { return k >= t_lo; };
          got = compact_range<kConsumerMode>(r, 0, r.len, keep, ckeys, cid, cap, sh);
        }
        if (got == static_cast<int>(n)) {
          uint32_t thr;
          int32_t need_eq;
          refine_threshold(ckeys, got, hs.sel, want - static_cast<int32_t>(hs.above),
                           scratch + kHeadWords + kCandCap - 1024, sh, thr, need_eq);
          Row cr = r;
          cr.cached = ckeys;
          cr.ids = cid;
          cr.idx = nullptr;
          cr.len = got;
          cr.consumer = false;
          written = ordered_output(cr, thr, need_eq, out, want, sh);
          done = true;
        }
      }
      if (!done) {                      // a bin too full for the candidate space
        bool cached;
        const Stats st = cache_keys(r, keys, key_cap, sh, cached);
        written = select_ascending(r, want, out, sh, scratch, &st);
      }
    } else {
      bool done = false;
      if (!r.consumer && r.len > 1024 && r.len <= kShortChunks * 4 * kThreads) {
        // no score-stage histogram: count the row's top-12-bit bins here, in
        // the same pass that caches its keys. Scratch: the histogram (later
        // the refine's digit histogram), then candidate keys and positions.
        uint32_t* hist = scratch;
        uint32_t* ckeys = scratch + kHistBins;
        constexpr int kCap = (kHeadWords + kCandCap - kHistBins) / 2;
        int32_t* cid = reinterpret_cast<int32_t*>(ckeys + kCap);
        cache_and_count(r, keys, hist, sh);
        const HistSel hs = hist_select_word(
            reinterpret_cast<const uint4*>(hist)[kHistBins / 4 - 1 - tid], -1, want, sh);
        const uint32_t n = hs.above + hs.cbin;
        if (hs.E > static_cast<uint32_t>(want) && n <= static_cast<uint32_t>(kCap)) {
          const int got = compact_cached(r, hs.sel << (32 - kHistBits), keys, ckeys, cid, kCap, sh);
          if (got == static_cast<int>(n)) {
            uint32_t thr;
            int32_t need_eq;
            refine_threshold(ckeys, got, hs.sel, want - static_cast<int32_t>(hs.above), hist, sh,
                             thr, need_eq);
            Row cr = r;
            cr.cached = ckeys;
            cr.ids = cid;
            cr.idx = nullptr;
            cr.len = got;
            written = ordered_output(cr, thr, need_eq, out, want, sh);
            done = true;
          }
        }
      }
      if (!done) {
        bool cached;
        const Stats st = cache_keys(r, keys, key_cap, sh, cached);
        written = select_ascending(r, want, out, sh, scratch, &st);
      }
    }
    if (blocks) {                      // the pinned last visible block
      if (tid == 0) out[written] = (r.V + kBlock - 1) / kBlock - 1;
      written += 1;
    }
  }
  for (int k = written + tid; k < width; k += kThreads) out[k] = -1;
}

template <bool kFused, bool kConsumerMode>
__global__ void __launch_bounds__(kThreads) select_kernel(DevArgs a, int32_t key_cap,
                                                          int32_t region) {
  extern __shared__ uint32_t keys[];
  pdl_wait();
  __shared__ Shared sh;
  select_one<kFused, kConsumerMode>(a, blockIdx.x, blockIdx.y, key_cap, region, keys, sh);
}

__global__ void __launch_bounds__(kFT, kFPerSM) fast_select_kernel(DevArgs a) {
  extern __shared__ __align__(16) uint8_t fs_raw[];
  FastSmem& F = *reinterpret_cast<FastSmem*>(fs_raw);
  pdl_wait();
  int t, which;
  fast_row_id(a, static_cast<int32_t>(blockIdx.x), t, which);
  fast_row(a, t, which, a.tok_V[t], a.tok_b[t], F);
}

// The general selection for the rows fast_select_kernel listed, a
// persistent grid walking the list.
__global__ void __launch_bounds__(kThreads) select_list_kernel(DevArgs a, int32_t key_cap,
                                                               int32_t region) {
  extern __shared__ uint32_t keys[];
  pdl_wait();
  __shared__ Shared sh;
  const uint32_t n = __ldcg(a.counter);
  for (uint32_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int32_t item = __ldcg(a.flist + i);
    select_one<false, false>(a, item >> 1, item & 1, key_cap, region, keys, sh);
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_select(const DevArgs& d, cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  cudaError_t e;
  if (d.fhist == nullptr && d.mode != QLI_CAND_CONSUMER) {
    static std::atomic<uint64_t> done_fast{0};
    e = ensure_smem_limit(reinterpret_cast<const void*>(fast_select_kernel),
                          static_cast<int>(sizeof(FastSmem)), done_fast);
    if (e != cudaSuccess) return e;
    const int32_t rows = d.T * (d.mode == QLI_CAND_SOURCE ? 2 : 1);
    e = launch_pdl(fast_select_kernel, dim3(static_cast<unsigned>(rows)), dim3(kFT),
                   sizeof(FastSmem), s, d);
    if (e != cudaSuccess) return e;
  }
  if (d.lchunks > 0) {
    const dim3 g(static_cast<unsigned>(d.lchunks), static_cast<unsigned>(d.T),
                 d.mode == QLI_CAND_SOURCE ? 2u : 1u);
    if (d.fhist == nullptr) {   // no score-stage histogram: build the statistics here
      e = cudaMemsetAsync(d.lext, 0, d.long_zero_bytes, s);
      if (e != cudaSuccess) return e;
      lstat_kernel<<<g, kThreads, 0, s>>>(d);
      lhist_kernel<<<g, kThreads, 0, s>>>(d);
    }
    static std::atomic<uint64_t> lc_done{0};
    e = ensure_smem_limit(reinterpret_cast<const void*>(lcompact_kernel), 4 * kLongChunk, lc_done);
    if (e != cudaSuccess) return e;
    if (d.fhist != nullptr) {
      e = launch_pdl(lcompact_kernel, g, dim3(kThreads), 4 * kLongChunk, s, d);
      if (e != cudaSuccess) return e;
    } else {
      lcompact_kernel<<<g, kThreads, 4 * kLongChunk, s>>>(d);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t longest = d.Lrow > d.Brow ? d.Lrow : d.Brow;
  const int32_t cap = static_cast<int32_t>(longest < kSmemKeys ? longest : kSmemKeys);
  // candidate rows need room for kLongCandCap keys and ids
  const int32_t region = d.lchunks > 0 ? (cap > 2 * kLongCandCap ? cap : 2 * kLongCandCap) : cap;
  const int smem = 4 * (region + kHeadWords + kCandCap);
  if (d.fhist == nullptr && d.mode != QLI_CAND_CONSUMER) {
    // rows without a score-stage histogram: the many-rows-per-SM pass, then
    // the general selection for the rows it listed
    static std::atomic<uint64_t> done_list{0};
    e = ensure_smem_limit(reinterpret_cast<const void*>(select_list_kernel),
                          4 * (kSmemKeys + kHeadWords + kCandCap), done_list);
    if (e != cudaSuccess) return e;
    e = launch_pdl(select_list_kernel, dim3(static_cast<unsigned>(d.num_sms)), dim3(kThreads),
                   static_cast<size_t>(smem), s, d, cap, region);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  static std::atomic<uint64_t> done[4] = {{0}, {0}, {0}, {0}};
  void (*const kernels[4])(DevArgs, int32_t, int32_t) = {
      select_kernel<false, false>, select_kernel<false, true>, select_kernel<true, false>,
      select_kernel<true, true>};
  const int which = (d.fhist != nullptr ? 2 : 0) + (d.mode == QLI_CAND_CONSUMER ? 1 : 0);
  e = ensure_smem_limit(reinterpret_cast<const void*>(kernels[which]),
                        4 * (kSmemKeys + kHeadWords + kCandCap), done[which]);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(d.T), d.mode == QLI_CAND_SOURCE ? 2u : 1u);
  e = launch_pdl(kernels[which], grid, dim3(kThreads), static_cast<size_t>(smem), s, d, cap,
                 region);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int select_launches(const DevArgs& d) {
  if (d.T == 0) return 0;
  const int fast = (d.fhist == nullptr && d.mode != QLI_CAND_CONSUMER) ? 1 : 0;
  if (d.lchunks == 0) return 1 + fast;
  return (d.fhist != nullptr ? 2 : 4) + fast;
}

}  // namespace qli
