// Shared pieces of the selection: the selection row of a token (its scores,
// length and how many to keep) and the one-CTA-per-row ranking of rows that
// fit the candidate space (fast_row), used by the prefill selection kernel
// and by the single-launch path for small decode batches.
//
// Guide "DeepSeek V4.1 QLI V2 与候选集成", section 数据流: a token keeps its
// TopK positions in chronological order, padded with -1; in source mode also
// its best C-1 candidate blocks (ranked by block maximum) plus the last
// visible block. Ties rank by the lower position / block ID, with -0 == +0.
#pragma once

#include <cuda_fp16.h>

#include "qli_internal.h"
#include "qli_ptx.cuh"

namespace qli {
namespace {

// A row of the selection: entry s has a key (0 = not eligible) and an id.
struct Row {
  const float* vals;      // score row
  const int32_t* blocks;  // consumer: sorted candidate blocks (slot -> position)
  const uint32_t* cached; // keys in shared memory, or nullptr
  const int32_t* ids;     // candidate rows: the id of each cached key, or nullptr
  const int32_t* idx;     // sample-path candidates: entry s is row entry idx[s]
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
    const int32_t j = idx ? idx[s] : s;
    return cached ? cached[j] : key_from_global(j);
  }
  __device__ __forceinline__ int32_t id(int32_t s) const {
    if (ids) return ids[s];
    const int32_t j = idx ? idx[s] : s;
    return consumer ? blocks[j / kBlock] * kBlock + (j & (kBlock - 1)) : j;
  }
};

// Row 2t+which of the selection: which 0 = the token's positions (want K),
// which 1 = its source candidate blocks 0..nb-2 (want C-1; the last block is
// pinned separately). len 0 when there is nothing to rank.
__device__ __forceinline__ Row row_of(const DevArgs& a, int t, int which, int32_t V,
                                      int32_t owner, int32_t& want) {
  Row r;
  r.cached = nullptr;
  r.ids = nullptr;
  r.idx = nullptr;
  r.V = owner >= 0 ? V : 0;
  if (which == 0) {
    r.consumer = a.mode == QLI_CAND_CONSUMER;
    r.vals = a.scores + static_cast<int64_t>(t) * a.Lrow;
    r.blocks = r.consumer ? a.cand_list + static_cast<int64_t>(t) * a.C : nullptr;
    r.len = r.consumer ? (owner >= 0 ? a.cand_cnt[t] * kBlock : 0) : r.V;
    want = a.topk;
  } else {
    const int32_t nb = (r.V + kBlock - 1) / kBlock;
    r.consumer = false;
    r.vals = a.bscores + static_cast<int64_t>(t) * a.Brow;
    r.blocks = nullptr;
    r.len = nb > a.C ? nb - 1 : 0;
    want = a.C - 1;
  }
  return r;
}

// The same, with V(t) and the owner read from the planning stage's output.
__device__ __forceinline__ Row row_of(const DevArgs& a, int t, int which, int32_t& want) {
  return row_of(a, t, which, a.tok_V[t], a.tok_b[t], want);
}

// ---------------------------------------------------------------------------
// Rows without a score-stage histogram (the prefill path): one 256-thread
// CTA per row, four resident on each SM; index rows first, then candidate
// rows, the latest tokens first (the score stage wrote their rows last, so
// they are the likeliest to still be in L2). Each row is read from HBM once.
//
// A row longer than the candidate space first draws a sample of 1024 entries
// (16 evenly spread runs of 64); the key of a rank a little past the expected
// rank of the want-th best in the sample gives a provisional threshold. One
// pass over the row keeps every entry at or above it, compared as floats
// (slots claimed per warp step of 1024 entries, in no particular order), and
// counts the top 12 bits of the kept keys. An exact radix select on the
// candidates (digits of 12, 10 and 10 bits) finds the want-th best key; the
// winners are marked in position bitmaps, and one ordered scan of the bitmaps
// writes them in ascending order (equal keys at the threshold by lower
// position). Histograms hold two 16-bit counts per word. Where the sample
// misjudged the row (the pass kept fewer than `want` or more than kFCap
// entries) the sample rank is scaled by what the pass kept and the pass runs
// once more. A row this path cannot finish (longer than kFMaxLen entries, or
// misjudged twice) is appended to a list for the general selection
// (select_list_kernel), which ranks it exactly.
constexpr int kFT = 256;
constexpr int kFW = kFT / 32;
constexpr int kFPerSM = 4;                         // resident CTAs per SM
constexpr int kFCap = 4608;                        // candidates a row may keep
constexpr int kFMaxLen = kSmemKeys;                // longest row this path takes
constexpr int kBitWords = (kFMaxLen + 31) / 32;    // one bit per position of a row
constexpr int kSample = 1024;
constexpr int kFB = 8;                             // float4 loads per lane and step
constexpr int kFStep = 128 * kFB;                  // entries a warp covers per step
static_assert(kFMaxLen <= 65536, "candidate positions are 16-bit");
static_assert(kFCap < 65536 && kSample < 65536, "histogram counts are 16-bit");
static_assert(kFB * 4 <= 32, "one mask bit per entry of a lane's step");

struct FastSmem {
  uint32_t shist[kHistBins / 2];   // the sample's top 12 key bits; then the 10-bit digits
  uint32_t h0[kHistBins / 2];      // the candidates' top 12 key bits
  uint32_t gtb[kBitWords];         // winners above the threshold key, by position
  uint32_t eqb[kBitWords];         // winners at the threshold key
  uint32_t ckey[kFCap];            // candidate keys (slot = position when a row fits)
  uint16_t cpos[kFCap];            // candidate positions (rows that were sampled)
  uint32_t wtot[kFW];
  uint32_t cnt;                    // candidates claimed
  uint32_t sel[4];
};

__device__ __forceinline__ void hist16_add(uint32_t* h, uint32_t bin) {
  atomicAdd(&h[bin >> 1], 1u << ((bin & 1u) << 4));
}

// The smallest score whose key is at least `key` (the inverse of order_key
// on a bin boundary). Below the key of -FLT_MAX every score qualifies: -inf.
__device__ __forceinline__ float key_floor(uint32_t key) {
  if (key < 0x00800000u) return -INFINITY;
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Inclusive scan over the CTA's 256 threads of one value each; `total` gets
// the sum. One barrier: F.wtot is rewritten only after a later barrier.
__device__ __forceinline__ uint32_t fast_scan(uint32_t v, uint32_t& total, FastSmem& F) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) F.wtot[warp] = incl;
  __syncthreads();
  uint32_t before = 0u, tot = 0u;
#pragma unroll
  for (int w = 0; w < kFW; ++w) {
    const uint32_t x = F.wtot[w];
    tot += x;
    before += w < warp ? x : 0u;
  }
  total = tot;
  return incl + before;
}

// The digit (from the top) of a packed histogram of kBins bins at which the
// running count reaches k (1 <= k <= the histogram's total): its value, the
// count above it and its own count, in F.sel[0..2] after the second barrier.
// Thread i holds bins kBins-1-kPer*i down to kBins-kPer*(i+1).
template <int kBins>
__device__ __forceinline__ void fast_pick(const uint32_t* hist, uint32_t k, FastSmem& F) {
  constexpr int kPer = kBins / kFT;
  static_assert(kPer == 16 || kPer == 4, "one or two 16-byte loads per thread");
  const int lo = kBins - kPer * (static_cast<int>(threadIdx.x) + 1);
  uint32_t w[kPer / 2];
  if constexpr (kPer == 16) {
    const uint4 a = reinterpret_cast<const uint4*>(hist + lo / 2)[0];
    const uint4 b = reinterpret_cast<const uint4*>(hist + lo / 2)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else {
    const uint2 a = reinterpret_cast<const uint2*>(hist + lo / 2)[0];
    w[0] = a.x; w[1] = a.y;
  }
  // the packed words add up without carries: a histogram's total is below 2^16
  uint32_t sum = 0u;
#pragma unroll
  for (int i = 0; i < kPer / 2; ++i) sum += w[i];
  const uint32_t mine = (sum & 0xffffu) + (sum >> 16);
  uint32_t tot;
  const uint32_t incl = fast_scan(mine, tot, F);
  uint32_t above = incl - mine;
  if (above < k && k <= incl) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {   // j-th bin from this thread's top
      const int i = kPer - 1 - j;
      const uint32_t c = (w[i >> 1] >> ((i & 1) << 4)) & 0xffffu;
      if (above + c >= k) {
        F.sel[0] = static_cast<uint32_t>(lo + i);
        F.sel[1] = above;
        F.sel[2] = c;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void enlist(const DevArgs& a, int t, int which) {
  if (threadIdx.x == 0) {
    const uint32_t i = atomicAdd(a.counter, 1u);
    a.flist[i] = 2 * t + which;
  }
}

// Row r of the walk: index rows first, then candidate rows; latest token first.
__device__ __forceinline__ void fast_row_id(const DevArgs& a, int32_t r, int& t, int& which) {
  which = r >= a.T ? 1 : 0;
  t = a.T - 1 - (which ? r - a.T : r);
}

// One row; every thread of the CTA calls it, and every decision that skips a
// barrier is block-uniform. V and owner are token t's visible count and
// request (-1: none).
__device__ __forceinline__ void fast_row(const DevArgs& a, int t, int which, int32_t V,
                                         int32_t owner, FastSmem& F) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool blocks = which == 1;
  const int32_t width = blocks ? a.C : a.topk;
  int32_t* out = blocks ? a.cand_out + static_cast<int64_t>(t) * a.C
                        : a.idx_out + static_cast<int64_t>(t) * a.topk;
  int32_t want;
  const Row r = row_of(a, t, which, V, owner, want);
  const int32_t nb = (r.V + kBlock - 1) / kBlock;
  const int32_t len = r.len;
  int32_t written = 0;
  if (len > kFMaxLen) {
    enlist(a, t, which);
    return;
  }
  if (blocks && len == 0) {
    // at most C visible blocks: all of them, in order
    for (int c = tid; c < nb; c += kFT) out[c] = c;
    written = nb;
  } else if (len <= want) {
    // every entry is selected (all entries of these rows are eligible)
    for (int s = tid; s < len; s += kFT) out[s] = s;
    written = len;
    if (blocks) {
      if (tid == 0) out[written] = nb - 1;            // the pinned last visible block
      written += 1;
    }
  } else {
    const float4* v4 = reinterpret_cast<const float4*>(r.vals);
    const bool sampled = len > kFCap;
    // ---- the sample's loads go out first; the shared state is cleared meanwhile
    const int32_t s0 = static_cast<int32_t>((static_cast<int64_t>(len) * (tid >> 4) / 16) & ~3LL) +
                       4 * (tid & 15);
    float4 sf = make_float4(0.f, 0.f, 0.f, 0.f);
    if (sampled) sf = __ldcg(v4 + (s0 >> 2));
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(F.shist)[tid] = z4;
    reinterpret_cast<uint4*>(F.shist)[tid + kFT] = z4;
    reinterpret_cast<uint4*>(F.h0)[tid] = z4;
    reinterpret_cast<uint4*>(F.h0)[tid + kFT] = z4;
    const int32_t words = (len + 31) >> 5;
    for (int i = tid; i < words; i += kFT) {
      F.gtb[i] = 0u;
      F.eqb[i] = 0u;
    }
    if (tid == 0) F.cnt = 0u;
    __syncthreads();
    const float kNaN = __uint_as_float(0x7fffffffu);
    if (!sampled) {
      // ---- a row that fits keeps every entry in place: slot = position;
      // keys and their first digit straight from the row
      for (int32_t e0 = 4 * tid; e0 < len; e0 += 4 * kFT) {
        const float4 f = __ldcg(v4 + (e0 >> 2));
        const float fv[4] = {f.x, f.y, f.z, f.w};
        uint32_t k[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          k[j] = order_key(fv[j]);
          if (e0 + j < len) hist16_add(F.h0, hist_bin(k[j]));
        }
        *reinterpret_cast<uint4*>(F.ckey + e0) = make_uint4(k[0], k[1], k[2], k[3]);
      }
      if (tid == 0) F.cnt = static_cast<uint32_t>(len);
    } else {
      // ---- provisional threshold from the sample
      const float fv[4] = {sf.x, sf.y, sf.z, sf.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (s0 + j < len) hist16_add(F.shist, hist_bin(order_key(fv[j])));
      __syncthreads();
      // a rank 10% past the want-th best's expected sample rank, plus 24
      uint32_t rank = static_cast<uint32_t>(
          (static_cast<int64_t>(want) * kSample * 11) / (10 * static_cast<int64_t>(len))) + 24u;
      constexpr uint32_t kRankMax = static_cast<uint32_t>(kSample) - 64u;
      if (rank >= kRankMax) {   // block-uniform
        enlist(a, t, which);
        return;
      }
      const int32_t seg = ((len + kFW - 1) / kFW + 127) & ~127;
      const int32_t lo = warp * seg, hi = min(len, lo + seg);
      for (int attempt = 0;; ++attempt) {
        fast_pick<kHistBins>(F.shist, rank, F);
        // ---- one pass over the row: the position of every entry with a key
        // at or above the picked bin's, found by a float compare against the
        // smallest score of that key (NaN, which passes no compare, pads past
        // the end); warp w owns a contiguous segment (whole 128-entry rows,
        // its last step possibly partial), lane l entries 4l..4l+3 of each 128
        const float f_p = key_floor(F.sel[0] << (32 - kHistBits));
        for (int32_t b = lo; b < hi; b += kFStep) {
          float v[4 * kFB];
#pragma unroll
          for (int u = 0; u < kFB; ++u) {
            const int32_t e0 = b + 128 * u + 4 * lane;
            const float4 f = e0 < hi ? __ldcg(v4 + (e0 >> 2)) : make_float4(kNaN, kNaN, kNaN, kNaN);
            v[4 * u] = f.x;
            v[4 * u + 1] = f.y;
            v[4 * u + 2] = f.z;
            v[4 * u + 3] = f.w;
          }
          if (b + kFStep > hi) {                          // warp-uniform: a segment's ragged end
#pragma unroll
            for (int e = 0; e < 4 * kFB; ++e)
              if (b + 128 * (e >> 2) + 4 * lane + (e & 3) >= hi) v[e] = kNaN;
          }
          uint32_t m = 0u;
#pragma unroll
          for (int e = 0; e < 4 * kFB; ++e) m |= v[e] >= f_p ? (1u << e) : 0u;
          const uint32_t c = __popc(m);
          uint32_t incl = c;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
          if (tot == 0u) continue;                        // warp-uniform
          uint32_t base = 0u;
          if (lane == 31) base = atomicAdd(&F.cnt, tot);
          base = __shfl_sync(0xffffffffu, base, 31);
          // a row whose candidates overflow the room is listed, so a step
          // whose slots do not all fit writes none of them (warp-uniform)
          if (base + tot > static_cast<uint32_t>(kFCap)) continue;
          // positions only, one per kept entry; the scores are read again below
          uint32_t w = base + incl - c;
          const uint32_t lane_pos = static_cast<uint32_t>(b + 4 * lane);
          while (m) {
            const uint32_t e = static_cast<uint32_t>(__ffs(m) - 1);
            m &= m - 1u;
            F.cpos[w++] = static_cast<uint16_t>(lane_pos + 128u * (e >> 2) + (e & 3u));
          }
        }
        __syncthreads();
        // a threshold that kept fewer than `want` or more than kFCap entries
        // (the sample misjudged the row) is moved once: the rank is scaled by
        // what it kept, aiming at the middle of [want, kFCap]
        const uint32_t got = F.cnt;
        const bool fits = got >= static_cast<uint32_t>(want) && got <= static_cast<uint32_t>(kFCap);
        if (attempt > 0 || fits) break;                 // block-uniform
        const uint32_t aim = (static_cast<uint32_t>(want) + kFCap) / 2u;
        uint32_t r2 = got == 0u ? 2u * rank + 32u
                                : static_cast<uint32_t>(static_cast<uint64_t>(rank) * aim / got);
        r2 = min(max(r2, 1u), kRankMax);
        if (r2 == rank) break;
        rank = r2;
        __syncthreads();                                // every thread has read F.cnt
        if (tid == 0) F.cnt = 0u;                       // (fast_pick's barrier orders it)
      }
      // the sample's histogram becomes the 10-bit digits' (added to after
      // the barrier that follows the gather below)
      reinterpret_cast<uint4*>(F.shist)[tid] = z4;
      reinterpret_cast<uint4*>(F.shist)[tid + kFT] = z4;
      // ---- the kept scores again (from L2), as keys, and their first digit;
      // a row that overflowed the room (and so left slots unwritten) is
      // listed below instead
      const uint32_t nk = F.cnt <= static_cast<uint32_t>(kFCap) ? F.cnt : 0u;
      const float* vals = r.vals;
#pragma unroll 4
      for (uint32_t i = tid; i < nk; i += kFT) {
        const uint32_t key = order_key(__ldcg(vals + F.cpos[i]));
        F.ckey[i] = key;
        hist16_add(F.h0, hist_bin(key));
      }
    }
    __syncthreads();
    const uint32_t n = F.cnt;
    if (n > static_cast<uint32_t>(kFCap) || n < static_cast<uint32_t>(want)) {   // block-uniform
      enlist(a, t, which);
      return;
    }
    // ---- the want-th best key among the candidates: digits of 12, 10, 10 bits
    // winners: every key >= t_ge, and (when ranking reached the last digit
    // with keys to spare) need_eq keys equal to prefix, the lowest positions
    fast_pick<kHistBins>(F.h0, static_cast<uint32_t>(want), F);
    uint32_t prefix = F.sel[0] << (32 - kHistBits);
    int32_t k2 = want - static_cast<int32_t>(F.sel[1]);
    bool settled = F.sel[2] == static_cast<uint32_t>(k2);
    uint32_t t_ge = prefix;
    int32_t need_eq = 0;
    if (!settled) {
      const uint32_t top = prefix >> 20;
      for (uint32_t i = tid; i < n; i += kFT) {
        const uint32_t key = F.ckey[i];
        if ((key >> 20) == top) hist16_add(F.shist, (key >> 10) & 1023u);
      }
      __syncthreads();
      fast_pick<1024>(F.shist, static_cast<uint32_t>(k2), F);
      prefix |= F.sel[0] << 10;
      k2 -= static_cast<int32_t>(F.sel[1]);
      settled = F.sel[2] == static_cast<uint32_t>(k2);
      t_ge = prefix;
    }
    if (!settled) {
      const uint32_t top = prefix >> 10;
      for (uint32_t i = tid; i < n; i += kFT) {
        const uint32_t key = F.ckey[i];
        if ((key >> 10) == top) hist16_add(F.shist + 512, key & 1023u);
      }
      __syncthreads();
      fast_pick<1024>(F.shist + 512, static_cast<uint32_t>(k2), F);
      prefix |= F.sel[0];
      k2 -= static_cast<int32_t>(F.sel[1]);
      if (F.sel[2] == static_cast<uint32_t>(k2)) {
        t_ge = prefix;
      } else {
        // keys of finite scores stay below 0xff800000, so this cannot wrap
        t_ge = prefix + 1u;
        need_eq = k2;
      }
    }
    // ---- winners into the position bitmaps (cleared at the start)
    if (!sampled) {
      // slot = position: lane l of warp w holds bit l of word (i - lane) / 32
      for (uint32_t i0 = tid - lane; i0 < n; i0 += kFT) {
        const uint32_t i = i0 + lane;
        const uint32_t key = i < n ? F.ckey[i] : 0u;
        const uint32_t g = __ballot_sync(0xffffffffu, i < n && key >= t_ge);
        const uint32_t e = __ballot_sync(0xffffffffu, i < n && need_eq != 0 && key == prefix);
        if (lane == 0) {
          F.gtb[i0 >> 5] = g;
          F.eqb[i0 >> 5] = e;
        }
      }
    } else if (need_eq == 0) {
      for (uint32_t i = tid; i < n; i += kFT) {
        const uint32_t pos = F.cpos[i];
        if (F.ckey[i] >= t_ge) atomicOr(&F.gtb[pos >> 5], 1u << (pos & 31));
      }
    } else {
      for (uint32_t i = tid; i < n; i += kFT) {
        const uint32_t key = F.ckey[i];
        const uint32_t pos = F.cpos[i];
        if (key >= t_ge) atomicOr(&F.gtb[pos >> 5], 1u << (pos & 31));
        else if (key == prefix) atomicOr(&F.eqb[pos >> 5], 1u << (pos & 31));
      }
    }
    __syncthreads();
    // ---- ordered scan: consecutive threads own consecutive bit ranges of
    // the bitmaps, whole words (words/256 of them) when a row has at least
    // 256 words, otherwise 1/parts of a word; the counts of both bitmaps
    // travel as one packed scan (each below 2^16). The positions go to
    // shared memory in order (over the keys, no longer needed), then out in
    // coalesced stores.
    int32_t parts = 1;
    while (parts < 32 && words * parts * 2 <= kFT) parts *= 2;   // block-uniform
    int32_t w0, w1;
    uint32_t mask = 0xffffffffu;
    if (parts == 1) {
      const int32_t per = (words + kFT - 1) / kFT;
      w0 = min(words, tid * per);
      w1 = min(words, w0 + per);
    } else {
      const int32_t sb = 32 / parts;
      w0 = min(words, tid / parts);
      w1 = min(words, w0 + 1);
      mask = (0xffffffffu >> (32 - sb)) << ((tid % parts) * sb);
    }
    uint32_t cg = 0u, ce = 0u;
    for (int32_t w = w0; w < w1; ++w) {
      cg += __popc(F.gtb[w] & mask);
      ce += __popc(F.eqb[w] & mask);
    }
    uint32_t tot;
    const uint32_t mine = cg | (ce << 16);
    const uint32_t before = fast_scan(mine, tot, F) - mine;
    const uint32_t gt_tot = tot & 0xffffu, eq_tot = tot >> 16;
    const uint32_t ne = static_cast<uint32_t>(need_eq);
    uint32_t* const staged = F.ckey;
    const uint32_t cap = static_cast<uint32_t>(want);
    if (ne == 0u) {                                    // block-uniform
      uint32_t o = before & 0xffffu;
      for (int32_t w = w0; w < w1; ++w) {
        uint32_t bits = F.gtb[w] & mask;
        while (bits) {
          const uint32_t bpos = static_cast<uint32_t>(__ffs(bits) - 1);
          bits &= bits - 1u;
          if (o < cap) staged[o] = static_cast<uint32_t>(w) * 32u + bpos;
          ++o;
        }
      }
    } else {
      uint32_t eq_seen = before >> 16;
      uint32_t o = (before & 0xffffu) + min(eq_seen, ne);
      for (int32_t w = w0; w < w1; ++w) {
        const uint32_t g = F.gtb[w] & mask, e = F.eqb[w] & mask;
        uint32_t bits = g | e;
        while (bits) {
          const uint32_t bpos = static_cast<uint32_t>(__ffs(bits) - 1);
          bits &= bits - 1u;
          bool take = true;
          if (!((g >> bpos) & 1u)) {
            take = eq_seen < ne;
            ++eq_seen;
          }
          if (take) {
            if (o < cap) staged[o] = static_cast<uint32_t>(w) * 32u + bpos;
            ++o;
          }
        }
      }
    }
    written = min(static_cast<int32_t>(gt_tot + min(eq_tot, ne)), want);
    __syncthreads();
    for (int k = tid; k < written; k += kFT) out[k] = static_cast<int32_t>(staged[k]);
    if (blocks) {
      if (tid == 0) out[written] = nb - 1;            // the pinned last visible block
      written += 1;
    }
  }
  for (int k = written + tid; k < width; k += kFT) out[k] = -1;
}

}  // namespace
}  // namespace qli
