// Sparse attention over the positions the indexer selected (the compressed
// attention stage that consumes the indices).
//
// Sources (web pages): blog "DeepSeek V4.1-Flash 登陆昇腾 · 需求故事（PR 16925）",
// section 四 (the attention forward feeds the indexer's compressed indices to
// the sparse attention and inverse-rotates the output's tail in place);
// guide "DeepSeek V4.1 QLI V2 与候选集成", section 编译范围 (BF16 TND queries
// over the PA_BBND paged cache, a single-KV-head specialisation); section
// 数据流 and the blog's page packing (KV rows first in each page row).
// Readings: one shared KV head, 512 BF16 values (1024 bytes) per compressed
// position at kv_offset + row * 1024 of its page, serving as key and value;
// for token t, head h and the listed positions J (-1 skipped):
//   s_j = scale * q[t,h,:] . kv_j,  o = softmax(s) . kv,  lse = log sum exp s.
//
// One CTA per (token, group of 32 heads); 7 warps. The listed positions are
// taken 32 at a time (a chunk: 32 rows of 1 KB), five chunks in flight:
//   warps 0-1  gather: the group's queries, then each chunk's KV rows with
//              16-byte cp.async copies (every row lives in its own page, so no
//              tensor map fits), coalesced 512 bytes per warp instruction,
//              into a 128-byte-swizzled layout whose 128 rows are the pairs
//              (quarter of the 512 values, position)
//   warp 2     TMEM allocation and the MMA issuer (tcgen05, BF16, FP32 in
//              TMEM). Scores: M = 128 rows (quarter e, position p) x N = 128
//              (quarter e', head) x K = 128 values of the quarter, against
//              the queries stacked by quarter, so the block e = e' holds the
//              quarter's partial dot products; the four blocks sum to S.
//              Values: O^T[e] += V^T . P^T per quarter (M = 128 values,
//              N = 64: 32 heads and 32 zero columns, K = 32 positions), from
//              the same chunk read MN-major. Scores of chunk n+1 run while
//              chunk n's softmax does
//   warps 3-6  softmax: warp e loads quarter e's block (lane = position),
//              the blocks are summed in shared memory, warp w then owns heads
//              8w..8w+7 for the chunk's 32 positions: maxima by warp
//              shuffles, an online softmax that rescales O^T only when a
//              head's maximum grows by more than kRescale (the stale maximum
//              keeps every weight below e^kRescale), P^T as BF16; at the end
//              O / l and the LSE
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "qli_internal.h"
#include "qli_ptx.cuh"

namespace qli {
namespace attn {
namespace {

constexpr int kD = 512;                    // values per KV row
constexpr int kRowBytes = kD * 2;
constexpr int kHeads = 32;                 // heads per CTA
constexpr int kCP = 32;                    // positions per chunk
constexpr int kChunkBytes = kCP * kRowBytes;       // 32 KB
constexpr int kRegionBytes = 128 * 128;    // 128 rows x 64 values (BF16)
constexpr int kSlots = 5;                  // chunk ring
constexpr int kQBytes = 2 * kRegionBytes;  // 128 rows (quarter, head) x 128 values
constexpr int kPBytes = kCP * 128;         // 32 positions x 64 heads (BF16)
constexpr int kThreads = 224;
constexpr int kGatherThreads = 64;
constexpr int kEpiWarp0 = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;              // two score buffers of 128 columns
constexpr uint32_t kOCol = 256;            // O^T: 4 quarters x 64 columns
constexpr float kRescale = 8.0f;           // natural-log slack before O is rescaled
constexpr float kLog2e = 1.4426950408889634f;

struct Smem {
  uint8_t kv[kSlots][kChunkBytes];         // 1024-aligned
  uint8_t q[kQBytes];                      // 1024-aligned
  uint8_t p[2][kPBytes];                   // 1024-aligned, by chunk parity
  float xs[4][kCP][33];                    // quarter blocks of the scores (padded rows)
  float alpha[kHeads];
  float mfin[kHeads], lfin[kHeads];
  int32_t chflag[4];
  int32_t slot[qli::kMaxTopK];             // listed entry -> page * R + row, -1: skipped
  uint64_t full[kSlots], empty[kSlots], qfull, tfull, sfull[2], pready[2], pvdone, ofull;
  uint32_t tmem_base;
};
constexpr int kSmemBytes = static_cast<int>(sizeof(Smem)) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "attention kernel shared memory");

struct Args {
  const uint16_t* q;
  int64_t q_st, q_sh;
  int32_t T, H, B;
  const int32_t* cu;
  const uint8_t* cache;
  int64_t page_stride, num_pages, kv_off;
  int32_t R;
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* idx;
  int32_t K;
  float scale;
  uint16_t* out;
  int64_t o_st, o_sh;
  float* lse;
  uint32_t* err;
};

// Instruction descriptor, kind::f16 with BF16 A and B, FP32 D, M = 128,
// N = n; a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// Shared-memory descriptor with the 128-byte swizzle and explicit leading /
// stride byte offsets. K-major: SBO = 1024 between 8-row groups (LBO unused).
// MN-major: LBO = bytes between 64-value atoms along M or N, SBO = bytes
// between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Byte offset of 16-byte unit u (values 8u..8u+7 of a 64-value atom row) of
// row r in a 128-byte-swizzled region.
__device__ __forceinline__ uint32_t sw(uint32_t r, uint32_t u) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((u ^ (r & 7u)) << 4);
}

// 2^x by the SFU's approximation (ex2.approx.ftz: a few ulp; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Position j of request b as page * R + row, or -1 when j is negative, lies
// outside the block table or names a page outside the pool (the last two
// flagged).
__device__ __forceinline__ int32_t slot_of(const Args& a, int32_t b, int32_t j, bool& bad) {
  if (j < 0) return -1;
  if (static_cast<int64_t>(j) >= static_cast<int64_t>(a.bt_stride) * a.R) {
    bad = true;
    return -1;
  }
  const int32_t page = __ldg(a.bt + static_cast<int64_t>(b) * a.bt_stride + j / a.R);
  if (page < 0 || page >= a.num_pages) {
    bad = true;
    return -1;
  }
  return page * a.R + j % a.R;
}

__global__ void __launch_bounds__(kThreads, 1) attn_kernel(Args a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y, h0 = blockIdx.x * kHeads;
  const int nchunks = (a.K + kCP - 1) / kCP;

  if (warp == 2) tmem_alloc(&S.tmem_base, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&S.full[s], kGatherThreads);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.qfull, kGatherThreads);
    mbar_init(&S.tfull, kGatherThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.sfull[s], 1);
      mbar_init(&S.pready[s], 4);
    }
    mbar_init(&S.pvdone, 1);
    mbar_init(&S.ofull, 1);
    fence_mbar_init();
  }
  // P^T columns 32..63 (padding heads) stay zero for the whole call
  if (warp >= kEpiWarp0 && tid - 32 * kEpiWarp0 < 2 * kCP) {
    const int r = tid - 32 * kEpiWarp0;
#pragma unroll
    for (int u = 4; u < 8; ++u)
      *reinterpret_cast<uint4*>(&S.p[r >> 5][sw(r & 31, u)]) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  // the token's request: the last b with cu[b] <= t
  int32_t b = 0;
  {
    int32_t lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (__ldg(a.cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  const int32_t* idx_row = a.idx + static_cast<int64_t>(t) * a.K;
  bool ok = true;

  if (warp < 2) {
    // ---------------- gather
    const int g = tid;                                   // 0..63
    const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(
        a.q + static_cast<int64_t>(t) * a.q_st + static_cast<int64_t>(h0) * a.q_sh);
    // queries: row (quarter e, head h) of the stacked operand holds values
    // 128e .. 128e+127 of head h
    for (int u = g; u < kHeads * (kD / 8); u += kGatherThreads) {
      const int h = u / (kD / 8), du = u % (kD / 8);
      const int e = du >> 4, kq = du & 15;
      cp16(&S.q[(kq >> 3) * kRegionBytes + sw(e * 32 + h, kq & 7)],
           qsrc + static_cast<int64_t>(h) * a.q_sh * 2 + du * 16, 16);
    }
    cp_arrive(&S.qfull);
    // the slot of every listed entry, once: all index loads first, then all
    // block-table loads, so the dependent round trips are paid once per call
    bool bad = false;
    {
      constexpr int kPer = qli::kMaxTopK / kGatherThreads;   // 32
      int32_t j[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = g + i * kGatherThreads;
        j[i] = e < a.K ? __ldg(idx_row + e) : -1;
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = g + i * kGatherThreads;
        if (e < a.K) S.slot[e] = slot_of(a, b, j[i], bad);
      }
    }
    mbar_arrive(&S.tfull);
    if (lane == 0) ok = mbar_wait_bounded(&S.tfull, 0);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    // lane l resolves row l of each chunk; a warp instruction copies 512
    // contiguous bytes of one row (units 32w .. 32w+31 of its 64)
    const auto row_addr = [&](int n) -> const uint8_t* {
      const int e = n * kCP + lane;
      const int32_t sl = (n < nchunks && e < a.K) ? S.slot[e] : -1;
      if (sl < 0) return nullptr;
      return a.cache + static_cast<int64_t>(sl / a.R) * a.page_stride + a.kv_off +
             static_cast<int64_t>(sl % a.R) * kRowBytes;
    };
    const int ur = warp * 32 + lane;                     // this lane's 16-byte unit of a row
    const int ue = ur >> 4, ukq = ur & 15;               // quarter, unit within the quarter
    const uint32_t dst_col = (ukq >> 3) * kRegionBytes;
    for (int n = 0; n < nchunks && ok; ++n) {
      const uint8_t* ptr = row_addr(n);
      const int s = n % kSlots;
      if (lane == 0) ok = mbar_wait_bounded(&S.empty[s], ((n / kSlots) & 1) ^ 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* dst = S.kv[s] + dst_col;
#pragma unroll 8
      for (int p = 0; p < kCP; ++p) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(ptr), p));
        cp16(dst + sw(ue * 32 + p, ukq & 7), src ? src + ur * 16 : a.cache, src ? 16u : 0u);
      }
      cp_arrive(&S.full[s]);
    }
    if (bad && a.err) atomicOr(a.err, QLI_DEVERR_PAGE);
    cp_wait_all();                                       // nothing in flight at exit
    if (!ok && lane == 0 && a.err) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  } else if (warp == 2) {
    // ---------------- MMA issuer: scores of chunk n, then values of chunk n-1
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(128, false, false);
      const uint32_t id_pv = idesc_bf16(64, true, true);
      const uint32_t qb = smem_u32(S.q);
      ok = mbar_wait_bounded(&S.qfull, 0);
      for (int n = 0; n <= nchunks && ok; ++n) {
        if (n < nchunks) {
          const int s = n % kSlots;
          if (!mbar_wait_bounded(&S.full[s], (n / kSlots) & 1)) { ok = false; break; }
          fence_proxy_async_smem();                      // cp.async writes -> tensor core
          tc_fence_after();
          const uint32_t kvb = smem_u32(S.kv[s]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t r = kk >> 2, koff = (kk & 3) * 32;
            mma_f16_ss(tmem + kSCol + (n & 1) * 128,
                       sdesc_sw128(kvb + r * kRegionBytes + koff, 16, 1024),
                       sdesc_sw128(qb + r * kRegionBytes + koff, 16, 1024), id_qk, kk ? 1u : 0u);
          }
          mma_commit(&S.sfull[n & 1]);
        }
        if (n >= 1) {
          const int m = n - 1, s = m % kSlots;
          if (!mbar_wait_bounded(&S.pready[m & 1], (m >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kvb = smem_u32(S.kv[s]), pb = smem_u32(S.p[m & 1]);
#pragma unroll
          for (int kk = 0; kk < kCP / 16; ++kk) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              mma_f16_ss(tmem + kOCol + e * 64,
                         sdesc_sw128(kvb + e * 4096 + kk * 2048, kRegionBytes, 1024),
                         sdesc_sw128(pb + kk * 2048, 1024, 1024), id_pv, (m | kk) ? 1u : 0u);
          }
          mma_commit(&S.empty[s]);
          mma_commit(&S.pvdone);
        }
      }
      mma_commit(&S.ofull);                              // every MMA of the CTA is done
      (void)mbar_wait_drain(&S.ofull, 0);
      if (!ok && a.err) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- softmax and output
    // Every epilogue warp runs the same sequence of named barriers whatever
    // happens: a wait that gives up clears `ok`, later waits are skipped and
    // the remaining chunks are run through on whatever TMEM holds (the call
    // then reports QLI_DEVERR_TIMEOUT and its outputs are not written).
    const int qw = warp & 3;                             // TMEM lane quarter / quarter of values
    const int ew = warp - kEpiWarp0;                     // 0..3: heads 8ew .. 8ew+7
    const uint32_t lane_addr = static_cast<uint32_t>(32 * qw) << 16;
    float m_used[8], l_part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      m_used[j] = -INFINITY;
      l_part[j] = 0.0f;
    }
    const float sl2 = a.scale * kLog2e;
    if (!mbar_wait_warp(&S.tfull, 0)) ok = false;       // the slot table is written
    for (int n = 0; n < nchunks; ++n) {
      const int e_idx = n * kCP + lane;
      const bool valid = e_idx < a.K && S.slot[e_idx] >= 0;
      if (ok && !mbar_wait_warp(&S.sfull[n & 1], (n >> 1) & 1)) ok = false;
      tc_fence_after();
      {
        // block (quarter qw, quarter qw): this position's partial dots of 32 heads
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + lane_addr + kSCol + (n & 1) * 128 + 32 * qw, r);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 32; ++h) S.xs[qw][lane][h] = __uint_as_float(r[h]);
      }
      named_bar(1, 128);
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int h = 8 * ew + j;
        const float sc = (S.xs[0][lane][h] + S.xs[1][lane][h]) + (S.xs[2][lane][h] + S.xs[3][lane][h]);
        x[j] = valid ? sc * sl2 : -INFINITY;
      }
      // per-head maxima over the chunk's 32 positions (the eight shuffle
      // chains side by side), then each head's decision, branch-free: the
      // reference maximum moves only when the chunk's exceeds it by more
      // than kRescale (or on the first positions the head sees)
      float mt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mt[j] = x[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) mt[j] = fmaxf(mt[j], __shfl_xor_sync(0xffffffffu, mt[j], o));
      }
      bool changed = false;
      float alpha[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool up = mt[j] > m_used[j] + kRescale * kLog2e;   // false while mt is -inf
        alpha[j] = up ? ex2(m_used[j] - mt[j]) : 1.0f;           // 0 when m_used was -inf
        m_used[j] = up ? mt[j] : m_used[j];
        changed |= up;
      }
      if (lane < 8) {
        float al = alpha[0];
#pragma unroll
        for (int j = 1; j < 8; ++j) al = lane == j ? alpha[j] : al;
        S.alpha[8 * ew + lane] = al;
      }
      if (lane == 0) S.chflag[ew] = changed ? 1 : 0;
      named_bar(1, 128);                                 // scores read, alphas published
      const bool rescale = n > 0 && (S.chflag[0] | S.chflag[1] | S.chflag[2] | S.chflag[3]) != 0;
      uint32_t pk[4];
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float pa = x[j] == -INFINITY ? 0.0f : ex2(x[j] - m_used[j]);
        const float pb = x[j + 1] == -INFINITY ? 0.0f : ex2(x[j + 1] - m_used[j + 1]);
        l_part[j] = l_part[j] * alpha[j] + pa;
        l_part[j + 1] = l_part[j + 1] * alpha[j + 1] + pb;
        const __nv_bfloat162 pp = __floats2bfloat162_rn(pa, pb);
        pk[j / 2] = *reinterpret_cast<const uint32_t*>(&pp);
      }
      *reinterpret_cast<uint4*>(&S.p[n & 1][sw(lane, ew)]) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      if (rescale) {
        // O^T (lane = value, column = head) times each head's alpha, once the
        // values of the previous chunk are accumulated
        if (ok && !mbar_wait_warp(&S.pvdone, (n - 1) & 1)) ok = false;
        tc_fence_after();
#pragma unroll 1
        for (int e = 0; e < 4; ++e) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tmem + lane_addr + kOCol + e * 64, o);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 32; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * S.alpha[h]);
          tmem_st_32x32b_x32(tmem + lane_addr + kOCol + e * 64, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();                          // P^T -> tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pready[n & 1]);
    }
    // totals of this warp's heads (sum over the 32 positions of each chunk)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        S.lfin[8 * ew + j] = l_part[j];
        S.mfin[8 * ew + j] = m_used[j];
      }
    }
    named_bar(1, 128);
    if (ok && !mbar_wait_warp(&S.ofull, 0)) ok = false;
    tc_fence_after();
    if (ok) {
      if (ew == 0 && a.lse) {
        const float l = S.lfin[lane];
        a.lse[static_cast<int64_t>(t) * a.H + h0 + lane] =
            l > 0.0f ? (S.mfin[lane] + log2f(l)) * (1.0f / kLog2e) : -INFINITY;
      }
      float inv_l[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) inv_l[h] = S.lfin[h] > 0.0f ? 1.0f / S.lfin[h] : 0.0f;
      uint16_t* orow = a.out + static_cast<int64_t>(t) * a.o_st + static_cast<int64_t>(h0) * a.o_sh;
#pragma unroll 1
      for (int e = 0; e < 4; ++e) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_addr + kOCol + e * 64, o);
        tmem_ld_wait();
        const int v = e * 128 + 32 * qw + lane;          // value of this TMEM lane
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(o[h]) * inv_l[h]);
          orow[static_cast<int64_t>(h) * a.o_sh + v] = *reinterpret_cast<const uint16_t*>(&bv);
        }
      }
    }
    if (!ok && lane == 0 && a.err) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

std::atomic<uint64_t> g_smem_attn{0};

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

}  // namespace
}  // namespace attn
}  // namespace qli

extern "C" qli_status qli_sparse_attention(const qli_attn_args* a, void* stream) {
  using namespace qli::attn;
  if (a == nullptr) return QLI_ERR_INVALID_ARG;
  if (a->D != kD || a->H < kHeads || a->H % kHeads != 0 || a->H > 128) return QLI_ERR_UNSUPPORTED;
  if (a->rows_per_page != 64 && a->rows_per_page != 128) return QLI_ERR_UNSUPPORTED;
  if (a->T < 0 || a->B < 0 || (a->B == 0 && a->T != 0)) return QLI_ERR_INVALID_ARG;
  if (a->K < 1 || a->K > qli::kMaxTopK) return QLI_ERR_INVALID_ARG;
  if (!(a->scale == a->scale) || std::isinf(a->scale)) return QLI_ERR_INVALID_ARG;
  if (a->T == 0) return QLI_OK;
  if (a->q == nullptr || a->cu_seqlens_q == nullptr || a->cache == nullptr ||
      a->block_table == nullptr || a->indices == nullptr || a->out == nullptr)
    return QLI_ERR_INVALID_ARG;
  if (a->num_pages > (int64_t{1} << 24)) return QLI_ERR_UNSUPPORTED;   // page * R fits 31 bits
  if (a->bt_stride < 1 || a->num_pages < 1 || a->page_stride <= 0 || a->kv_offset < 0 ||
      a->kv_offset + static_cast<int64_t>(a->rows_per_page) * kRowBytes > a->page_stride)
    return QLI_ERR_INVALID_ARG;
  if (a->q_stride_h < kD || a->q_stride_t < static_cast<int64_t>(a->H) * kD ||
      a->out_stride_h < kD || a->out_stride_t < static_cast<int64_t>(a->H) * kD)
    return QLI_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || a->q_stride_t % 8 || a->q_stride_h % 8 || !aligned(a->cache, 16) ||
      a->page_stride % 16 || a->kv_offset % 16 || !aligned(a->out, 2) ||
      !aligned(a->cu_seqlens_q, 4) || !aligned(a->block_table, 4) || !aligned(a->indices, 4) ||
      (a->lse && !aligned(a->lse, 4)) || (a->err_word && !aligned(a->err_word, 4)))
    return QLI_ERR_ALIGNMENT;
  int sms = 0;
  qli_status st = qli::device_sms(&sms);
  if (st != QLI_OK) return st;
  Args d{};
  d.q = a->q;
  d.q_st = a->q_stride_t;
  d.q_sh = a->q_stride_h;
  d.T = a->T;
  d.H = a->H;
  d.B = a->B;
  d.cu = a->cu_seqlens_q;
  d.cache = a->cache;
  d.page_stride = a->page_stride;
  d.num_pages = a->num_pages;
  d.kv_off = a->kv_offset;
  d.R = a->rows_per_page;
  d.bt = a->block_table;
  d.bt_stride = a->bt_stride;
  d.idx = a->indices;
  d.K = a->K;
  d.scale = a->scale;
  d.out = a->out;
  d.o_st = a->out_stride_t;
  d.o_sh = a->out_stride_h;
  d.lse = a->lse;
  d.err = a->err_word;
  cudaError_t e = qli::ensure_smem_limit(reinterpret_cast<const void*>(attn_kernel), kSmemBytes,
                                         g_smem_attn);
  if (e != cudaSuccess) return QLI_ERR_CUDA;
  attn_kernel<<<dim3(static_cast<unsigned>(a->H / kHeads), static_cast<unsigned>(a->T)), kThreads,
                kSmemBytes, static_cast<cudaStream_t>(stream)>>>(d);
  return cudaGetLastError() == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

extern "C" int64_t qli_attn_args_size(void) { return static_cast<int64_t>(sizeof(qli_attn_args)); }
