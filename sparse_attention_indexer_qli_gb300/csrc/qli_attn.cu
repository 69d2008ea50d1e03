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
// One CTA per (token, group of 32 heads); 7 warps:
//   warps 0-1  gather: the group's queries and, tile by tile, the KV rows of
//              128 listed positions, with 16-byte cp.async copies (each row
//              lives in its own page, so no tensor map fits) into 128-byte-
//              swizzled 32 KB chunks of 128 rows x 128 values (5-chunk ring)
//   warp 2     TMEM allocation and the MMA issuer (tcgen05, BF16, FP32
//              accumulators): S^T = KV_tile . Q^T (M = 128 positions, N = 32
//              heads, K = 512), then O^T += KV_tile^T . P^T (M = 128 values
//              per chunk, N = 64 (32 heads, zero padded), K = 128 positions),
//              reading the same swizzled chunks K-major and MN-major
//   warps 3-6  softmax: thread = position (TMEM lane); per-head tile maxima
//              by a transpose-reduction across lanes, an online softmax that
//              rescales O^T only when a head's maximum grows by more than
//              kRescale (the stale maximum keeps every weight below e^kRescale),
//              P^T as BF16 into shared memory; at the end O / l and the LSE.
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
constexpr int kTileRows = 128;             // positions per tile (MMA M of S^T)
constexpr int kChunkD = 128;               // values per chunk
constexpr int kChunks = kD / kChunkD;      // 4 chunks per tile
constexpr int kChunkBytes = kTileRows * kChunkD * 2;   // 32 KB
constexpr int kRegionBytes = kTileRows * 128;          // 64 values x 128 rows
constexpr int kSlots = 5;                  // chunk ring
constexpr int kQRegion = kHeads * 128;     // 64 values x 32 heads
constexpr int kQBytes = kHeads * kD * 2;   // 32 KB
constexpr int kPBytes = kTileRows * 128;   // 128 positions x 64 heads (BF16)
constexpr int kThreads = 224;
constexpr int kGatherThreads = 64;
constexpr int kEpiWarp0 = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;              // S^T: 32 columns
constexpr uint32_t kOCol = 64;             // O^T: 4 chunks x 64 columns
constexpr float kRescale = 8.0f;           // natural-log slack before O is rescaled
constexpr float kLog2e = 1.4426950408889634f;

struct Smem {
  uint8_t kv[kSlots][kChunkBytes];         // 1024-aligned
  uint8_t q[kQBytes];                      // 1024-aligned
  uint8_t p[kPBytes];                      // 1024-aligned
  const uint8_t* rowptr[kTileRows];        // this tile's row addresses (nullptr: zero row)
  float red[4][32];
  uint64_t full[kSlots], empty[kSlots], qfull, sfull, pready, ofull;
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

// v[0..31] of each lane -> lane L returns op over the warp's lanes of v[L].
// Five exchange rounds: each lane keeps half of its values and combines them
// with the partner's copy of that half.
template <class Op>
__device__ __forceinline__ float transpose_reduce(float (&v)[32], Op op) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = upper ? v[j] : v[j + w];
      const float keep = upper ? v[j + w] : v[j];
      v[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, w));
    }
  }
  return v[0];
}

// The address of position j's KV row for request b, or nullptr when j lies
// outside the block table or names a page outside the pool (flagged).
__device__ __forceinline__ const uint8_t* row_of(const Args& a, int32_t b, int32_t j, bool& bad) {
  if (j < 0) return nullptr;
  if (static_cast<int64_t>(j) >= static_cast<int64_t>(a.bt_stride) * a.R) {
    bad = true;
    return nullptr;
  }
  const int32_t page = __ldg(a.bt + static_cast<int64_t>(b) * a.bt_stride + j / a.R);
  if (page < 0 || page >= a.num_pages) {
    bad = true;
    return nullptr;
  }
  return a.cache + static_cast<int64_t>(page) * a.page_stride + a.kv_off +
         static_cast<int64_t>(j % a.R) * kRowBytes;
}

__global__ void __launch_bounds__(kThreads, 1) attn_kernel(Args a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y, h0 = blockIdx.x * kHeads;
  const int ntiles = (a.K + kTileRows - 1) / kTileRows;

  if (warp == 2) tmem_alloc(&S.tmem_base, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&S.full[s], kGatherThreads);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.qfull, kGatherThreads);
    mbar_init(&S.sfull, 1);
    mbar_init(&S.pready, 4);
    mbar_init(&S.ofull, 1);
    fence_mbar_init();
  }
  // P^T columns 32..63 (padding heads) stay zero for the whole call
  if (warp >= kEpiWarp0) {
    const int p = tid - 32 * kEpiWarp0;
#pragma unroll
    for (int u = 4; u < 8; ++u) *reinterpret_cast<uint4*>(&S.p[sw(p, u)]) = make_uint4(0, 0, 0, 0);
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
    for (int u = g; u < kHeads * (kD / 8); u += kGatherThreads) {
      const int h = u / (kD / 8), du = u % (kD / 8);
      cp16(&S.q[(du >> 3) * kQRegion + sw(h, du & 7)],
           qsrc + static_cast<int64_t>(h) * a.q_sh * 2 + du * 16, 16);
    }
    cp_arrive(&S.qfull);
    // lanes 0-15 and 16-31 of a warp copy two rows' 256-byte chunk pieces
    // per instruction (coalesced); warp w copies rows 4k + 2w + half, whose
    // addresses its own lanes look up (lane k: rows 4k + 2w and 4k + 2w + 1),
    // so the two gather warps never wait on each other
    const int half = lane >> 4, u = lane & 15;
    bool bad = false;
    for (int i = 0; i < ntiles && ok; ++i) {
      __syncwarp();                                      // the last tile's copies are issued
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int p = 4 * lane + 2 * warp + hh;
        const int e = i * kTileRows + p;
        S.rowptr[p] = e < a.K ? row_of(a, b, __ldg(idx_row + e), bad) : nullptr;
      }
      __syncwarp();
      for (int c = 0; c < kChunks; ++c) {
        const int n = i * kChunks + c, s = n % kSlots;
        if (lane == 0) ok = mbar_wait_bounded(&S.empty[s], ((n / kSlots) & 1) ^ 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        uint8_t* dst = S.kv[s];
#pragma unroll 4
        for (int k = 0; k < kTileRows / 4; ++k) {
          const int p = 4 * k + 2 * warp + half;
          const uint8_t* src = S.rowptr[p];
          cp16(dst + (u >> 3) * kRegionBytes + sw(p, u & 7),
               src ? src + c * (kChunkD * 2) + u * 16 : a.cache, src ? 16u : 0u);
        }
        cp_arrive(&S.full[s]);
      }
    }
    if (bad && a.err) atomicOr(a.err, QLI_DEVERR_PAGE);
    cp_wait_all();                                       // nothing in flight at exit
    if (!ok && lane == 0 && a.err) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  } else if (warp == 2) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(kHeads, false, false);
      const uint32_t id_pv = idesc_bf16(64, true, true);
      const uint32_t qb = smem_u32(S.q), pb = smem_u32(S.p);
      ok = mbar_wait_bounded(&S.qfull, 0);
      for (int i = 0; i < ntiles && ok; ++i) {
        // S^T = KV_tile . Q^T over the four chunks
        for (int c = 0; c < kChunks && ok; ++c) {
          const int n = i * kChunks + c, s = n % kSlots;
          if (!mbar_wait_bounded(&S.full[s], (n / kSlots) & 1)) { ok = false; break; }
          fence_proxy_async_smem();                      // cp.async writes -> tensor core
          tc_fence_after();
          const uint32_t kvb = smem_u32(S.kv[s]);
#pragma unroll
          for (int kk = 0; kk < kChunkD / 16; ++kk) {
            const uint32_t r = kk >> 2, koff = (kk & 3) * 32;
            mma_f16_ss(tmem + kSCol, sdesc_sw128(kvb + r * kRegionBytes + koff, 16, 1024),
                       sdesc_sw128(qb + (2 * c + r) * kQRegion + koff, 16, 1024), id_qk,
                       (c | kk) != 0 ? 1u : 0u);
          }
        }
        if (!ok) break;
        mma_commit(&S.sfull);
        // O^T += KV_tile^T . P^T, chunk by chunk; each chunk's slot is
        // returned to the gather when its MMAs are done
        if (!mbar_wait_bounded(&S.pready, i & 1)) { ok = false; break; }
        tc_fence_after();
        for (int c = 0; c < kChunks; ++c) {
          const int n = i * kChunks + c, s = n % kSlots;
          const uint32_t kvb = smem_u32(S.kv[s]);
#pragma unroll
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_f16_ss(tmem + kOCol + c * 64, sdesc_sw128(kvb + kk * 2048, kRegionBytes, 1024),
                       sdesc_sw128(pb + kk * 2048, 1024, 1024), id_pv, (i | kk) != 0 ? 1u : 0u);
          mma_commit(&S.empty[s]);
        }
      }
      mma_commit(&S.ofull);                              // every MMA of the CTA is done
      (void)mbar_wait_drain(&S.ofull, 0);
      if (!ok && a.err) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- softmax and output: thread = TMEM lane
    const int quarter = warp & 3;
    const int pos = 32 * quarter + lane;                 // position within a tile / value within a chunk
    const uint32_t lane_addr = static_cast<uint32_t>(32 * quarter) << 16;
    const int ew = warp - kEpiWarp0;                     // 0..3
    float m_own = -INFINITY;                             // lane L: head L's reference maximum
    float l_part[kHeads];                                // this position's running sums
#pragma unroll
    for (int h = 0; h < kHeads; ++h) l_part[h] = 0.0f;
    const float sl2 = a.scale * kLog2e;
    // every epilogue warp runs the same sequence of named barriers whatever
    // happens: a wait that gives up clears `ok`, later waits are skipped and
    // the remaining tiles are run through on whatever TMEM holds (the call
    // then reports QLI_DEVERR_TIMEOUT and its outputs are not written)
    for (int i = 0; i < ntiles; ++i) {
      const int e = i * kTileRows + pos;
      bool bad = false;
      const bool valid = e < a.K && row_of(a, b, __ldg(idx_row + e), bad) != nullptr;
      if (ok && !mbar_wait_warp(&S.sfull, i & 1)) ok = false;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + lane_addr + kSCol, r);
      tmem_ld_wait();
      // scores in log2 units: x = s * scale * log2(e)
      float x[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) x[h] = valid ? __uint_as_float(r[h]) * sl2 : -INFINITY;
      float v[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) v[h] = x[h];
      S.red[ew][lane] = transpose_reduce(v, [](float p, float q) { return fmaxf(p, q); });
      named_bar(1, 128);
      const float mt = fmaxf(fmaxf(S.red[0][lane], S.red[1][lane]), fmaxf(S.red[2][lane], S.red[3][lane]));
      named_bar(1, 128);                                 // red is reused next tile
      // lane L decides head L's reference maximum (log2 units)
      float m_new = m_own;
      if (mt > -INFINITY && (m_own == -INFINITY || mt > m_own + kRescale * kLog2e)) m_new = mt;
      const float alpha = (m_new == m_own) ? 1.0f : (m_own == -INFINITY ? 0.0f : exp2f(m_own - m_new));
      const bool changed = __any_sync(0xffffffffu, m_new != m_own);
      m_own = m_new;
      // P for this position, all 32 heads; running sums
      uint32_t pk[kHeads / 2];
#pragma unroll
      for (int h = 0; h < kHeads; h += 2) {
        const float ma = __shfl_sync(0xffffffffu, m_own, h), mb = __shfl_sync(0xffffffffu, m_own, h + 1);
        const float pa = (x[h] == -INFINITY) ? 0.0f : exp2f(x[h] - ma);
        const float pb = (x[h + 1] == -INFINITY) ? 0.0f : exp2f(x[h + 1] - mb);
        if (changed) {
          l_part[h] *= __shfl_sync(0xffffffffu, alpha, h);
          l_part[h + 1] *= __shfl_sync(0xffffffffu, alpha, h + 1);
        }
        l_part[h] += pa;
        l_part[h + 1] += pb;
        const __nv_bfloat162 pp = __floats2bfloat162_rn(pa, pb);
        pk[h / 2] = *reinterpret_cast<const uint32_t*>(&pp);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4*>(&S.p[sw(pos, u)]) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      if (changed && i > 0) {
        // O^T (lane = value, column = head) times alpha of each head; the
        // MMAs of the previous tile are complete (S^T of this tile is)
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tmem + lane_addr + kOCol + c * 64, o);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < kHeads; ++h)
            o[h] = __float_as_uint(__uint_as_float(o[h]) * __shfl_sync(0xffffffffu, alpha, h));
          tmem_st_32x32b_x32(tmem + lane_addr + kOCol + c * 64, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();                          // P^T -> tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pready);
    }
    // totals: l of head L in lane L, the same in every epilogue warp
    const float lw = transpose_reduce(l_part, [](float p, float q) { return p + q; });
    named_bar(1, 128);
    S.red[ew][lane] = lw;
    named_bar(1, 128);
    const float l = (S.red[0][lane] + S.red[1][lane]) + (S.red[2][lane] + S.red[3][lane]);
    const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
    if (ok && !mbar_wait_warp(&S.ofull, 0)) ok = false;
    tc_fence_after();
    if (ok) {
      if (ew == 0 && a.lse)
        a.lse[static_cast<int64_t>(t) * a.H + h0 + lane] =
            l > 0.0f ? (m_own + log2f(l)) * (1.0f / kLog2e) : -INFINITY;
      uint16_t* orow = a.out + static_cast<int64_t>(t) * a.o_st + static_cast<int64_t>(h0) * a.o_sh;
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_addr + kOCol + c * 64, o);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          const float val = __uint_as_float(o[h]) * __shfl_sync(0xffffffffu, inv_l, h);
          const __nv_bfloat16 bv = __float2bfloat16_rn(val);
          orow[static_cast<int64_t>(h) * a.o_sh + c * kChunkD + pos] =
              *reinterpret_cast<const uint16_t*>(&bv);
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
