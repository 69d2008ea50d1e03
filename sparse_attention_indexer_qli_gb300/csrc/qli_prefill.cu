// Scoring stage for prefill-shaped calls (many query tokens per request).
//
// Here the contraction dominates (each K row meets thousands of query
// tokens), so the kernel is built around the tensor core:
//  * kconv_kernel widens each request's paged INT8 index K once into a dense
//    FP16 [cap, 128] array and its FP16 scales into FP32, in the workspace
//    (a few MB per request: L2-resident while the main kernel runs);
//  * prefill_kernel is persistent, one CTA per SM. A unit is one token group
//    (up to 4 tokens of one request, MMA N = tokens*64 <= 256) and a range of
//    its position tiles: the tiles of all groups are split evenly into one
//    contiguous range per CTA, and a group's queries stay in shared memory
//    (FP16 * 2^-10, 128-byte swizzle) across its part of the range; K tiles
//    stream in
//    by TMA (128-byte swizzle) through a 4-stage ring; the 128 x N FP32
//    accumulator is double-buffered across all 512 TMEM columns.
// Warp roles: warp 0 producer, warp 1 MMA issuer, warps 2-17 epilogue (four
// warps per TMEM lane quarter, each summing the heads of one token, or of two
// tokens when N = 32).
//
// Numerics are those of the streaming kernel (see qli_score.cu): exact
// FP16 products of INT8 values, exact FP32 sums, the accumulator holding
// s/1024, then the golden chain of the guide "DeepSeek V4.1 QLI V2 与候选集成"
// (section 当前 A3 契约) per head in ascending order.
#include <cuda.h>
#include <cuda_fp16.h>

#include "qli_internal.h"
#include "qli_ptx.cuh"

namespace qli {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 576;
constexpr int kABytes = kTile * kHeadDim * 2;     // 32 KB FP16 tile (two 16 KB K halves)
constexpr int kBBytes = kMaxMmaN * kHeadDim * 2;  // 64 KB: 4 tokens x 64 heads
constexpr uint32_t kTmemCols = 512;

struct Smem {
  uint8_t a[kStages][kABytes];   // 1024-aligned
  uint8_t b[kBBytes];            // 1024-aligned
  alignas(16) __half wq[2][kMaxMmaN];   // by unit parity: a warp may still sum the previous unit
  uint64_t full[kStages], empty[kStages], dfull[2], dempty[2], bfull, bempty;
  uint32_t tmem_base;
};
constexpr int kSmemBytes = static_cast<int>(sizeof(Smem)) + 1024;

__device__ __forceinline__ uint32_t sw128(uint32_t rows, uint32_t n, uint32_t c) {
  return (c >> 3) * (rows * 128u) + (n >> 3) * 1024u + (n & 7u) * 128u +
         (((c & 7u) ^ (n & 7u)) << 4);
}

// 8 INT8 -> 8 FP16 (exact), optionally times 2^-10 (exact for |x| <= 128).
__device__ __forceinline__ uint4 widen8(uint2 v, bool div1024) {
  const uint32_t u0 = v.x ^ 0x80808080u, u1 = v.y ^ 0x80808080u;
  uint32_t h[4] = {__byte_perm(u0, 0x64646464u, 0x5140), __byte_perm(u0, 0x64646464u, 0x7362),
                   __byte_perm(u1, 0x64646464u, 0x5140), __byte_perm(u1, 0x64646464u, 0x7362)};
  const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);
  const __half2 sc = __floats2half2_rn(1.0f / 1024.0f, 1.0f / 1024.0f);
  uint4 r;
  uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __half2 x = __hsub2(*reinterpret_cast<__half2*>(&h[k]), bias);
    if (div1024) x = __hmul2(x, sc);
    o[k] = *reinterpret_cast<uint32_t*>(&x);
  }
  return r;
}

// ---- K widening: a CTA per 128-row tile of a request, 8 threads per row
// (16 INT8 values each) and 4 rows per thread; every load of the tile is in
// flight before the first conversion, so the kernel takes one pass of three
// round trips (length, block table, rows) instead of waves of them
constexpr int kConvThreads = 256;
constexpr int kConvRows = kTile;                        // rows per CTA
constexpr int kConvRPT = kConvRows / (kConvThreads / 8);  // rows per thread

__global__ void __launch_bounds__(kConvThreads) kconv_kernel(DevArgs a) {
  const int b = blockIdx.y;
  const int lk = a.req_lk[b];
  const int row0 = blockIdx.x * kConvRows;
  const int padded = (lk + kTile - 1) / kTile * kTile;
  if (row0 >= padded) return;
  const int ch = threadIdx.x & 7;                       // 16-byte piece of the row
  const int rsub = threadIdx.x >> 3;                    // 0..31
  const int64_t base = static_cast<int64_t>(b) * a.kstride;
  int32_t page[kConvRPT];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kConvRPT; ++i) {
    const int row = row0 + rsub + 32 * i;
    page[i] = row < lk ? a.bt[static_cast<int64_t>(b) * a.bt_stride + row / a.R] : 0;
  }
  uint4 v[kConvRPT];
  uint16_t sc[kConvRPT];
#pragma unroll
  for (int i = 0; i < kConvRPT; ++i) {
    const int row = row0 + rsub + 32 * i;
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    sc[i] = 0;
    if (row < lk) {
      if (page[i] < 0 || page[i] >= a.num_pages) {
        bad = true;
        page[i] = 0;
      }
      const uint8_t* pg = a.cache + static_cast<int64_t>(page[i]) * a.page_stride;
      const int r = row % a.R;
      v[i] = __ldg(reinterpret_cast<const uint4*>(pg + a.k_off + r * kHeadDim) + ch);
      if (ch == 0) sc[i] = __ldg(reinterpret_cast<const uint16_t*>(pg + a.s_off) + r);
    }
  }
  if (bad && ch == 0) atomicOr(a.err, QLI_DEVERR_PAGE);
#pragma unroll
  for (int i = 0; i < kConvRPT; ++i) {
    const int row = row0 + rsub + 32 * i;
    if (row >= padded) continue;
    // rows past the request's length are the zero tail of the last tile
    uint4* dst = reinterpret_cast<uint4*>(a.kf16 + (base + row) * kHeadDim) + 2 * ch;
    const uint2 lo = make_uint2(v[i].x, v[i].y), hi = make_uint2(v[i].z, v[i].w);
    const bool live = row < lk;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    dst[0] = live ? (a.fp8 ? e4m3x8_to_f16x8(lo, false) : widen8(lo, false)) : z;
    dst[1] = live ? (a.fp8 ? e4m3x8_to_f16x8(hi, false) : widen8(hi, false)) : z;
    if (ch == 0) a.ks32[base + row] = live ? __half2float(__ushort_as_half(sc[i])) : 0.0f;
  }
}

// ---- work walk -----------------------------------------------------------
// The position tiles of all token groups, group after group, are split into
// one contiguous range per CTA (equal within one tile). A CTA walks its range
// as segments, one per group: the group's queries are staged once for the
// segment, whose tiles then stream through.
struct Seg {
  int32_t g, t0, cnt, b, tile0, ntiles, end;   // end: the group's end in the tile list
};

// Group g's part of the range [tb, te).
__device__ __forceinline__ Seg seg_of_group(const DevArgs& a, int32_t g, int32_t tb, int32_t te) {
  Seg x;
  x.g = g;
  x.t0 = a.grp_t0[g];
  x.cnt = a.grp_cnt[g];
  x.b = a.tok_b[x.t0];
  const int32_t s0 = a.unit_start[g];
  x.end = a.unit_start[g + 1];
  const int32_t lo = max(tb, s0);
  x.tile0 = lo - s0;
  x.ntiles = min(te, x.end) - lo;
  return x;
}

// The first segment: the group holding tile tb (the last group starting at
// or before it; groups without tiles start where the next one does).
__device__ __forceinline__ Seg seg_first(const DevArgs& a, int32_t tb, int32_t te) {
  int32_t lo = 0, hi = a.Gmax - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (a.unit_start[mid] <= tb) lo = mid; else hi = mid - 1;
  }
  return seg_of_group(a, lo, tb, te);
}

// The segment after x, when x.end < te: the next group with tiles.
__device__ __forceinline__ Seg seg_next(const DevArgs& a, const Seg& x, int32_t te) {
  int32_t g = x.g + 1;
  while (a.unit_start[g + 1] <= x.end) ++g;
  return seg_of_group(a, g, x.end, te);
}

// 18 warps: the four SM sub-partitions hold 5, 5, 4 and 4 of them in 16K
// registers each, which caps a thread at 96 registers
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(
    const __grid_constant__ CUtensorMap tm_k, DevArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t U = a.unit_start[a.Gmax];   // position tiles of all groups
  const int32_t tb = static_cast<int32_t>(static_cast<int64_t>(U) * blockIdx.x / gridDim.x);
  const int32_t te = static_cast<int32_t>(static_cast<int64_t>(U) * (blockIdx.x + 1) / gridDim.x);
  if (tb >= te) return;

  if (warp == 0) tmem_alloc(&S.tmem_base, kTmemCols);
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.dfull[s], 1);
      mbar_init(&S.dempty[s], 16);
    }
    mbar_init(&S.bfull, 16);
    mbar_init(&S.bempty, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool ok = true;

  if (warp == 0) {
    // ---------------- producer: FP16 K tiles by TMA
    int k = 0;
    for (Seg x = seg_first(a, tb, te); ok; x = seg_next(a, x, te)) {
      for (int i = 0; i < x.ntiles && ok; ++i, ++k) {
        const int s = k % kStages;
        const uint32_t ph = (k / kStages) & 1;
        if (lane == 0) {
          ok = mbar_wait_bounded<true>(&S.empty[s], ph ^ 1);
          if (ok) {
            mbar_arrive_expect_tx(&S.full[s], kABytes);
            const int32_t y = x.b * static_cast<int32_t>(a.kstride) + (x.tile0 + i) * kTile;
            tma_load_3d(&S.a[s][0], &tm_k, 0, y, 0, &S.full[s]);
            tma_load_3d(&S.a[s][kABytes / 2], &tm_k, 64, y, 0, &S.full[s]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (x.end >= te) break;
    }
    if (lane == 0) {
      for (int j = max(0, k - kStages); j < k; ++j)
        (void)mbar_wait_drain(&S.full[j % kStages], (j / kStages) & 1);
      if (!ok) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      int k = 0, n = 0;              // n: segments (groups) so far
      const uint32_t b0 = smem_u32(&S.b[0]);
      for (Seg x = seg_first(a, tb, te); ok; x = seg_next(a, x, te), ++n) {
        const uint32_t nmma = static_cast<uint32_t>(x.cnt * a.N);
        const uint32_t idesc = idesc_f16_m128(nmma);
        // the group's queries, staged by the epilogue warps
        if (!mbar_wait_bounded<true>(&S.bfull, n & 1)) { ok = false; break; }
        for (int i = 0; i < x.ntiles; ++i, ++k) {
          const int s = k % kStages, ds = k & 1;
          if (!mbar_wait_bounded<true>(&S.full[s], (k / kStages) & 1) ||
              !mbar_wait_bounded<true>(&S.dempty[ds], ((k >> 1) & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(&S.a[s][0]);
          const uint32_t d = tmem + ds * 256;
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk) {
            const uint32_t kb = kk >> 2, koff = (kk & 3) * 32;
            mma_f16_ss(d, sdesc_k_sw128(a0 + kb * (kABytes / 2) + koff),
                       sdesc_k_sw128(b0 + kb * (nmma * 128) + koff), idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&S.empty[s]);
          mma_commit(&S.dfull[ds]);
        }
        mma_commit(&S.bempty);   // the group's queries are no longer read
        if (x.end >= te) break;
      }
      if (k > 0) (void)mbar_wait_drain(&S.dfull[(k - 1) & 1], ((k - 1) >> 1) & 1);
      if (!ok) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- epilogue (and query staging), 16 warps: warp e handles
    // TMEM lane quarter (warp & 3) and token slot e / 4 of the group; with
    // N = 64 that is one token (heads 0-31 and 32-63), with N = 32 two tokens
    // (slot and slot + 4). Both TMEM loads are issued before one wait.
    const int e = warp - 2;                 // 0..15
    const int quarter = warp & 3;
    const int slot = e >> 2;                // 0..3
    const int row = 32 * quarter + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * quarter) << 16;
    const int etid = tid - 64;              // 0..511
    int k = 0, n = 0;                // n: segments (groups) so far
    for (Seg x = seg_first(a, tb, te); ok; x = seg_next(a, x, te), ++n) {
      const int nrows = x.cnt * a.N;
      {
        // the group's queries and weights are loaded first (one global
        // latency, overlapping the previous group's last tiles), then stored
        // once the buffers are free
        constexpr int kPer = kMaxMmaN * 16 / 512;
        uint2 v[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = etid + 512 * i;
          const int nn = idx >> 4, ch = idx & 15;
          const int gi = nn / a.N, h = nn % a.N;
          if (idx < nrows * 16)
            v[i] = *reinterpret_cast<const uint2*>(a.q + static_cast<int64_t>(x.t0 + gi) * a.q_st +
                                                   static_cast<int64_t>(h) * a.q_sh + ch * 8);
        }
        uint16_t wb = 0, qb = 0;
        if (etid < nrows) {
          const int64_t o = static_cast<int64_t>(x.t0) * a.N + etid;   // tokens are consecutive
          wb = a.w[o];
          qb = a.qs[o];
        }
        // before overwriting the queries and this parity's weights: every
        // epilogue warp has loaded this warp's last tile (the previous
        // segment's), so it is done with the segment before that, and the
        // previous segment's MMAs are complete
        if (k > 0 && !mbar_wait_warp<true>(&S.dempty[(k - 1) & 1], ((k - 1) >> 1) & 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait_warp<true>(&S.bempty, (n & 1) ^ 1)) { ok = false; break; }
        if (etid < nrows) S.wq[n & 1][etid] = __hmul(__ushort_as_half(wb), __ushort_as_half(qb));
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = etid + 512 * i;
          const int nn = idx >> 4, ch = idx & 15;
          if (idx < nrows * 16)
            *reinterpret_cast<uint4*>(&S.b[sw128(nrows, nn, ch)]) =
                a.fp8 ? e4m3x8_to_f16x8(v[i], true) : widen8(v[i], true);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.bfull);
        // every warp's staging is complete (and visible) once bfull flips
        if (!mbar_wait_warp<true>(&S.bfull, n & 1)) { ok = false; break; }
      }

      // the (up to two) tokens this warp sums, and the TMEM columns of each
      // 32-column half it loads
      const bool wide = a.N == 64;
      const int g0 = slot, g1 = wide ? slot : slot + 4;
      const bool has0 = g0 < x.cnt, has1 = wide ? has0 : g1 < x.cnt;
      const int32_t V0 = has0 ? a.tok_V[x.t0 + g0] : 0;
      const int32_t V1 = has1 ? a.tok_V[x.t0 + g1] : 0;
      const uint32_t c0 = static_cast<uint32_t>(g0 * a.N);
      const uint32_t c1 = wide ? c0 + 32 : static_cast<uint32_t>(g1 * a.N);
      // this warp's tokens' w * q_scale pairs, read 16 bytes (four head pairs)
      // at a time from a base fixed for the unit
      const uint4* w0 = reinterpret_cast<const uint4*>(&S.wq[n & 1][c0]);
      const uint4* w1 = reinterpret_cast<const uint4*>(&S.wq[n & 1][c1]);
      // per-unit row pointers of the (up to two) tokens this warp scores
      const int32_t ta = x.t0 + g0, tb = x.t0 + g1;
      float* const srow0 = a.scores + static_cast<int64_t>(ta) * a.Lrow;
      float* const srow1 = a.scores + static_cast<int64_t>(tb) * a.Lrow;
      float* const brow0 = a.bscores + static_cast<int64_t>(ta) * a.Brow;
      float* const brow1 = a.bscores + static_cast<int64_t>(tb) * a.Brow;
      const float* const ksrow = a.ks32 + static_cast<int64_t>(x.b) * a.kstride;
      const bool source = a.mode == QLI_CAND_SOURCE;
      // one golden chain over 32 heads (a 32-column accumulator half)
      const auto chain = [&](float acc, const uint32_t (&r)[32], const uint4* w) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 wq = w[q];
          const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
          for (int ii = 0; ii < 4; ++ii)
            acc = head_pair_acc(acc, __uint_as_float(r[8 * q + 2 * ii]),
                                __uint_as_float(r[8 * q + 2 * ii + 1]), wv[ii]);
        }
        return acc;
      };
      const auto emit = [&](float acc, float ks, int32_t pos, int32_t V, float* srow, float* brow) {
        const float score = __fmul_rn(acc, ks);
        const bool elig = pos < V;
        if (elig) srow[pos] = score;
        if (source) {
          float m = elig ? score : -INFINITY;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((row & (kBlock - 1)) == 0 && elig) brow[pos / kBlock] = m;
        }
      };
      for (int i = 0; i < x.ntiles; ++i, ++k) {
        const int ds = k & 1;
        if (!mbar_wait_warp<true>(&S.dfull[ds], (k >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const int32_t pos = (x.tile0 + i) * kTile + row;
        const float ks = ksrow[pos];
        const uint32_t base = tmem + lane_addr + ds * 256;
        // the two 32-column halves one after the other (32 live registers):
        // heads 0-31 and 32-63 of one token, or two tokens of 32 heads
        uint32_t r[32];
        float acc0 = 0.0f;
        if (has0) {                           // uniform across the warp
          tmem_ld_32x32b_x32(base + c0, r);
          tmem_ld_wait();
          acc0 = chain(0.0f, r, w0);
        }
        if (has1) {
          tmem_ld_32x32b_x32(base + c1, r);
          tmem_ld_wait();
        }
        // the accumulator is in registers: hand the TMEM stage back now
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.dempty[ds]);
        if (wide) {
          if (has0) emit(chain(acc0, r, w1), ks, pos, V0, srow0, brow0);
        } else {
          if (has0) emit(acc0, ks, pos, V0, srow0, brow0);
          if (has1) emit(chain(0.0f, r, w1), ks, pos, V1, srow1, brow1);
        }
      }
      if (x.end >= te) break;
    }
    if (!ok && lane == 0) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Tensor map over the widened K of every request: x = 128 FP16 of a row, y =
// row (B * cap rows of 256 B); box = 64 FP16 (128 B) x 128 rows, 128-byte
// swizzle (the layout the MMA's smem descriptor reads).
bool encode_kf16_map(const DevArgs& d, CUtensorMap* m) {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim),
                              static_cast<cuuint64_t>(d.B) * static_cast<cuuint64_t>(d.kstride), 1};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2),
                                 static_cast<cuuint64_t>(kHeadDim * 2) * dims[1]};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTile), 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, d.kf16, dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

std::atomic<uint64_t> g_smem_prefill_kernel{0};

cudaError_t launch_prefill(const DevArgs& d, cudaStream_t s) {
  if (d.T == 0 || d.B == 0) return cudaSuccess;
  dim3 cgrid(static_cast<unsigned>((d.kstride + kConvRows - 1) / kConvRows),
             static_cast<unsigned>(d.B));
  kconv_kernel<<<cgrid, kConvThreads, 0, s>>>(d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tm;
  if (!encode_kf16_map(d, &tm)) return cudaErrorInvalidValue;
  e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_kernel), kSmemBytes,
                        g_smem_prefill_kernel);
  if (e != cudaSuccess) return e;
  prefill_kernel<<<d.num_sms, kThreads, kSmemBytes, s>>>(tm, d);
  return cudaGetLastError();
}

int prefill_launches(const DevArgs& d) { return (d.T > 0 && d.B > 0) ? 2 : 0; }

}  // namespace qli
