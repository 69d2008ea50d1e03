// Scoring stage: paged index-K gather, the Q.K contraction on the tcgen05
// tensor cores, and the fused golden epilogue.
//
// Numeric golden (guide "DeepSeek V4.1 QLI V2 与候选集成", section 当前 A3 契约):
// INT32 QK / 1024 -> FP16, FP16 ReLU, times FP16(weight * q_scale), FP32
// reduction over the heads, then times the per-token K scale.
//
// sm_103a has no INT8 tensor-core MMA (tcgen05 kind::i8 is not available on
// this target), so the INT8 operands are widened to FP16 and contracted with
// kind::f16 into FP32. The FP8 variant (quant mode 1, E4M3 codes) widens its
// codes to FP16 the same way (exactly); there the FP32 sums are the tensor
// core's, no longer exact, so its scores match the exact dot to within the
// rounding of those sums. This is exact: every INT8 value is an FP16 integer,
// every product is an integer below 2^15, and every partial sum of the 128
// terms is an integer of magnitude <= 128*128*128 = 2^21 < 2^24. The queries
// are pre-multiplied by 2^-10 (exact in FP16 for |q| <= 128), so the FP32
// accumulator holds exactly s/1024, the value the golden rounds to FP16.
//
// Orientation: A (M = 128) = the K rows of a tile of 128 positions, B (N) =
// the queries' heads (up to 256/N tokens of one request share a tile), so
// TMEM lane i holds every head's dot for position i and the epilogue thread
// of lane i sums its heads sequentially in FP32 — the order the golden's
// reduction is read with.
//
// Page addressing (section 数据流, PA_BBND): position j of a request lives in
// page block_table[b][j / R], row j % R; its 128 INT8 values at
// k_offset + row*128 and its FP16 scale at scale_offset + row*2 in that page.
#include <cuda.h>
#include <cuda_fp16.h>

#include "qli_internal.h"
#include "qli_ptx.cuh"

namespace qli {
namespace {

// Byte offset of 16-byte chunk c (8 FP16 values, c in 0..15) of row n in a
// K-major tile with the 128-byte swizzle: two 64-element K halves of
// rows*128 bytes each; rows grouped by 8 (1024 B); the chunk index XORed with
// the row within its group.
__device__ __forceinline__ uint32_t sw128_off(uint32_t rows, uint32_t n, uint32_t c) {
  return (c >> 3) * (rows * 128u) + (n >> 3) * 1024u + (n & 7u) * 128u +
         (((c & 7u) ^ (n & 7u)) << 4);
}

// 8 INT8 values -> 8 FP16 values (exact): (x + 128) placed in the mantissa
// of 1024.0h gives 1024 + x + 128, then 1152 is subtracted.
__device__ __forceinline__ uint4 i8x8_to_f16x8(uint2 v) {
  const uint32_t u0 = v.x ^ 0x80808080u, u1 = v.y ^ 0x80808080u;
  uint32_t h[4];
  h[0] = __byte_perm(u0, 0x64646464u, 0x5140);
  h[1] = __byte_perm(u0, 0x64646464u, 0x7362);
  h[2] = __byte_perm(u1, 0x64646464u, 0x5140);
  h[3] = __byte_perm(u1, 0x64646464u, 0x7362);
  const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);
  uint4 r;
  uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __half2 x = __hsub2(*reinterpret_cast<__half2*>(&h[k]), bias);
    o[k] = *reinterpret_cast<uint32_t*>(&x);
  }
  return r;
}

// Same, times 2^-10 (exact: |x| <= 128).
__device__ __forceinline__ uint4 i8x8_to_f16x8_div1024(uint2 v) {
  uint4 r = i8x8_to_f16x8(v);
  const __half2 s = __floats2half2_rn(1.0f / 1024.0f, 1.0f / 1024.0f);
  uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __half2 x = __hmul2(*reinterpret_cast<__half2*>(&o[k]), s);
    o[k] = *reinterpret_cast<uint32_t*>(&x);
  }
  return r;
}

// ---------------------------------------------------------------------------
// Streaming kernel: one token per tile (decode batches and consumer mode).
//
// Persistent, one CTA per SM, each CTA owns a contiguous range of the
// (token, tile) list, so the token's queries stay in shared memory across
// its tiles. Warp roles:
//   warp 0      producer: TMA copies of the tile's INT8 K rows (128-byte
//               swizzle) and FP16 scales into an 8-stage shared-memory ring
//               (whole pages for dense tiles; 1 KB + 16 B per 8-position
//               block in consumer mode); for dense tiles lane j resolves the
//               page IDs of tile k0+j once per 32 tiles, so no block-table
//               load sits between two copies
//   warp 19     consumer mode only: a second producer, warp 0 taking the
//               even tiles and warp 19 the odd ones. A candidate tile is 16
//               copies and each holds its issuing thread for hundreds of
//               cycles, so one issuer would cap the tile rate; dense tiles
//               (one or two copies) run faster with a single producer
//   warps 1-2   MMA, one issuing thread per tile parity: 8 x tcgen05.mma
//               (A from TMEM, B = the token's queries from shared memory),
//               committed to the A slot's and the accumulator's barriers.
//               Back-to-back MMAs into rotating accumulators cost about 59
//               cycles each, but a commit stalls its thread about 128 cycles
//               and each barrier probe about 60, so one issuer would leave
//               the tensor core idle; two hide each other's bookkeeping.
//   warps 3-10  converters, two groups of four taking alternate tiles: row =
//               position; INT8 -> FP16 in registers, stored to TMEM as the
//               MMA's A operand; queries -> FP16 * 2^-10 in 128-byte-swizzled
//               shared memory when the token changes
//   warps 11-18 epilogue, two groups of four taking alternate tiles: the
//               golden chain per position (a 64-long dependent FP32 add chain,
//               so two tiles are summed at once), score store, block max
// Each tile parity p runs converter group p -> MMA warp p -> epilogue group
// p, and owns A slots p, p + 2 and accumulator slots p, p + 2 (in consumer
// mode also producer p and K stages p, p + 2, ...): the two parities are
// independent in-order pipelines, so every barrier's previous phase belongs
// to the same parity and has already been consumed. (With an odd slot
// count, one parity's epilogue could meet a slot still a phase behind,
// waiting on the other parity's MMA issuer.)
namespace stream {

constexpr int kKStages = 8;                          // shared-memory K ring
// TMEM holds two rings: the MMA's A operands (the converted K tiles, 64
// columns each), freed when the tensor core has read them, and the
// accumulators (64 columns each), freed when the epilogue has loaded them.
// Converters therefore wait only on the tensor core, and the tensor core
// only on the epilogue.
constexpr int kASlots = 4;                           // columns 0 .. 255
constexpr int kDSlots = 4;                           // columns 256 .. 511
static_assert(kASlots % 2 == 0 && kDSlots % 2 == 0, "each tile parity owns its slots");
constexpr uint32_t kSlotCols = 64;
constexpr uint32_t kDCol0 = kASlots * kSlotCols;
static_assert(kDCol0 + kDSlots * kSlotCols == 512, "TMEM column budget");
// warp roles: 0 producer, 1-2 MMA, then two groups of four converter warps,
// then two groups of four epilogue warps, then the second producer
constexpr int kProdWarp0 = 0, kMmaWarp0 = 1, kConvWarp0 = 3, kEpiWarp0 = kConvWarp0 + 8,
              kProdWarp1 = kEpiWarp0 + 8;
// block size: the dense instance has no second producer
constexpr int threads_for(bool cand) { return 32 * (kProdWarp1 + (cand ? 1 : 0)); }
static_assert(threads_for(false) == 608 && threads_for(true) == 640, "stream kernel block size");
constexpr int kKBytes = kTile * kHeadDim;            // 16 KB of INT8 rows per tile
// A K stage (17 KB): the tile's 128 rows of 128 B from 0 (one 128-row page,
// two 64-row pages, or 16 candidate blocks of 8 rows), their FP16 scales from
// kScOff, brought by a second copy per page (by the producer's stores for
// candidate tiles). A 128-row page whose scales follow its rows (kfused) is
// fetched by one copy of 130 rows instead: the scales arrive in rows 128-129,
// swizzled like the K rows. (Two 64-row pages cannot both carry their scale
// row in a 17 KB stage without breaking the 1024-byte alignment that the
// swizzle needs; stages of 18 KB that held them were slower.)
constexpr int kStageBytes = 17 * 1024;
constexpr uint32_t kScOff = kKBytes;
static_assert(kScOff + kTile * 2 <= kStageBytes && (kKBytes + 2 * kHeadDim) <= kStageBytes &&
                  kStageBytes % 1024 == 0, "K stage layout");
constexpr int kBBytes = 64 * kHeadDim * 2;           // 16 KB: up to 64 heads, FP16
constexpr uint32_t kTmemCols = 512;

// wq and K scales of tile k live in slot k % kSlots, written by the
// converter and read by the epilogue after it has released the tile's
// accumulator. The converter of tile k + kSlots waits for the MMA of tile
// k + kSlots - kASlots, which needed the accumulator slot that the epilogue
// of tile k + kSlots - kASlots - kDSlots released; for kSlots >= 10 (even)
// that is a later tile of the same epilogue group, so tile k's epilogue has
// finished reading its slot.
constexpr int kSlots = 16;
static_assert(kSlots >= 2 + kASlots + kDSlots && kSlots % 2 == 0, "wq / ks slot reuse distance");

struct Smem {
  uint8_t k[kKStages][kStageBytes];                  // 1024-aligned (offset 0)
  uint8_t b[2][kBBytes];                             // 1024-aligned; one per converter group
  alignas(16) __half wq[kSlots][64];
  float ks[kSlots][kTile];
  uint64_t full[kKStages], empty[kKStages];
  uint64_t afull[kASlots], afree[kASlots], dfull[kDSlots], dfree[kDSlots];
  uint64_t kready[kSlots];                           // wq / ks of the slot's tile written
#ifdef QLI_TEST_STALL_EPILOGUE
  uint64_t never;                                    // test build: nothing arrives here
#endif
  uint32_t tmem_base;
};
constexpr int kSmemBytes = static_cast<int>(sizeof(Smem)) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "stream kernel shared memory");

// Walks the CTA's units in order: (token, tile within the token).
struct Cursor {
  int32_t t, tile, end_t;
  // The token owning unit u (< unit_start[T]): the last t with unit_start[t]
  // <= u. The whole warp searches, 32 probes per round trip, so T <= 1024
  // takes two rounds instead of a scalar search's log2(T) dependent loads.
  __device__ void init(const DevArgs& a, int32_t u) {
    const int lane = threadIdx.x & 31;
    int32_t lo = 0, hi = a.T;          // unit_start[lo] <= u < unit_start[hi]
    while (hi - lo > 1) {
      const int32_t step = (hi - lo + 31) >> 5;
      const int32_t p = lo + (lane + 1) * step;
      const bool le = p < hi && __ldg(a.unit_start + p) <= u;
      lo += __popc(__ballot_sync(0xffffffffu, le)) * step;
      hi = min(hi, lo + step);
    }
    t = lo;
    tile = u - a.unit_start[t];
    end_t = a.unit_start[t + 1];
  }
  // The same search by one thread (t and tile only).
  __device__ void init_scalar(const DevArgs& a, int32_t u) {
    int32_t lo = 0, hi = a.T - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (a.unit_start[mid] <= u) lo = mid; else hi = mid - 1;
    }
    t = lo;
    tile = u - a.unit_start[t];
  }
  __device__ void next(const DevArgs& a, int32_t u_next) {
    ++tile;
    if (u_next >= end_t) {
      do { ++t; } while (t + 1 <= a.T && a.unit_start[t + 1] <= u_next);
      tile = 0;
      end_t = (t < a.T) ? a.unit_start[t + 1] : u_next;
    }
  }
};

__device__ __forceinline__ void cvt_row16(const uint4 v, uint32_t* out8) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t u = w[k] ^ 0x80808080u;
    uint32_t lo = __byte_perm(u, 0x64646464u, 0x5140);
    uint32_t hi = __byte_perm(u, 0x64646464u, 0x7362);
    __half2 x = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
    __half2 y = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
    out8[2 * k] = *reinterpret_cast<uint32_t*>(&x);
    out8[2 * k + 1] = *reinterpret_cast<uint32_t*>(&y);
  }
}

// tm_page: box of R rows x 128 B (a whole page's index K); tm_blk: box of
// 8 rows x 128 B (one candidate block). Both use the 128-byte swizzle, so
// row r's 16-byte chunk c lands at r*128 + ((c ^ (r & 7)) * 16).
// 19 warps (20 with the second producer): the four SM sub-partitions hold
// at most 5 of them each in 16K registers, which caps a thread at 96
// registers (allocated in steps of 8): a larger per-thread budget would make
// the launch fail
template <bool kFp8, bool kCand>
__global__ void __launch_bounds__(threads_for(kCand), 1) stream_kernel(
    const __grid_constant__ CUtensorMap tm_page, const __grid_constant__ CUtensorMap tm_blk,
    DevArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  // setup that reads nothing the plan writes runs while the plan finishes
  if (tid == 0) {
    prefetch_tensormap(&tm_page);
    prefetch_tensormap(&tm_blk);
  }
  if (warp == 0) tmem_alloc(&S.tmem_base, kTmemCols);
  if (tid == 32) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 4);
    }
    for (int s = 0; s < kASlots; ++s) {
      mbar_init(&S.afull[s], 4);      // the converting group's four warps
      mbar_init(&S.afree[s], 1);      // MMA commit
    }
    for (int s = 0; s < kDSlots; ++s) {
      mbar_init(&S.dfull[s], 1);      // MMA commit
      mbar_init(&S.dfree[s], 4);      // the epilogue group's four warps
    }
    for (int s = 0; s < kSlots; ++s) mbar_init(&S.kready[s], 4);   // converter warps
#ifdef QLI_TEST_STALL_EPILOGUE
    mbar_init(&S.never, 1);
#endif
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  pdl_wait();   // the plan's outputs (and zeroed histograms) are ready
  const int32_t U = a.unit_start[a.T];
  const int32_t u0 = static_cast<int32_t>(static_cast<int64_t>(U) * blockIdx.x / gridDim.x);
  const int32_t u1 = static_cast<int32_t>(static_cast<int64_t>(U) * (blockIdx.x + 1) / gridDim.x);
  if (u0 >= u1) {
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  const int32_t nk = u1 - u0;
  const bool consumer = a.mode == QLI_CAND_CONSUMER;   // == kCand
  bool ok = true;

  if (!kCand && warp == kProdWarp0) {
    // ---------------- producer of the dense instance. It keeps the general
    // form (with a candidate-tile branch that consumer calls, launched on the
    // other instance, never reach): without that branch the code ptxas
    // builds for 64-row pages is ~3% slower on the 1M-context workload.
    // index K is read once: its lines leave L2 first, ahead of the score
    // rows and histograms the selection reads next
    const uint64_t kpol = l2_policy_evict_first();
    Cursor c;
    c.init(a, u0);
    int issued = 0;
    int32_t pg0 = 0, pg1 = -1;     // dense: this lane's look-ahead tile's pages
    // consumer: tile k's candidate count, this lane's block and its page,
    // loaded while tile k-1 was issued (one round trip, off the critical path)
    int32_t cn_nc = 0, cn_blk = 0, cn_page = 0;
    uint4 cn_sc = make_uint4(0u, 0u, 0u, 0u);
    const auto consumer_fetch = [&](const Cursor& at) {
      const int32_t t = at.t;
      const int64_t i = static_cast<int64_t>(t) * a.C + at.tile * (kTile / kBlock) + lane;
      cn_nc = a.cand_cnt[t];
      if (at.tile * (kTile / kBlock) + lane < a.C) {
        cn_blk = a.cand_list[i];
        cn_page = a.cand_page[i];
        cn_sc = a.cand_sc[i];
      }
    };
    if (consumer && nk > 0) consumer_fetch(c);
    for (int k = 0; k < nk && ok; ++k) {
      const int s = k % kKStages;
      const uint32_t ph = (k / kKStages) & 1;
      if (!consumer && (k & 31) == 0) {
        // lane j resolves tile k+j: token, request, pages (one or two per
        // tile). The token comes from the next 32 token boundaries after the
        // base's (one load per lane): tile k+j lies in token c.t + (the
        // boundaries at or below its unit), found by a shuffle search. The
        // base (c.t, c.tile) is unit u0+k's token and tile, or a tile past
        // that token's last when u0+k starts a later one.
        const int32_t uj = u0 + k + lane;
        const int32_t bi = c.t + 1 + lane;
        const int32_t nb = bi <= a.T ? __ldg(a.unit_start + bi) : 0x7fffffff;
        int32_t cnt = 0;
#pragma unroll
        for (int w = 16; w > 0; w >>= 1)
          if (__shfl_sync(0xffffffffu, nb, cnt + w - 1) <= uj) cnt += w;
        if (__shfl_sync(0xffffffffu, nb, cnt) <= uj) ++cnt;      // 0..32
        const int32_t below = __shfl_sync(0xffffffffu, nb, cnt > 0 ? cnt - 1 : 0);
        Cursor m;
        m.t = c.t;
        m.tile = 0;
        if (k + lane < nk) {
          if (cnt < 32) {
            m.t = c.t + cnt;
            m.tile = uj - (cnt > 0 ? below : u0 + k - c.tile);
          } else {
            m.init_scalar(a, uj);      // past 32 boundaries (tokens without tiles)
          }
          const int32_t b = a.tok_b[m.t], V = a.tok_V[m.t];
          const int64_t row = static_cast<int64_t>(b) * a.bt_stride;
          const int32_t j0 = m.tile * kTile;
          const bool two = a.R < kTile && j0 + a.R < V;   // 64-row pages: second half visible
          pg0 = a.bt[row + j0 / a.R];
          pg1 = two ? a.bt[row + j0 / a.R + 1] : 0;
          if (pg0 < 0 || pg0 >= a.num_pages || pg1 < 0 || pg1 >= a.num_pages) {
            atomicOr(a.err, QLI_DEVERR_PAGE);
            if (pg0 < 0 || pg0 >= a.num_pages) pg0 = 0;
            if (pg1 < 0 || pg1 >= a.num_pages) pg1 = 0;
          }
          if (!two) pg1 = -1;
        }
        // the next batch's base: one tile past lane 31's (used only when
        // tile k+32 exists, i.e. lane 31 resolved a tile)
        c.t = __shfl_sync(0xffffffffu, m.t, 31);
        c.tile = __shfl_sync(0xffffffffu, m.tile, 31) + 1;
      }
      if (lane == 0) ok = mbar_wait_bounded(&S.empty[s], ph ^ 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (!consumer) {
        const int32_t p0 = __shfl_sync(0xffffffffu, pg0, k & 31);
        const int32_t p1 = __shfl_sync(0xffffffffu, pg1, k & 31);
        if (lane == 0) {
          const int npages = p1 >= 0 ? 2 : 1;
          const int box_rows = a.kfused ? a.R + 2 : a.R;
          mbar_arrive_expect_tx(&S.full[s],
                                npages * (box_rows * kHeadDim + (a.kfused ? 0 : a.R * 2)));
          for (int p = 0; p < npages; ++p) {
            const int32_t page = p == 0 ? p0 : p1;
            tma_load_3d_hint(&S.k[s][p * a.R * kHeadDim], &tm_page, 0, 0, page, &S.full[s], kpol);
            if (!a.kfused) {
              const uint8_t* pg = a.cache + static_cast<int64_t>(page) * a.page_stride;
              bulk_g2s_hint(&S.k[s][kScOff + p * a.R * 2], pg + a.s_off, a.R * 2, &S.full[s], kpol);
            }
          }
        }
      } else {
        // pages were looked up (and range-checked) by the candidate kernel
        const int32_t first = c.tile * (kTile / kBlock);
        const int32_t nblk = min(kTile / kBlock, cn_nc - first);
        const int32_t blk = cn_blk, page = cn_page;
        // the block's scales (gathered by the candidate kernel) go to the
        // stage by plain stores, ordered before lane 0's arrival on it
        if (lane < nblk) *reinterpret_cast<uint4*>(&S.k[s][kScOff + lane * kBlock * 2]) = cn_sc;
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&S.full[s], nblk * (kBlock * kHeadDim));
        __syncwarp();
        if (lane < nblk) {
          const int32_t row = (blk * kBlock) % a.R;
          tma_load_3d_hint(&S.k[s][lane * kBlock * kHeadDim], &tm_blk, 0, row, page, &S.full[s], kpol);
        }
        c.next(a, u0 + k + 1);
        if (k + 1 < nk) consumer_fetch(c);
      }
      __syncwarp();
      ++issued;
    }
    // never leave a copy in flight: wait for the last stages issued
    if (lane == 0) {
      for (int k = max(0, issued - kKStages); k < issued; ++k)
        (void)mbar_wait_drain(&S.full[k % kKStages], (k / kKStages) & 1);
    }
    if (!ok && lane == 0) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  } else if (kCand && (warp == kProdWarp0 || warp == kProdWarp1)) {
    // ---------------- producers of candidate tiles: warp kProdWarp0 takes
    // the even tiles, kProdWarp1 the odd ones; a tile's candidate count,
    // this lane's block, its page and scales are loaded while the
    // producer's previous tile is issued
    const int pp = warp == kProdWarp0 ? 0 : 1;
    const uint64_t kpol = l2_policy_evict_first();
    Cursor c;
    c.init(a, u0 + pp);
    int last = -1;
    int32_t cn_nc = 0, cn_blk = 0, cn_page = 0;
    uint4 cn_sc = make_uint4(0u, 0u, 0u, 0u);
    const auto fetch = [&](const Cursor& at) {
      const int32_t t = at.t;
      const int64_t i = static_cast<int64_t>(t) * a.C + at.tile * (kTile / kBlock) + lane;
      cn_nc = a.cand_cnt[t];
      if (at.tile * (kTile / kBlock) + lane < a.C) {
        cn_blk = a.cand_list[i];
        cn_page = a.cand_page[i];
        cn_sc = a.cand_sc[i];
      }
    };
    if (pp < nk) fetch(c);
    for (int k = pp; k < nk && ok; k += 2) {
      const int s = k % kKStages;
      const uint32_t ph = (k / kKStages) & 1;
      if (lane == 0) ok = mbar_wait_bounded(&S.empty[s], ph ^ 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // pages were looked up (and range-checked) by the candidate kernel
      const int32_t first = c.tile * (kTile / kBlock);
      const int32_t nblk = min(kTile / kBlock, cn_nc - first);
      const int32_t blk = cn_blk, page = cn_page;
      // the block's scales (gathered by the candidate kernel) go to the
      // stage by plain stores, ordered before lane 0's arrival on it
      if (lane < nblk) *reinterpret_cast<uint4*>(&S.k[s][kScOff + lane * kBlock * 2]) = cn_sc;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&S.full[s], nblk * (kBlock * kHeadDim));
      __syncwarp();
      if (lane < nblk) {
        const int32_t row = (blk * kBlock) % a.R;
        tma_load_3d_hint(&S.k[s][lane * kBlock * kHeadDim], &tm_blk, 0, row, page, &S.full[s],
                         kpol);
      }
      c.next(a, u0 + k + 1);
      c.next(a, u0 + k + 2);
      if (k + 2 < nk) fetch(c);
      __syncwarp();
      last = k;
    }
    // never leave a copy in flight: wait for this producer's last stages
    if (lane == 0) {
      for (int k = max(pp, last - kKStages + 2); k <= last; k += 2)
        (void)mbar_wait_drain(&S.full[k % kKStages], (k / kKStages) & 1);
    }
    if (!ok && lane == 0) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  } else if (warp < kConvWarp0) {
    // ---------------- MMA issuers: warp kMmaWarp0 + p takes tiles k = p mod 2
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_m128(static_cast<uint32_t>(a.N));
      int last = -1;
      for (int k = warp - kMmaWarp0; k < nk; k += 2) {
        const int sa = k % kASlots, sd = k % kDSlots;
        if (!mbar_wait_bounded(&S.afull[sa], (k / kASlots) & 1)) { ok = false; break; }
        if (!mbar_wait_bounded(&S.dfree[sd], ((k / kDSlots) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_col = tmem + sa * kSlotCols;
        const uint32_t d_col = tmem + kDCol0 + sd * kSlotCols;
        const uint32_t b0 = smem_u32(&S.b[k & 1][0]);     // the converting group's queries
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t kb = kk >> 2, koff = (kk & 3) * 32;
          mma_f16_ts(d_col, a_col + kk * 8, sdesc_k_sw128(b0 + kb * (a.N * 128) + koff), idesc,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit(&S.afree[sa]);
        mma_commit(&S.dfull[sd]);
        last = k;
      }
      // this thread's MMAs are complete before the block tears down TMEM
      if (last >= 0) (void)mbar_wait_drain(&S.dfull[last % kDSlots], (last / kDSlots) & 1);
      if (!ok) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
    }
  } else if (warp < kEpiWarp0) {
    // ---------------- converters: row = TMEM lane; group g takes tiles k = g mod 2
    const int grp = (warp - kConvWarp0) >> 2;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int ctid = tid - 32 * kConvWarp0 - 128 * grp;   // 0..127 within the group
    int32_t btok = -1;                       // token whose queries sit in the group's buffer
    int32_t wtok = -1;                       // token whose w * q_scale this thread holds
    __half wq_own = __ushort_as_half(0);
    Cursor c;
    c.init(a, u0);
    if (grp == 1) c.next(a, u0 + 1);
    for (int k = grp; k < nk; k += 2) {
      const int sa = k % kASlots, sk = k % kKStages;
      // the A slot must be free: the tensor core has read tile k - kASlots
      if (!mbar_wait_warp(&S.afree[sa], ((k / kASlots) & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      const int32_t t = c.t;
      const int slot = k % kSlots;
      // on a token change its weights and queries are loaded before waiting
      // for the K tile, so the global loads overlap the TMA; within a token
      // the weight * Q scale product stays in a register
      const bool has_w = ctid < a.N;
      if (wtok != t) {
        wtok = t;
        const int64_t wo = static_cast<int64_t>(t) * a.N + ctid;
        const uint16_t wb = has_w ? a.w[wo] : 0, qb = has_w ? a.qs[wo] : 0;
        wq_own = __hmul(__ushort_as_half(wb), __ushort_as_half(qb));
      }
      if (btok != t) {
        // the group's previous tile may still be in the tensor core, reading
        // this buffer: its MMA completes before the buffer is rewritten
        if (k >= 2 && !mbar_wait_warp(&S.afree[(k - 2) % kASlots], ((k - 2) / kASlots) & 1)) {
          ok = false;
          break;
        }
        // queries of token t: FP16 * 2^-10, K-major, 128-byte swizzle
        constexpr int kPer = 64 * 16 / 128;   // chunks per thread at N = 64
        uint2 v[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = ctid + 128 * i;
          const int n = idx >> 4, ch = idx & 15;
          if (idx < a.N * 16)
            v[i] = *reinterpret_cast<const uint2*>(a.q + static_cast<int64_t>(t) * a.q_st +
                                                   static_cast<int64_t>(n) * a.q_sh + ch * 8);
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = ctid + 128 * i;
          const int n = idx >> 4, ch = idx & 15;
          if (idx < a.N * 16)
            *reinterpret_cast<uint4*>(&S.b[grp][sw128_off(a.N, n, ch)]) =
                kFp8 ? e4m3x8_to_f16x8(v[i], true) : i8x8_to_f16x8_div1024(v[i]);
        }
        btok = t;
      }
      if (has_w) S.wq[slot][ctid] = wq_own;
      if (!mbar_wait_warp(&S.full[sk], (k / kKStages) & 1)) { ok = false; break; }
      // this thread's K row, stored 128-byte swizzled by the TMA: logical
      // chunk ch (K elements 16ch..16ch+15) sits at chunk ch ^ (row & 7); a
      // quarter-warp (8 consecutive rows) reads 8 distinct bank groups.
      // Two halves of 64 K values (32 TMEM columns) each.
      // The whole row and its scale go to registers first, so the K stage
      // returns to the producer before any conversion work.
      // a fused page's scale bytes b = 2*row sit in box row 128 + b/128,
      // whose swizzle phase is b/128 (128 is a multiple of 8)
      uint32_t s_at = kScOff + 2 * row;
      if (!consumer && a.kfused) {
        const uint32_t b = 2u * row;
        s_at = kKBytes + (b >> 7) * 128u + ((((b >> 4) & 7u) ^ ((b >> 7) & 7u)) << 4) + (b & 15u);
      }
      const uint8_t* src = &S.k[sk][row * kHeadDim];
      uint4 raw[8];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        raw[ch] = *reinterpret_cast<const uint4*>(src + ((ch ^ (row & 7)) << 4));
      S.ks[slot][row] = __half2float(*reinterpret_cast<const __half*>(&S.k[sk][s_at]));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.empty[sk]);
        mbar_arrive(&S.kready[slot]);
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t regs[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (kFp8) {
            e4m3x16_to_f16x16(raw[4 * half + j], &regs[8 * j]);
          } else {
            cvt_row16(raw[4 * half + j], &regs[8 * j]);
          }
        }
        tmem_st_32x32b_x32(tmem + lane_addr + sa * kSlotCols + 32 * half, regs);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.afull[sa]);
      c.next(a, u0 + k + 1);
      c.next(a, u0 + k + 2);
    }
    if (!ok && lane == 0) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  } else {
    // ---------------- epilogue: row = TMEM lane; group g takes tiles k = g mod 2
    const int grp = (warp - kEpiWarp0) >> 2;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    Cursor c;
    c.init(a, u0);
    if (grp == 1) c.next(a, u0 + 1);
    int32_t vt = -1, V = 0;          // V of the current token, loaded once per token
#ifdef QLI_TEST_STALL_EPILOGUE
    // test build only: the group waits on a barrier nothing arrives on, gives
    // up, and every role that depends on it gives up in turn
    if (!mbar_wait_warp(&S.never, 0)) ok = false;
#endif
    const int k_end = ok ? nk : 0;
    for (int k = grp; k < k_end; k += 2) {
      const int sd = k % kDSlots;
      if (c.t != vt) {
        vt = c.t;
        V = a.tok_V[vt];
      }
      // kready orders the converter's wq / ks writes before this epilogue's
      // reads (its phase cannot run two ahead: the converter of tile
      // k + kSlots needs an accumulator slot this group releases later);
      // dfull says the accumulator is complete
      const int slot = k % kSlots;
      bool w1 = mbar_wait_warp(&S.kready[slot], (k / kSlots) & 1);
      bool w2 = w1 && mbar_wait_warp(&S.dfull[sd], (k / kDSlots) & 1);
      if (!(w1 && w2)) { ok = false; break; }
      tc_fence_after();
      const int32_t t = c.t;
      const uint32_t d_col = tmem + lane_addr + kDCol0 + sd * kSlotCols;
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(d_col, r0);                  // heads 0-31
      if (a.N == 64) tmem_ld_32x32b_x32(d_col + 32, r1);   // heads 32-63 (uniform)
      tmem_ld_wait();
      // the accumulator is in registers: hand its slot back now
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dfree[sd]);
      // w * q_scale pairs, four at a time (16-byte shared loads)
      const uint4* wq4 = reinterpret_cast<const uint4*>(&S.wq[slot][0]);
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = wq4[q];
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          acc = head_pair_acc(acc, __uint_as_float(r0[8 * q + 2 * i]),
                              __uint_as_float(r0[8 * q + 2 * i + 1]), wv[i]);
      }
      if (a.N == 64) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = wq4[4 + q];
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            acc = head_pair_acc(acc, __uint_as_float(r1[8 * q + 2 * i]),
                                __uint_as_float(r1[8 * q + 2 * i + 1]), wv[i]);
        }
      }
      const float score = __fmul_rn(acc, S.ks[slot][row]);

      // scores, and their selection-key histograms for the select stage
      float* srow = a.scores + static_cast<int64_t>(t) * a.Lrow;
      uint32_t* hist = a.fhist + 2 * static_cast<int64_t>(t) * kHistBins;
      if (!consumer) {
        const int32_t pos = c.tile * kTile + row;
        const bool elig = pos < V;
        if (elig) {
          srow[pos] = score;
          atomicAdd(&hist[hist_bin(order_key(score))], 1u);
        }
        if (a.mode == QLI_CAND_SOURCE) {
          float m = elig ? score : -INFINITY;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((row & (kBlock - 1)) == 0 && pos < V) {
            a.bscores[static_cast<int64_t>(t) * a.Brow + pos / kBlock] = m;
            atomicAdd(&hist[kHistBins + hist_bin(order_key(m))], 1u);
          }
        }
      } else {
        const int32_t slot = c.tile * kTile + row;
        if (slot < a.cand_cnt[t] * kBlock) {
          const int32_t pos =
              a.cand_list[static_cast<int64_t>(t) * a.C + slot / kBlock] * kBlock + (row & 7);
          if (pos < V) {
            srow[slot] = score;
            atomicAdd(&hist[hist_bin(order_key(score))], 1u);
          }
        }
      }
      c.next(a, u0 + k + 1);
      c.next(a, u0 + k + 2);
    }
    if (!ok && lane == 0) atomicOr(a.err, QLI_DEVERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace stream

// Tensor map over the index-K rows of the page pool: x = the 128 bytes of a
// row, y = row within the page (`rows` rows, 128 B apart: R, or 130 when a
// 128-row page's 256 bytes of scales follow its rows), z = page (page_stride
// apart); the box is 128 B x box_rows x 1 page, 128-byte swizzle.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_k_map(const DevArgs& d, int rows, int box_rows, CUtensorMap* m) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(d.num_pages)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim),
                                 static_cast<cuuint64_t>(d.page_stride)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  void* base = const_cast<uint8_t*>(d.cache + d.k_off);
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

std::atomic<uint64_t> g_smem_stream_kernel[4] = {{0}, {0}, {0}, {0}};

cudaError_t launch_score(const DevArgs& d, cudaStream_t s) {
  if (d.T == 0) return cudaSuccess;
  if (d.stream_path) {
    CUtensorMap tm_page, tm_blk;
    // with the scales right after a 128-row page's rows, its box runs on
    // over them (two more rows)
    const int page_rows = d.kfused ? d.R + 2 : d.R;
    if (!encode_k_map(d, page_rows, page_rows, &tm_page) || !encode_k_map(d, d.R, kBlock, &tm_blk))
      return cudaErrorInvalidValue;
    // one instance per code type: INT8 (quant mode 2) or E4M3 (quant mode 1)
    // one instance per code type (INT8, quant mode 2, or E4M3, quant mode 1)
    // and per tile kind (dense or candidate blocks)
    const bool cand = d.mode == QLI_CAND_CONSUMER;
    void (*const kinds[4])(CUtensorMap, CUtensorMap, DevArgs) = {
        stream::stream_kernel<false, false>, stream::stream_kernel<false, true>,
        stream::stream_kernel<true, false>, stream::stream_kernel<true, true>};
    const int which = (d.fp8 ? 2 : 0) + (cand ? 1 : 0);
    auto* kern = kinds[which];
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), stream::kSmemBytes,
                                      g_smem_stream_kernel[which]);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(d.num_sms), dim3(stream::threads_for(cand)), stream::kSmemBytes, s,
                   tm_page, tm_blk, d);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  return launch_prefill(d, s);
}

int score_launches(const DevArgs& d) {
  if (d.T == 0) return 0;
  return d.stream_path ? 1 : prefill_launches(d);
}

}  // namespace qli
