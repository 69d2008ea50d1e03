// Small decode batches (at most 64 tokens and 64 requests, contexts of at
// most 4096 compressed positions, INT8, none or source mode): the whole
// indexer in one kernel, so that a call is one memset and one launch.
//
// Guide "DeepSeek V4.1 QLI V2 与候选集成", sections 数据流 and 当前 A3 契约:
// score(t, j) = ks(j) * sum_h FP16(relu(FP16(q_h . k_j / 1024)) * FP16(w_h * qs_h))
// with the head terms added in FP32 in ascending h; then the TopK positions
// (and in source mode the candidate blocks) in ascending order, -1 padded.
//
// CTA (tile, t) scores positions 64*tile .. +63 of token t: the K rows are
// gathered through the block table into shared memory, the INT32 dots come
// from __dp4a (exact), and the chain runs per position in the same FP16/FP32
// operations as the streaming kernel's epilogue (head_pair_acc). The scores
// (and source block maxima) go to the workspace rows; the last CTA of a token
// to finish (a counter that a one-CTA kernel launched just before zeroed)
// ranks the token's rows with the shared one-CTA selection (fast_row), which
// for rows this short keeps every entry in shared memory and never defers to
// the general selection. The scoring kernel starts while the zeroing kernel
// runs (programmatic launch) and waits for it only before it touches the
// counters or the error word.
#include <cuda_fp16.h>

#include "qli_fast_select.cuh"
#include "qli_internal.h"
#include "qli_meta.cuh"
#include "qli_ptx.cuh"

namespace qli {
namespace {

constexpr int kST = kFT;                    // threads; fast_row runs on the same CTA
constexpr int kSmallMaxB = 64;
constexpr int kKWords = kHeadDim / 4;       // 32 words of four INT8 per K row
constexpr int kKPitch = kKWords + 1;        // padded row pitch: column reads are conflict-free
constexpr int kSP = 64;                     // positions per CTA
constexpr int kPI = kSP / 32;               // positions per lane
static_assert(kST == 256 && kSP % 32 == 0, "thread mapping: 32 lanes x kPI positions, 8 head groups");

struct SmallSmem {
  int32_t q0s[kSmallMaxB], q1s[kSmallMaxB], lks[kSmallMaxB], ress[kSmallMaxB];
  int32_t V, owner, last;
  uint32_t err;                             // error bits, reported once the counters are zeroed
  int32_t page[kSP];                        // each row's page (checked)
  uint32_t k[kSP * kKPitch];                // the CTA's K rows (words of 4 INT8)
  uint32_t qT[kKWords * 64];                // queries transposed: word c of head h at [c][h]
  float dT[64 * kSP];                       // q.k / 1024 (exact), head-major
  __half wq[64];                            // FP16(w * q_scale)
  float ks[kSP];                            // K scales
};
constexpr size_t kSmallSmem = sizeof(SmallSmem) > sizeof(FastSmem) ? sizeof(SmallSmem)
                                                                    : sizeof(FastSmem);

template <int N>
__global__ void __launch_bounds__(kST, 1) small_kernel(DevArgs a) {
  extern __shared__ __align__(16) uint8_t raw[];
  SmallSmem& S = *reinterpret_cast<SmallSmem*>(raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, t = blockIdx.y;
  const bool reporter = tile == 0 && t == 0;

  // ---- the token's queries and weights go out first (they need no metadata)
  constexpr int kQPer = N * 8 / kST;                // 16-byte pieces of q per thread
  const int8_t* qt = a.q + static_cast<int64_t>(t) * a.q_st;
  uint4 qv[kQPer];
#pragma unroll
  for (int j = 0; j < kQPer; ++j) {
    const int i = tid + j * kST, h = i >> 3, ch = i & 7;
    qv[j] = __ldg(reinterpret_cast<const uint4*>(qt + static_cast<int64_t>(h) * a.q_sh) + ch);
  }
  uint16_t wb = 0, qb = 0;
  if (tid < N) {
    wb = a.w[static_cast<int64_t>(t) * N + tid];
    qb = a.qs[static_cast<int64_t>(t) * N + tid];
  }
  // ---- metadata, read as the planning stage reads it
  if (tid == 0) S.err = 0u;
  __syncthreads();
  if (tid < a.B) {
    int32_t q0, q1, lk, res;
    const uint32_t e = sanitize_request(a, tid, q0, q1, lk, res);
    S.q0s[tid] = q0;
    S.q1s[tid] = q1;
    S.lks[tid] = lk;
    S.ress[tid] = res;
    if (e && reporter) atomicOr(&S.err, e);
  }
  __syncthreads();
  if (tid == 0) {
    int32_t owner;
    S.V = token_owner(a, S.q0s, S.q1s, S.lks, S.ress, t, owner);
    S.owner = owner;
  }
  __syncthreads();
  const int32_t V = S.V, owner = S.owner;
  const int32_t p0 = tile * kSP;
  const int32_t npos = min(max(V - p0, 0), kSP);

  if (npos > 0) {
    // ---- each row's page from the block table; a page outside the pool
    // sets QLI_DEVERR_PAGE and reads page 0 instead
    const int64_t bt_row = static_cast<int64_t>(owner) * a.bt_stride;
    if (tid < npos) {
      int32_t page = a.bt[bt_row + (p0 + tid) / a.R];
      if (page < 0 || page >= a.num_pages) {
        atomicOr(&S.err, QLI_DEVERR_PAGE);
        page = 0;
      }
      S.page[tid] = page;
    }
#pragma unroll
    for (int j = 0; j < kQPer; ++j) {
      const int i = tid + j * kST, h = i >> 3, ch = i & 7;
      S.qT[(4 * ch + 0) * N + h] = qv[j].x;
      S.qT[(4 * ch + 1) * N + h] = qv[j].y;
      S.qT[(4 * ch + 2) * N + h] = qv[j].z;
      S.qT[(4 * ch + 3) * N + h] = qv[j].w;
    }
    if (tid < N) S.wq[tid] = __hmul(__ushort_as_half(wb), __ushort_as_half(qb));
    __syncthreads();
    // ---- the tile's K rows and scales, all loads in flight at once
    constexpr int kKPer = kSP * 8 / kST;
    uint4 kv[kKPer];
#pragma unroll
    for (int j = 0; j < kKPer; ++j) {
      const int i = tid + j * kST, r = i >> 3, ch = i & 7;
      kv[j] = make_uint4(0u, 0u, 0u, 0u);
      if (r < npos) {
        const uint8_t* pg = a.cache + static_cast<int64_t>(S.page[r]) * a.page_stride;
        kv[j] = __ldg(reinterpret_cast<const uint4*>(
                          pg + a.k_off + static_cast<int64_t>((p0 + r) % a.R) * kHeadDim) + ch);
      }
    }
    if (tid < npos) {
      const uint8_t* pg = a.cache + static_cast<int64_t>(S.page[tid]) * a.page_stride;
      S.ks[tid] = __half2float(__ushort_as_half(
          __ldg(reinterpret_cast<const uint16_t*>(pg + a.s_off) + (p0 + tid) % a.R)));
    }
#pragma unroll
    for (int j = 0; j < kKPer; ++j) {
      const int i = tid + j * kST, r = i >> 3, ch = i & 7;
      uint32_t* dst = S.k + r * kKPitch + 4 * ch;
      dst[0] = kv[j].x;
      dst[1] = kv[j].y;
      dst[2] = kv[j].z;
      dst[3] = kv[j].w;
    }
    __syncthreads();
    // ---- exact INT32 dots: lane l takes positions l + 32i, warp w heads
    // w*HPT .. w*HPT + HPT-1
    constexpr int HPT = N / 8;
    int32_t acc[kPI][HPT];
#pragma unroll
    for (int i = 0; i < kPI; ++i)
#pragma unroll
      for (int h = 0; h < HPT; ++h) acc[i][h] = 0;
#pragma unroll 4
    for (int c = 0; c < kKWords; ++c) {
      int32_t kw[kPI];
#pragma unroll
      for (int i = 0; i < kPI; ++i) kw[i] = static_cast<int32_t>(S.k[(lane + 32 * i) * kKPitch + c]);
      int32_t qw[HPT];
#pragma unroll
      for (int h4 = 0; h4 < HPT; h4 += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(&S.qT[c * N + warp * HPT + h4]);
        qw[h4] = static_cast<int32_t>(v.x);
        qw[h4 + 1] = static_cast<int32_t>(v.y);
        qw[h4 + 2] = static_cast<int32_t>(v.z);
        qw[h4 + 3] = static_cast<int32_t>(v.w);
      }
#pragma unroll
      for (int i = 0; i < kPI; ++i)
#pragma unroll
        for (int h = 0; h < HPT; ++h) acc[i][h] = __dp4a(kw[i], qw[h], acc[i][h]);
    }
    // |dot| < 2^21, so dot / 1024 is exact in FP32
#pragma unroll
    for (int i = 0; i < kPI; ++i)
#pragma unroll
      for (int h = 0; h < HPT; ++h)
        S.dT[(warp * HPT + h) * kSP + lane + 32 * i] = static_cast<float>(acc[i][h]) * (1.0f / 1024.0f);
    __syncthreads();
    // ---- the chain per position, heads in ascending order, as the
    // streaming kernel's epilogue computes it
    if (tid < kSP) {
      const int32_t pos = p0 + tid;
      const bool elig = tid < npos;
      float sacc = 0.0f;
      const uint32_t* wq2 = reinterpret_cast<const uint32_t*>(S.wq);
#pragma unroll
      for (int h = 0; h < N; h += 2)
        sacc = head_pair_acc(sacc, S.dT[h * kSP + tid], S.dT[(h + 1) * kSP + tid], wq2[h >> 1]);
      const float score = __fmul_rn(sacc, S.ks[tid]);
      if (elig) a.scores[static_cast<int64_t>(t) * a.Lrow + pos] = score;
      if (a.mode == QLI_CAND_SOURCE) {
        float m = elig ? score : -INFINITY;
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        if ((tid & (kBlock - 1)) == 0 && elig)
          a.bscores[static_cast<int64_t>(t) * a.Brow + pos / kBlock] = m;
      }
    }
  }

  // ---- the last CTA of token t ranks its rows (the counters and the error
  // word are zeroed by the kernel launched before this one). The counter is
  // an acquire-release atomic: it publishes this CTA's scores (ordered
  // before it by the barrier) and, in the last CTA, makes every other CTA's
  // scores visible to the threads that read them after the next barrier.
  __syncthreads();
  pdl_wait();
  if (tid == 0) {
    if (S.err) atomicOr(a.err, S.err);
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(old) : "l"(a.done + t) : "memory");
    S.last = old == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!S.last) return;
  if (tid == 0) {
    a.tok_V[t] = V;
    a.tok_b[t] = owner;
  }
  __syncthreads();
  FastSmem& F = *reinterpret_cast<FastSmem*>(raw);
  fast_row(a, t, 0, V, owner, F);
  if (a.mode == QLI_CAND_SOURCE) {
    __syncthreads();
    fast_row(a, t, 1, V, owner, F);
  }
}

// The error word, the spare counter and the per-token counters, zeroed.
__global__ void __launch_bounds__(128) small_zero_kernel(uint32_t* words, int32_t n) {
  pdl_trigger();
  for (int i = threadIdx.x; i < n; i += blockDim.x) words[i] = 0u;
}

}  // namespace

bool use_small_path(const qli_args& a) {
  const int64_t cap = static_cast<int64_t>(a.bt_stride) * a.rows_per_page;
  return a.T > 0 && a.cand_mode != QLI_CAND_CONSUMER && a.quant_mode == QLI_QUANT_INT8 &&
         use_stream_path(a) && a.B <= kSmallMaxB && a.T <= kSmallMaxT && cap <= kSmallMaxPositions;
}

cudaError_t launch_small_zero(const DevArgs& d, size_t bytes, cudaStream_t s) {
  small_zero_kernel<<<1, 128, 0, s>>>(d.err, static_cast<int32_t>(bytes / 4));
  return cudaGetLastError();
}

cudaError_t launch_small(const DevArgs& d, cudaStream_t s) {
  static std::atomic<uint64_t> done[2] = {{0}, {0}};
  void (*const kern)(DevArgs) = d.N == 64 ? small_kernel<64> : small_kernel<32>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), static_cast<int>(kSmallSmem),
                                    done[d.N == 64 ? 1 : 0]);
  if (e != cudaSuccess) return e;
  const unsigned tiles = static_cast<unsigned>((d.cap + kSP - 1) / kSP);
  e = launch_pdl(kern, dim3(tiles > 0 ? tiles : 1u, static_cast<unsigned>(d.T)), dim3(kST),
                 kSmallSmem, s, d);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qli
