// Query quantiser and index-K cache writer: the steps either side of the
// indexer's paged gather (guide "DeepSeek V4.1 QLI V2 与候选集成", section
// 数据流: queries quantised per head to INT8 with an FP16-representable scale;
// index K and its FP16 scales packed after the KV inside each page).
//
// Both are one pass over HBM: read 256 B of BF16 per row, write 128 B of
// codes and a 2 B scale. A half-warp owns a row (lane j holds values
// 8j..8j+7, one 16-byte load), so a warp instruction moves two rows; each
// warp keeps four row pairs in flight. Per row:
//   amax = max |x|, s = FP16(amax / 127) (FP32 quotient, round to nearest
//   even, capped at 65504), q = clamp(rint(x / s), -127, 127) with an FP32
//   quotient; s rounding to zero gives codes 0 and scale +0. The per-element
//   quotient comes from the row's reciprocal and one correction step (a
//   multiply and two FMAs instead of a divide).
// The FP8 variant (quant mode 1, which the guide's section 编译范围 names for
// the A5 build) reads the same scheme with E4M3's largest finite value 448 in
// place of 127: s = FP16(amax / 448), c = E4M3(x / s) from the same FP32
// quotient, rounded to nearest even on the E4M3 grid and saturated to +-448
// (the hardware's satfinite conversion).
#include <cuda_fp16.h>

#include "qli_internal.h"
#include "qli_ptx.cuh"

namespace qli {
namespace {

constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;
constexpr int kQDepth = 4;            // row pairs in flight per warp
constexpr int kRowValues = 128;

// x / sf in FP32, rounded to nearest even, from y = RN(1 / sf): the product
// q0 = RN(x * y) is within about an ulp of the quotient, so the residual
// x - q0 * sf is exact in one FMA and RN(q0 + residual * y) is the correctly
// rounded quotient (Markstein's correction step: P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990). Inputs are BF16 values and FP16 scales, so the domain
// is finite: qli_check_quant_rounding compares every pair with IEEE
// division.
__device__ __forceinline__ float quotient(float x, float sf, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, sf, x);
  return __fmaf_rn(r, y, q0);
}

__device__ __forceinline__ int code_of(float x, float sf, float y) {
  // clamped before the conversion (same result as clamping the integer)
  return __float2int_rn(fminf(fmaxf(quotient(x, sf, y), -127.0f), 127.0f));
}

// FP16(amax / qmax) with the FP32 quotient rounded to nearest even, through
// the same correction step from RN(1/qmax) (qmax 127, or 448 for E4M3);
// capped at the largest finite FP16. The check entry point compares it with
// IEEE division for every BF16 amax.
template <bool kFp8>
__device__ __forceinline__ uint16_t scale_bits_of(float amax) {
  const float qmax = kFp8 ? 448.0f : 127.0f;
  const float rcp = kFp8 ? __uint_as_float(0x3b124925u)    // FP32 nearest 1/448
                         : __uint_as_float(0x3c010204u);   // FP32 nearest 1/127
  const float q = quotient(amax, qmax, rcp);
  uint16_t sb = __half_as_ushort(__float2half_rn(q));
  if (sb == 0x7c00u) sb = 0x7bffu;    // +inf: the largest finite FP16
  return sb;
}

// Two FP32 values to E4M3 codes (round to nearest even, saturated to the
// largest finite magnitude 448): the low byte holds lo's code.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t code_byte(float x, float sf, float y) {
  return static_cast<uint32_t>(code_of(x, sf, y)) & 0xffu;
}

// The half-warp's row: v = this lane's 8 BF16 values. All 32 lanes call it
// (the reduction stays inside each half). Returns the lane's 8 codes.
template <bool kFp8>
__device__ __forceinline__ uint2 quant_half_row(const uint4 v, uint16_t& scale_bits) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  uint16_t sb = scale_bits_of<kFp8>(m);
  const float sf = __half2float(__ushort_as_half(sb));
  uint32_t lo = 0u, hi = 0u;
  if (sf != 0.0f) {
    const float y = __frcp_rn(sf);
    if constexpr (kFp8) {
      // the quotient's sign is x's (s > 0); copysign keeps it where the
      // correction step returns +0 for a negative x below ~2^-100 (an E4M3
      // code of -0 then, as the IEEE quotient gives)
      float c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = copysignf(quotient(x[i], sf, y), x[i]);
      lo = e4m3x2_of(c[0], c[1]) | (e4m3x2_of(c[2], c[3]) << 16);
      hi = e4m3x2_of(c[4], c[5]) | (e4m3x2_of(c[6], c[7]) << 16);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        lo |= code_byte(x[i], sf, y) << (8 * i);
        hi |= code_byte(x[4 + i], sf, y) << (8 * i);
      }
    }
  } else {
    sb = 0u;
  }
  scale_bits = sb;
  return make_uint2(lo, hi);
}

// Row r's destination: the plain [rows, 128] layout, or a page slot.
struct DenseOut {
  int8_t* q;
  uint16_t* scale;
  __device__ __forceinline__ int64_t key(int64_t r) const { return r; }
  __device__ __forceinline__ bool dest(int64_t r, uint2*& codes, uint16_t*& sc) const {
    codes = reinterpret_cast<uint2*>(q + r * kRowValues);
    sc = scale + r;
    return true;
  }
};

struct PagedOut {
  const int64_t* slot;
  uint8_t* cache;
  int64_t slots_total, page_stride, k_offset, scale_offset;
  int32_t R, log2R;                                // R is 64 or 128
  uint32_t* err;
  // the slot, loaded with the row (before any store of the warp)
  __device__ __forceinline__ int64_t key(int64_t r) const { return __ldg(slot + r); }
  __device__ __forceinline__ bool dest(int64_t m, uint2*& codes, uint16_t*& sc) const {
    if (m < 0) return false;                       // padding
    if (m >= slots_total) {
      if (err != nullptr) atomicOr(err, QLI_DEVERR_PAGE);
      return false;
    }
    const int64_t page = m >> log2R, row = m & (R - 1);
    uint8_t* p = cache + page * page_stride;
    codes = reinterpret_cast<uint2*>(p + k_offset + row * kRowValues);
    sc = reinterpret_cast<uint16_t*>(p + scale_offset + row * 2);
    return true;
  }
};

template <class Out, bool kFp8>
__global__ void __launch_bounds__(kQThreads) quant_kernel(const uint16_t* __restrict__ x,
                                                          int64_t rows, Out out) {
  const int lane = threadIdx.x & 31, half = lane >> 4, j = lane & 15;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQWarps;
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * kQWarps + (threadIdx.x >> 5);
  // a warp takes row pairs warp, warp + nwarps, ... kQDepth at a time
  for (int64_t p0 = warp; 2 * p0 < rows; p0 += kQDepth * nwarps) {
    uint4 v[kQDepth];
    int64_t key[kQDepth];
#pragma unroll
    for (int d = 0; d < kQDepth; ++d) {
      const int64_t r = 2 * (p0 + d * nwarps) + half;
      v[d] = make_uint4(0u, 0u, 0u, 0u);
      key[d] = -1;
      if (r < rows) {
        v[d] = __ldcs(reinterpret_cast<const uint4*>(x + r * kRowValues) + j);
        key[d] = out.key(r);
      }
    }
#pragma unroll
    for (int d = 0; d < kQDepth; ++d) {
      const int64_t r = 2 * (p0 + d * nwarps) + half;
      uint16_t sb;
      const uint2 c = quant_half_row<kFp8>(v[d], sb);
      uint2* codes;
      uint16_t* sc;
      if (r < rows && out.dest(key[d], codes, sc)) {
        codes[j] = c;
        if (j == 0) *sc = sb;
      }
    }
  }
}

// Every pair a row can produce: block b takes scale bits b + 1, each thread
// a strided share of the 65536 x patterns. A row has |x| <= amax, and
// amax / s < 1.5 qmax unless s is the 65504 cap (s = FP16(amax / qmax):
// within 2^-11 relative when normal, within 2^-25 absolute when subnormal,
// s >= 2^-24), i.e. below 192 (INT8) or 672 (E4M3); so the pairs are
// |x| <= 768 s, and every finite x for s = 65504.
// counts[0] += pairs whose INT8 code differs from clamp(rint(IEEE x / s)) or
// whose E4M3 code differs from the one of the IEEE quotient, and (the last
// two blocks) BF16 values amax whose scale FP16(amax / 127) or
// FP16(amax / 448) differs from the one an IEEE division gives;
// counts[1] += pairs with |x| >= 2^-100 whose FP32 quotient differs from the
// IEEE one (below that the residual x - q0 s can fall under the FP32 range and
// the correction step loses its exactness; those quotients are < 2^-85 and
// their codes 0 either way, which counts[0] covers).
constexpr unsigned kCheckScaleBlocks = 0x7bffu;   // scale bits 1 .. 0x7bff
__global__ void __launch_bounds__(256) rounding_check_kernel(unsigned long long* counts) {
  if (blockIdx.x >= kCheckScaleBlocks) {
    // the scale: every non-negative finite BF16 amax, for 127 and for 448
    const bool fp8 = blockIdx.x > kCheckScaleBlocks;
    unsigned bad = 0;
    for (uint32_t b = threadIdx.x; b < 0x7f80u; b += blockDim.x) {
      const float m = __uint_as_float(b << 16);
      uint16_t want = __half_as_ushort(__float2half_rn(__fdiv_rn(m, fp8 ? 448.0f : 127.0f)));
      if (want == 0x7c00u) want = 0x7bffu;
      bad += (fp8 ? scale_bits_of<true>(m) : scale_bits_of<false>(m)) != want;
    }
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(counts, bad);
    return;
  }
  const float sf = __half2float(__ushort_as_half(static_cast<uint16_t>(blockIdx.x + 1)));
  const float y = __frcp_rn(sf);
  const float xmax = sf == 65504.0f ? 3.4028235e38f : 768.0f * sf;
  unsigned code_bad = 0, quot_bad = 0;
  for (uint32_t b = threadIdx.x; b < 65536u; b += blockDim.x) {
    const float x = __uint_as_float(b << 16);
    if (!(fabsf(x) <= xmax)) continue;              // also skips Inf and NaN
    const float ieee = __fdiv_rn(x, sf);
    const float fast = quotient(x, sf, y);
    const int want = min(max(__float2int_rn(ieee), -127), 127);
    code_bad += code_of(x, sf, y) != want;
    code_bad += (e4m3x2_of(copysignf(fast, x), 0.0f) & 0xffu) != (e4m3x2_of(ieee, 0.0f) & 0xffu);
    quot_bad += fabsf(x) >= 7.88860905e-31f && __float_as_uint(fast) != __float_as_uint(ieee);
  }
  for (int o = 16; o > 0; o >>= 1) {
    code_bad += __shfl_xor_sync(0xffffffffu, code_bad, o);
    quot_bad += __shfl_xor_sync(0xffffffffu, quot_bad, o);
  }
  if ((threadIdx.x & 31) == 0 && (code_bad | quot_bad)) {
    atomicAdd(counts, code_bad);
    atomicAdd(counts + 1, quot_bad);
  }
}

unsigned quant_grid(int64_t rows, int sms) {
  const int64_t pairs = (rows + 1) / 2;
  const int64_t want = (pairs + kQWarps - 1) / kQWarps;
  const int64_t cap = static_cast<int64_t>(sms) * (2048 / kQThreads);
  return static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <bool kFp8>
qli_status quantize_rows(const uint16_t* x, int64_t rows, void* q_out, uint16_t* scale_out,
                         void* stream) {
  if (rows < 0) return QLI_ERR_INVALID_ARG;
  if (rows == 0) return QLI_OK;
  if (!x || !q_out || !scale_out) return QLI_ERR_INVALID_ARG;
  if (!aligned_to(x, 16) || !aligned_to(q_out, 16) || !aligned_to(scale_out, 2))
    return QLI_ERR_ALIGNMENT;
  int sms = 0;
  const qli_status st = device_sms(&sms);
  if (st != QLI_OK) return st;
  quant_kernel<DenseOut, kFp8>
      <<<quant_grid(rows, sms), kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(
          x, rows, DenseOut{static_cast<int8_t*>(q_out), scale_out});
  return cudaGetLastError() == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

template <bool kFp8>
qli_status write_rows(const uint16_t* k, int64_t n, const int64_t* slot_mapping, uint8_t* cache,
                      int64_t num_pages, int64_t page_stride, int32_t rows_per_page,
                      int64_t k_offset, int64_t scale_offset, uint32_t* err_word, void* stream) {
  if (n < 0 || num_pages < 0) return QLI_ERR_INVALID_ARG;
  if (n == 0) return QLI_OK;
  if (!k || !slot_mapping || !cache) return QLI_ERR_INVALID_ARG;
  if (rows_per_page != 64 && rows_per_page != 128) return QLI_ERR_UNSUPPORTED;
  if (page_stride <= 0 || k_offset < 0 || scale_offset < 0 ||
      k_offset + static_cast<int64_t>(rows_per_page) * 128 > page_stride ||
      scale_offset + static_cast<int64_t>(rows_per_page) * 2 > page_stride)
    return QLI_ERR_INVALID_ARG;
  if (!aligned_to(k, 16) || !aligned_to(cache, 16) || page_stride % 16 != 0 || k_offset % 16 != 0 ||
      scale_offset % 2 != 0 || !aligned_to(slot_mapping, 8) ||
      (err_word != nullptr && !aligned_to(err_word, 4)))
    return QLI_ERR_ALIGNMENT;
  int sms = 0;
  const qli_status st = device_sms(&sms);
  if (st != QLI_OK) return st;
  const PagedOut out{slot_mapping, cache, num_pages * rows_per_page, page_stride, k_offset,
                     scale_offset, rows_per_page, rows_per_page == 64 ? 6 : 7, err_word};
  quant_kernel<PagedOut, kFp8>
      <<<quant_grid(n, sms), kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(k, n, out);
  return cudaGetLastError() == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

}  // namespace
}  // namespace qli

extern "C" qli_status qli_quantize_q(const uint16_t* x, int64_t rows, int8_t* q_out,
                                     uint16_t* scale_out, void* stream) {
  return qli::quantize_rows<false>(x, rows, q_out, scale_out, stream);
}

extern "C" qli_status qli_quantize_q_fp8(const uint16_t* x, int64_t rows, uint8_t* q_out,
                                         uint16_t* scale_out, void* stream) {
  return qli::quantize_rows<true>(x, rows, q_out, scale_out, stream);
}

extern "C" qli_status qli_write_index_k(const uint16_t* k, int64_t n, const int64_t* slot_mapping,
                                        uint8_t* cache, int64_t num_pages, int64_t page_stride,
                                        int32_t rows_per_page, int64_t k_offset,
                                        int64_t scale_offset, uint32_t* err_word, void* stream) {
  return qli::write_rows<false>(k, n, slot_mapping, cache, num_pages, page_stride, rows_per_page,
                                k_offset, scale_offset, err_word, stream);
}

extern "C" qli_status qli_write_index_k_fp8(const uint16_t* k, int64_t n,
                                            const int64_t* slot_mapping, uint8_t* cache,
                                            int64_t num_pages, int64_t page_stride,
                                            int32_t rows_per_page, int64_t k_offset,
                                            int64_t scale_offset, uint32_t* err_word,
                                            void* stream) {
  return qli::write_rows<true>(k, n, slot_mapping, cache, num_pages, page_stride, rows_per_page,
                               k_offset, scale_offset, err_word, stream);
}

extern "C" qli_status qli_check_quant_rounding(unsigned long long* counts, void* stream) {
  using namespace qli;
  if (!counts) return QLI_ERR_INVALID_ARG;
  if (!aligned_to(counts, 8)) return QLI_ERR_ALIGNMENT;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(counts, 0, 2 * sizeof(unsigned long long), st) != cudaSuccess)
    return QLI_ERR_CUDA;
  rounding_check_kernel<<<kCheckScaleBlocks + 2, 256, 0, st>>>(counts);
  return cudaGetLastError() == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

