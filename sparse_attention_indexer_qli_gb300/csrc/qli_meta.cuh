// Device-side reading of the per-request metadata, shared by the planning
// stage and the single-launch path for small batches, so that both clamp,
// flag and assign tokens identically.
//
// Guide "DeepSeek V4.1 QLI V2 与候选集成", section 数据流: raw query boundaries
// (cu_seqlens_q), compressed K lengths and the raw length mod ratio (absent
// for ratio 1). Causal mask mode 3 is read as: the queries of a request are
// the last q_len of its S = k_len*ratio + residual raw tokens, and compressed
// position j (raw span [j*r, j*r + r - 1]) is visible to the query at raw
// position pos once pos >= j*r + r - 1, i.e. V = floor((pos + 1) / r).
#pragma once

#include "qli_internal.h"

namespace qli {
namespace {

__device__ __forceinline__ int32_t visible_count(int32_t lk, int32_t res, int32_t ratio,
                                                 int32_t q_len, int32_t i) {
  const int64_t S = static_cast<int64_t>(lk) * ratio + res;
  const int64_t seen = S - q_len + i + 1;   // raw tokens at or before the query
  if (seen <= 0) return 0;
  const int64_t v = seen / ratio;
  return static_cast<int32_t>(v < lk ? v : lk);
}

// Request b on its own: the query range clamped into [0, T], the compressed
// length into [0, cap] and the residual into [0, ratio); returns the error
// bits of what was clamped.
__device__ __forceinline__ uint32_t sanitize_request(const DevArgs& a, int b, int32_t& q0,
                                                     int32_t& q1, int32_t& lk, int32_t& res) {
  uint32_t e = 0u;
  const int32_t c0 = a.cu[b], c1 = a.cu[b + 1];
  lk = a.k_lens[b];
  res = a.residual ? a.residual[b] : 0;
  q0 = min(max(c0, 0), a.T);
  q1 = min(max(c1, q0), a.T);
  if (c0 != q0 || c1 != q1 || (b == 0 && c0 != 0) || (b == a.B - 1 && c1 != a.T))
    e |= QLI_DEVERR_SEQLENS;
  if (lk < 0 || lk > a.cap) {
    e |= QLI_DEVERR_KLEN;
    lk = lk < 0 ? 0 : static_cast<int32_t>(a.cap);
  }
  if (res < 0 || res >= a.ratio) {
    e |= QLI_DEVERR_RESIDUAL;
    res = 0;
  }
  return e;
}

// Token t's request is the last one starting at or before it (the sanitised
// starts never decrease for valid metadata; a token no request covers has
// V = 0 and owner -1). Returns V(t).
__device__ __forceinline__ int32_t token_owner(const DevArgs& a, const int32_t* q0s,
                                               const int32_t* q1s, const int32_t* lks,
                                               const int32_t* ress, int t, int32_t& owner) {
  int32_t lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (q0s[mid] <= t) lo = mid; else hi = mid - 1;
  }
  owner = -1;
  if (a.B > 0 && q0s[lo] <= t && t < q1s[lo]) {
    owner = lo;
    return visible_count(lks[lo], ress[lo], a.ratio, q1s[lo] - q0s[lo], t - q0s[lo]);
  }
  return 0;
}

}  // namespace
}  // namespace qli
