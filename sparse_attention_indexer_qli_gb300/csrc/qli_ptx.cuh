// Thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers, the tcgen05 tensor-core path (TMEM allocation, MMA, commit,
// TMEM loads) and bounded waits. Every wait here gives up after a time limit
// and reports it, so that no kernel can spin forever.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace qli {

// Give up an on-chip pipeline wait after this long (ns of %globaltimer).
// A test build lowers it (QLI_WAIT_LIMIT_NS) to check the give-up path.
#ifndef QLI_WAIT_LIMIT_NS
#define QLI_WAIT_LIMIT_NS (200ull * 1000ull * 1000ull)
#endif
constexpr uint64_t kWaitLimitNs = QLI_WAIT_LIMIT_NS;
// Waits for a thread's own asynchronous work (TMA copies it issued, MMAs it
// committed) before teardown. That work completes by itself, so this limit
// stays long in every build: a role that gave up on its pipeline still
// drains what it started before the CTA frees TMEM or exits.
constexpr uint64_t kDrainLimitNs = 200ull * 1000ull * 1000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ----------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One probe of the phase with the given parity. The thread may be parked by
// the hardware until the phase completes or a time passes, so a waiting warp
// does not spin on the shared-memory pipe: the system-defined time, or with
// kLongSuspend a 20 us hint. The hint measured ~3% slower per tile in the
// streaming kernel and the attention, and ~3.5% faster in the prefill
// kernel, which takes it.
template <bool kLongSuspend = false>
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kLongSuspend) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false once
// `limit_ns` have passed without it.
template <bool kLongSuspend = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait<kLongSuspend>(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait<kLongSuspend>(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// The same for the drain of a thread's own copies or MMAs at teardown.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  return mbar_wait_bounded(bar, parity, kDrainLimitNs);
}

// Same, for a whole warp waiting on one barrier: lane 0 probes, the result
// is broadcast, and __syncwarp orders the other lanes after lane 0's
// observation of the completed phase.
template <bool kLongSuspend = false>
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded<kLongSuspend>(bar, parity);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bulk (non-tensor) TMA copy global -> shared, completing `bytes` on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled TMA load of a 3-D box (x = bytes of a row, y = row, z = page)
// into shared memory, completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int32_t x, int32_t y,
                                            int32_t z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// An L2 policy that marks lines for early eviction: for data read exactly
// once (the index-K stream), so that it does not push out what a later
// kernel reads again (score rows, histograms).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_3d / bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const void* tmap, int32_t x, int32_t y,
                                                 int32_t z, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Pulls a kernel-parameter tensor map into the descriptor cache ahead of its
// first TMA use.
__device__ __forceinline__ void prefetch_tensormap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---- programmatic dependent launch -----------------------------------------
// A kernel launched with programmatic stream serialisation may start before
// its predecessor finishes; pdl_wait() blocks until the predecessor grid has
// completed and its writes are visible (a no-op for a normal launch), so it
// must precede every read of the predecessor's outputs. pdl_trigger() lets
// the next kernel in the stream begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- proxy / tcgen05 fences ---------------------------------------------
// Makes generic-proxy writes to shared memory visible to the async proxy
// (the tensor core reads its operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- TMEM allocation (one full warp) -----------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// ---- descriptors ---------------------------------------------------------
// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: 8-row groups of 128-byte rows, 1024 bytes apart (SBO);
// the leading-dimension offset is unused for this layout. Bits: start
// address >> 4 at [0,14), LBO >> 4 at [16,30), SBO >> 4 at [32,46), the
// descriptor version 1 at [46,49), swizzle mode 2 (128 B) at [61,64).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;                 // LBO: 16 B (ignored)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // SBO: 1024 B
  d |= static_cast<uint64_t>(1) << 46;                 // version
  d |= static_cast<uint64_t>(2) << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: FP16 A and B (K-major), FP32 D,
// M = 128, N = n (multiple of 16, 16..256). D format at [4,6), A/B formats
// at [7,10)/[10,13) (0 = F16), N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16_m128(uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A is 128 lanes (rows) x K/2 columns,
// two FP16 values per 32-bit column (lower K index in the low half).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (warp's lane quarter base + i), columns col..col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 32 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 64 consecutive 32-bit columns from registers: thread i of the
// warp writes lane (warp's lane quarter base + i), columns col..col+63.
__device__ __forceinline__ void tmem_st_32x32b_x64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]),
      "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]),
      "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]),
      "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]),
      "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- FP8 (E4M3) codes -------------------------------------------------------
// Every E4M3 value (largest 448, smallest 2^-9) is an FP16 value, so these
// widenings are exact; so is the product by 2^-10 (the results stay FP16
// values, subnormals included: the smallest is 2^-19).
// Two codes (the low byte is the lower K index) -> two FP16 values.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(r)
      : "r"(two_codes));
  return r;
}
// 8 codes -> 8 FP16 values, optionally times 2^-10.
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 v, bool div1024) {
  uint32_t o[4] = {e4m3x2_to_f16x2(v.x & 0xFFFFu), e4m3x2_to_f16x2(v.x >> 16),
                   e4m3x2_to_f16x2(v.y & 0xFFFFu), e4m3x2_to_f16x2(v.y >> 16)};
  if (div1024) {
    const __half2 s = __floats2half2_rn(1.0f / 1024.0f, 1.0f / 1024.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 x = __hmul2(*reinterpret_cast<__half2*>(&o[k]), s);
      o[k] = *reinterpret_cast<uint32_t*>(&x);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// 16 codes -> 16 FP16 values as 8 words (lower K index in the low half).
__device__ __forceinline__ void e4m3x16_to_f16x16(const uint4 v, uint32_t* out8) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    out8[2 * k] = e4m3x2_to_f16x2(w[k] & 0xFFFFu);
    out8[2 * k + 1] = e4m3x2_to_f16x2(w[k] >> 16);
  }
}

// ---- selection keys -------------------------------------------------------
// Order-preserving map of a finite FP32 score to a non-zero uint32 key
// (larger score -> larger key; -0 and +0 map to the same key). Key 0 is kept
// for "not eligible". The score stage histograms the top 12 key bits.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0) u = 0;   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
__device__ __forceinline__ uint32_t hist_bin(uint32_t key) { return key >> (32 - kHistBits); }

// ---- the golden chain, one head ----------------------------------------
// acc += fp32( fp16( relu(fp16(s)) * wq ) ), where s already holds the
// exact INT32 dot / 1024 in FP32 and wq = fp16(w * q_scale).
__device__ __forceinline__ float head_term_acc(float acc, float s, __half wq) {
  uint16_t x, p;
  asm("cvt.rn.relu.f16.f32 %0, %1;" : "=h"(x) : "f"(s));
  asm("mul.rn.f16 %0, %1, %2;" : "=h"(p) : "h"(x), "h"(__half_as_ushort(wq)));
  float r;
  asm("{\n\t.reg .f16 t;\n\tmov.b16 t, %1;\n\tadd.rn.f32.f16 %0, t, %2;\n\t}"
      : "=f"(r)
      : "h"(p), "f"(acc));
  return r;
}

// Two heads of the golden chain at once: x = fp16x2(relu(s_hi), relu(s_lo))
// (one rounding each), p = x * wq2 (IEEE FP16 multiplies), then
// acc += fp32(p.lo); acc += fp32(p.hi) — head `lo` before head `hi`.
__device__ __forceinline__ float head_pair_acc(float acc, float s_lo, float s_hi, uint32_t wq2) {
  uint32_t x, p;
  asm("cvt.rn.relu.f16x2.f32 %0, %1, %2;" : "=r"(x) : "f"(s_hi), "f"(s_lo));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(x), "r"(wq2));
  float r;
  asm("{\n\t.reg .f16 lo, hi;\n\t.reg .f32 t;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.f16 t, lo, %2;\n\tadd.rn.f32.f16 %0, hi, t;\n\t}"
      : "=f"(r)
      : "r"(p), "f"(acc));
  return r;
}

}  // namespace qli
