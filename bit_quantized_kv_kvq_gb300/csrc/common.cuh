// Device helpers shared by the kvq kernels: packing geometry, the fp32
// quantizer step, bounded mbarrier waits and 1-D bulk (TMA) copies.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "kvq_internal.h"

namespace kvq {

// ---------------------------------------------------------------------------
// Packing geometry: ten 3-bit codes per word (top two bits zero), eight
// 4-bit codes, four 8-bit codes.
// ---------------------------------------------------------------------------
template <int BITS> struct Pack {
  static constexpr int kCpw = BITS == 3 ? 10 : 32 / BITS;
  static constexpr int kWords = (kHeadDim + kCpw - 1) / kCpw;
  static constexpr uint32_t kMask = (1u << BITS) - 1u;
};

// ---------------------------------------------------------------------------
// Quantizer step in fp32 (TurboQuant 3-bit KV quantization page, §3.1):
// code = rne(d / s) with d = x - z already formed in fp32 and s the fp32
// value of the stored fp16 scale. The result must equal rint() of the IEEE
// quotient. r = RN(1/s) gives d*r within about 1.5 ulp of RN(d/s); the two
// can round to different integers only when d*r lies within that distance of
// a half-integer, so only then is the exact quotient formed.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int quant_step(float d, float s, float r) {
  float qa = __fmul_rn(d, r);
  float fl = floorf(qa);
  float fr = __fsub_rn(qa, fl);  // exact
  float tol = fmaxf(fabsf(qa), 1.0f) * 0x1p-20f;
  if (fabsf(__fsub_rn(fr, 0.5f)) <= tol) qa = __fdiv_rn(d, s);
  return __float2int_rn(qa);
}

// ---------------------------------------------------------------------------
// Status word: bits set by device-side checks, read by kvq_cache_status().
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk copy (cp.async.bulk, global -> shared) helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// try_wait that may suspend the thread for up to `hint_ns` while the phase
// is incomplete (the thread sleeps instead of issuing poll instructions).
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Bounded wait: gives up after `polls` suspended polls of at most hint_ns
// each and reports false, so no thread can wait forever.
__device__ __forceinline__ bool mbar_wait_limited(uint64_t* bar, uint32_t parity, int polls,
                                                  uint32_t hint_ns) {
  for (int it = 0; it < polls; ++it) {
    if (mbar_try_wait_hint(bar, parity, hint_ns)) return true;
  }
  return false;
}

// The kernels' wait: kWaitLimit polls of at most kWaitHintNs (about a second).
constexpr int kWaitLimit = 1 << 17;
constexpr uint32_t kWaitHintNs = 10000;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  return mbar_wait_limited(bar, parity, kWaitLimit, kWaitHintNs);
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (Blackwell f32x2 arithmetic, round to nearest even).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// dst (shared) and src (global) 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace kvq
