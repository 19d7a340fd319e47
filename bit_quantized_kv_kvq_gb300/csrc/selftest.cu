// Device self-tests (kvq_selftest.h): the quantizer's division-free code
// arithmetic against IEEE division over exhaustive or adversarial inputs,
// and the kernels' bounded wait made to give up on a barrier that is never
// completed.
#include <cstdint>
#include <cstdio>

#include "codebook.cuh"
#include "kvq_internal.h"
#include "kvq_selftest.h"
#include "prefill_fast.cuh"

namespace {

using kvq::pfx::div_levels;
using kvq::pfx::recip_bracket;
using kvq::pfx::resolve_code;
using kvq::pfx::rne_prod;

constexpr int kBlocks = 1216;  // 8 per SM of a 152-SM GPU
constexpr int kThreads = 256;

__device__ __forceinline__ void note_mismatch(unsigned long long* res, unsigned long long key) {
  atomicAdd(&res[0], 1ull);
  atomicMin(&res[1], key);
}

template <int L>
__global__ void __launch_bounds__(kThreads) div_levels_kernel(uint32_t a_first, uint32_t a_last,
                                                             unsigned long long* res) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)a_first + blockIdx.x * blockDim.x + threadIdx.x; i <= a_last; i += stride) {
    const float a = __uint_as_float((uint32_t)i);
    const float got = div_levels<L>(a);
    const float want = __fdiv_rn(a, (float)L);
    if (__float_as_uint(got) != __float_as_uint(want)) note_mismatch(res, i);
  }
}

// One thread per (scale, k); the dividends are RN((k + 1/2) s) +- j ulps.
__global__ void __launch_bounds__(kThreads) code_rounding_kernel(int method, uint32_t s_first, uint32_t s_count,
                                                                int k_first, int k_count, int ulps,
                                                                unsigned long long* res) {
  const uint64_t n = (uint64_t)s_count * k_count;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += stride) {
    const uint32_t sb = s_first + (uint32_t)(t / k_count);
    const int ki = (int)(t % k_count);
    const int k = k_first + ki;
    const float s = __half2float(__ushort_as_half((unsigned short)sb));
    const float d0 = __fmul_rn((float)k + 0.5f, s);
    if (d0 == 0.0f || !isfinite(d0)) continue;
    const float r = __frcp_rn(s);
    float rlo = 0.0f, rhi = 0.0f;
    if (method == 1) recip_bracket(s, rlo, rhi);
    for (int j = -ulps; j <= ulps; ++j) {
      // j units in the last place of |d0|, away from zero for j > 0
      const float d = __uint_as_float((uint32_t)((int32_t)__float_as_uint(d0) + j));
      if (d == 0.0f || !isfinite(d) || (d < 0.0f) != (d0 < 0.0f)) continue;
      const int want = __float2int_rn(__fdiv_rn(d, s));
      int got;
      if (method == 0) {
        got = kvq::quant_step(d, s, r);
      } else {
        const int a = rne_prod(d, rlo), b = rne_prod(d, rhi);
        got = a == b ? a : resolve_code(d, s, a);
      }
      if (got != want)
        note_mismatch(res, ((unsigned long long)sb << 32) | ((unsigned long long)ki << 8) | (unsigned)(j + ulps));
    }
  }
}

// Every (finite fp16 x, positive finite fp16 s): the codebook quantizer's
// quotient against IEEE division, compared as values (+0 == -0).
__global__ void __launch_bounds__(kThreads) codebook_quotient_kernel(unsigned long long* res) {
  const uint64_t n = (uint64_t)0x7BFFu * 0x10000u;  // s bits 0x0001..0x7BFF, x bits 0x0000..0xFFFF
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += stride) {
    const uint32_t sb = 1u + (uint32_t)(t >> 16), xb = (uint32_t)(t & 0xFFFFu);
    const float x = __half2float(__ushort_as_half((unsigned short)xb));
    if (!isfinite(x)) continue;
    const float s = __half2float(__ushort_as_half((unsigned short)sb));
    const float got = kvq::cb::quotient(x, s, __frcp_rn(s));
    const float want = __fdiv_rn(x, s);
    if (!(got == want)) note_mismatch(res, ((unsigned long long)sb << 16) | xb);
  }
}

// A barrier that nothing completes: the bounded wait must give up, raise
// the timeout bit and let the kernel return.
__global__ void wait_timeout_kernel(uint32_t* status, int polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    kvq::mbar_init(&bar, 1);
    kvq::mbar_fence_init();
  }
  __syncthreads();
  const bool done = kvq::mbar_wait_limited(&bar, 0, polls, kvq::kWaitHintNs);
  if (!done && threadIdx.x == 0) kvq::raise_status(status, kvq::kStatusTimeout);
}

kvq_status fail(kvq_status s, const char* msg) {
  kvq::set_error_message(msg);
  return s;
}

kvq_status launched(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    kvq::count_launches(1);
    return KVQ_OK;
  }
  char msg[256];
  snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
  kvq::set_error_message(msg);
  return KVQ_ERR_CUDA;
}

kvq_status reset_result(void* dev_result, cudaStream_t st) {
  if (!dev_result || (reinterpret_cast<uintptr_t>(dev_result) & 7u))
    return fail(KVQ_ERR_INVALID_ARG, "dev_result must be a non-NULL, 8-byte aligned device pointer");
  cudaError_t e = cudaMemsetAsync(dev_result, 0, 8, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(static_cast<char*>(dev_result) + 8, 0xFF, 8, st);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "clearing dev_result failed");
  return KVQ_OK;
}

}  // namespace

extern "C" {

KVQ_API kvq_status kvq_selftest_div_levels(int32_t levels, uint32_t a_first, uint32_t a_last,
                                           void* dev_result, void* stream) {
  if (a_first > a_last) return fail(KVQ_ERR_INVALID_ARG, "a_first > a_last");
  if (levels != 3 && levels != 7 && levels != 15 && levels != 127 && levels != 255)
    return fail(KVQ_ERR_INVALID_ARG, "levels must be 3, 7, 15, 127 or 255");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const kvq_status s = reset_result(dev_result, st);
  if (s != KVQ_OK) return s;
  auto* res = static_cast<unsigned long long*>(dev_result);
  switch (levels) {
    case 3: div_levels_kernel<3><<<kBlocks, kThreads, 0, st>>>(a_first, a_last, res); break;
    case 7: div_levels_kernel<7><<<kBlocks, kThreads, 0, st>>>(a_first, a_last, res); break;
    case 15: div_levels_kernel<15><<<kBlocks, kThreads, 0, st>>>(a_first, a_last, res); break;
    case 127: div_levels_kernel<127><<<kBlocks, kThreads, 0, st>>>(a_first, a_last, res); break;
    default: div_levels_kernel<255><<<kBlocks, kThreads, 0, st>>>(a_first, a_last, res); break;
  }
  return launched("div_levels self-test launch");
}

KVQ_API kvq_status kvq_selftest_code_rounding(int32_t method, int32_t k_first, int32_t k_last,
                                              int32_t ulps, void* dev_result, void* stream) {
  if (method != 0 && method != 1) return fail(KVQ_ERR_INVALID_ARG, "method must be 0 or 1");
  if (k_first > k_last) return fail(KVQ_ERR_INVALID_ARG, "k_first > k_last");
  if (method == 0 && (k_first < -4096 || k_last > 4096))
    return fail(KVQ_ERR_INVALID_ARG, "method 0 takes k in [-4096, 4096]");
  if (method == 1 && (k_first < 0 || k_last > 255))
    return fail(KVQ_ERR_INVALID_ARG, "method 1 takes k in [0, 255]");
  if (ulps < 0 || ulps > 64) return fail(KVQ_ERR_INVALID_ARG, "ulps must be in [0, 64]");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const kvq_status s = reset_result(dev_result, st);
  if (s != KVQ_OK) return s;
  // positive finite fp16 scales: all of them, or the normal ones
  const uint32_t s_first = method == 0 ? 0x0001u : 0x0400u;
  const uint32_t s_count = 0x7BFFu - s_first + 1u;
  code_rounding_kernel<<<kBlocks, kThreads, 0, st>>>(method, s_first, s_count, k_first, k_last - k_first + 1, ulps,
                                                     static_cast<unsigned long long*>(dev_result));
  return launched("code rounding self-test launch");
}

KVQ_API kvq_status kvq_selftest_codebook_quotient(void* dev_result, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const kvq_status s = reset_result(dev_result, st);
  if (s != KVQ_OK) return s;
  codebook_quotient_kernel<<<kBlocks, kThreads, 0, st>>>(static_cast<unsigned long long*>(dev_result));
  return launched("codebook quotient self-test launch");
}

KVQ_API kvq_status kvq_selftest_wait_timeout(kvq_cache* cache, int32_t polls, void* stream) {
  if (!cache) return fail(KVQ_ERR_INVALID_ARG, "cache handle is NULL");
  if (polls < 1 || polls > 100000) return fail(KVQ_ERR_INVALID_ARG, "polls must be in [1, 100000]");
  const kvq_status s = kvq::cache_device_is_current(cache);
  if (s != KVQ_OK) return s;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(kvq::cache_status_word(cache), polls);
  return launched("wait timeout self-test launch");
}

}  // extern "C"
