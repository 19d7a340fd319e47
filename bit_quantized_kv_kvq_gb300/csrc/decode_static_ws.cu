// Decode attention for callers that cannot allocate device memory.
//
// kvq_decode_attention needs a caller-provided workspace for the per-split
// partial results. Some callers have no way to obtain one: code running
// inside a host callback or a signal-safe path that may not call the CUDA
// allocator, plugins embedded in a host program that owns every allocation,
// or inference servers that forbid allocation after start-up. This file gives
// them kvq_decode_attention_static: the same computation, with its scratch in
// a fixed array that the library itself declares in device memory.
//
// The array lives in every GPU that loads this library until the process
// exits. Its address is looked up once per device (cudaGetSymbolAddress, with
// that device current) by the first call made on that device.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "kvq_internal.h"

namespace {

// Scratch for the split partials of one decode call: B * H_q * splits *
// (D + 2) floats plus alignment padding must fit in it.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

KVQ_API kvq_status kvq_decode_attention_static(kvq_cache* cache, int32_t layer, const void* q,
                                               int32_t num_q_heads, float softmax_scale,
                                               void* out, int32_t out_dtype, void* stream) {
  void* scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "static decode scratch lookup failed: %s", cudaGetErrorString(e));
    kvq::set_error_message(msg);
    return KVQ_ERR_CUDA;
  }
  const kvq_status s = kvq_decode_attention(cache, layer, q, num_q_heads, softmax_scale, out,
                                            out_dtype, scratch, kStaticScratchBytes, stream);
  if (s == KVQ_ERR_BUFFER_TOO_SMALL) {
    char msg[512];
    std::snprintf(msg, sizeof msg,
                  "this decode needs more split scratch than the static maximum of %zu bytes "
                  "(%s); call kvq_decode_attention with a caller workspace instead",
                  kStaticScratchBytes, kvq_last_error());
    kvq::set_error_message(msg);
  }
  return s;
}

}  // extern "C"
