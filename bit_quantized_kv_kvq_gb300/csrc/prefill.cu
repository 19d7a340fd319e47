// Prefill dispatch by value codec (the kernels live in prefill_impl.cuh).
#include "prefill_impl.cuh"

namespace kvq {

cudaError_t launch_prefill(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                           cudaStream_t st) {
  if (seq_len <= 0) return cudaSuccess;
  switch (L.v.bits) {
    case 3: return launch_prefill_v3(L, k, v, seq_len, st);
    case 4: return launch_prefill_v4(L, k, v, seq_len, st);
    default: return launch_prefill_v8(L, k, v, seq_len, st);
  }
}

}  // namespace kvq
