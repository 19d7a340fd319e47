// Prefill dispatch: codecs without outliers run the barrier-light kernel of
// prefill_fast.cuh; the rest (outliers, 256-token key blocks) the kernel of
// prefill_impl.cuh.
#include "prefill_impl.cuh"

namespace kvq {

cudaError_t launch_prefill_fast_v30(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                                    cudaStream_t st);
cudaError_t launch_prefill_fast_v40(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                                    cudaStream_t st);
cudaError_t launch_prefill_fast_v80(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                                    cudaStream_t st);
cudaError_t launch_prefill_fast_v81(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                                    cudaStream_t st);

static bool fast_prefill_supported(const LayerDev& L) {
  if (L.outliers != 0) return false;
  if (L.k.mode == KVQ_ASYM_PER_CHANNEL && L.k.group != 64 && L.k.group != 128) return false;
  return true;
}

cudaError_t launch_prefill(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                           cudaStream_t st) {
  if (seq_len <= 0) return cudaSuccess;
  if (fast_prefill_supported(L)) {
    if (L.v.bits == 3) return launch_prefill_fast_v30(L, k, v, seq_len, st);
    if (L.v.bits == 4) return launch_prefill_fast_v40(L, k, v, seq_len, st);
    if (L.v.mode == KVQ_SYM_PER_TOKEN) return launch_prefill_fast_v81(L, k, v, seq_len, st);
    return launch_prefill_fast_v80(L, k, v, seq_len, st);
  }
  switch (L.v.bits) {
    case 3: return launch_prefill_v3(L, k, v, seq_len, st);
    case 4: return launch_prefill_v4(L, k, v, seq_len, st);
    default: return launch_prefill_v8(L, k, v, seq_len, st);
  }
}

}  // namespace kvq
