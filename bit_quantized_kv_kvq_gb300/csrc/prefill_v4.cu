// Prefill-kernel instantiations for 4-bit values.
#include "prefill_impl.cuh"

namespace kvq {
cudaError_t launch_prefill_v4(const LayerDev& L, const __half* k, const __half* v, int s,
                              cudaStream_t st) {
  return pf::launch_prefill_v<4, false>(L, k, v, s, st);
}
}  // namespace kvq
