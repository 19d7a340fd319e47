// Prefill-kernel instantiations for 8-bit values.
#include "prefill_impl.cuh"

namespace kvq {
cudaError_t launch_prefill_v8(const LayerDev& L, const __half* k, const __half* v, int s,
                              cudaStream_t st) {
  if (L.v.mode == KVQ_SYM_PER_TOKEN) return pf::launch_prefill_v<8, true>(L, k, v, s, st);
  return pf::launch_prefill_v<8, false>(L, k, v, s, st);
}
}  // namespace kvq
