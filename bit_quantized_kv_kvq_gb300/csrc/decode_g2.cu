// Decode-kernel instantiations for 2 query head(s) per kv-head.
#include "decode_impl.cuh"

namespace kvq {
cudaError_t launch_decode_g2(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  return launch_decode_g<2>(L, a, st);
}
}  // namespace kvq
