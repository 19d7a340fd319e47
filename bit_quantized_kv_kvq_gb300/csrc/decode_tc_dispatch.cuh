// Launch of the tensor-core decode kernels (decode_tc.cuh) for one pair of
// key / value code widths, chosen by the including translation unit through
// KVQ_TC_KB and KVQ_TC_VB.
#pragma once
#include "decode_tc.cuh"

namespace kvq {

#define KVQ_TC_NAME3(a, b, c) a##b##c
#define KVQ_TC_NAME(b, c) KVQ_TC_NAME3(launch_decode_tc_k, b, c)

cudaError_t KVQ_TC_NAME(KVQ_TC_KB, KVQ_TC_VB)(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  constexpr int KB = KVQ_TC_KB, VB = KVQ_TC_VB;
  const bool outl = L.outliers > 0;
  const bool nt2 = a.gqa > 4;
  if (VB == 3 || L.v.group == 128) {
    if (nt2) return outl ? tc::launch_t<KB, VB, 128, 2, true>(L, a, st) : tc::launch_t<KB, VB, 128, 2, false>(L, a, st);
    return outl ? tc::launch_t<KB, VB, 128, 1, true>(L, a, st) : tc::launch_t<KB, VB, 128, 1, false>(L, a, st);
  }
  if constexpr (VB != 3) {
    if (nt2) return outl ? tc::launch_t<KB, VB, 64, 2, true>(L, a, st) : tc::launch_t<KB, VB, 64, 2, false>(L, a, st);
    return outl ? tc::launch_t<KB, VB, 64, 1, true>(L, a, st) : tc::launch_t<KB, VB, 64, 1, false>(L, a, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace kvq
