// Launch of the tensor-core decode kernels (decode_tc.cuh) for one pair of
// key / value code widths, chosen by the including translation unit through
// KVQ_TC_KB and KVQ_TC_VB.
#pragma once
#include "decode_tc.cuh"

namespace kvq {

#define KVQ_TC_NAME3(a, b, c) a##b##c
#define KVQ_TC_NAME(b, c) KVQ_TC_NAME3(launch_decode_tc_k, b, c)

namespace tc {
// One value-group width: the head-tile count, outliers, and (without
// outliers) the query heads per kv-head as a constant where every head slot
// is used or there is one.
template <int KB, int VB, int VG>
cudaError_t launch_vg(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  const bool outl = L.outliers > 0;
  const int g = a.gqa;
  if (g > 4) {
    if (outl) return launch_t<KB, VB, VG, 2, true>(L, a, st);
    return g == 8 ? launch_t<KB, VB, VG, 2, false, 8>(L, a, st) : launch_t<KB, VB, VG, 2, false>(L, a, st);
  }
  if (outl) return launch_t<KB, VB, VG, 1, true>(L, a, st);
  return g == 4 ? launch_t<KB, VB, VG, 1, false, 4>(L, a, st)
         : g == 1 ? launch_t<KB, VB, VG, 1, false, 1>(L, a, st) : launch_t<KB, VB, VG, 1, false>(L, a, st);
}
}  // namespace tc

cudaError_t KVQ_TC_NAME(KVQ_TC_KB, KVQ_TC_VB)(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  constexpr int KB = KVQ_TC_KB, VB = KVQ_TC_VB;
  if (VB == 3 || L.v.group == 128) return tc::launch_vg<KB, VB, 128>(L, a, st);
  if constexpr (VB != 3) return tc::launch_vg<KB, VB, 64>(L, a, st);
  return cudaErrorNotSupported;
}

}  // namespace kvq
