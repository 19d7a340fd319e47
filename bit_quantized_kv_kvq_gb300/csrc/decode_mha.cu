// MHA decode-kernel instantiations (one query head per kv-head).
#include "decode_mha.cuh"

namespace kvq {

bool decode_mha_supported(const LayerDev& L) {
  const TensorDev& k = L.k;
  const TensorDev& v = L.v;
  if (k.mode == KVQ_CODEBOOK_PER_TOKEN || v.mode == KVQ_CODEBOOK_PER_TOKEN) return false;
  if (k.bits == 3 || v.bits == 3) return false;
  // outliers: 4-bit asymmetric codes only (other pairs use the generic kernel)
  if (L.outliers > 0 && (k.bits != 4 || v.bits != 4 || k.mode == KVQ_SYM_PER_TOKEN)) return false;
  if (v.mode == KVQ_ASYM_PER_CHANNEL || v.group < 32) return false;
  if (k.mode != KVQ_ASYM_PER_CHANNEL && k.group < 32) return false;
  if ((k.mode == KVQ_SYM_PER_TOKEN) != (v.mode == KVQ_SYM_PER_TOKEN)) return false;
  return true;
}

cudaError_t launch_decode_mha(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  const int kb = L.k.bits, vb = L.v.bits, km = L.k.mode;
  if (L.outliers > 0) {
    if (km == KVQ_ASYM_PER_CHANNEL)
      return mha::launch_t<4, KVQ_ASYM_PER_CHANNEL, 4, KVQ_ASYM_PER_TOKEN, true>(L, a, st);
    return mha::launch_t<4, KVQ_ASYM_PER_TOKEN, 4, KVQ_ASYM_PER_TOKEN, true>(L, a, st);
  }
  if (km == KVQ_SYM_PER_TOKEN)
    return mha::launch_t<8, KVQ_SYM_PER_TOKEN, 8, KVQ_SYM_PER_TOKEN, false>(L, a, st);
#define KVQ_MHA(KB_, KM_)                                                                 \
  if (kb == KB_ && km == KM_) {                                                           \
    if (vb == 4) return mha::launch_t<KB_, KM_, 4, KVQ_ASYM_PER_TOKEN, false>(L, a, st);  \
    return mha::launch_t<KB_, KM_, 8, KVQ_ASYM_PER_TOKEN, false>(L, a, st);               \
  }
  KVQ_MHA(4, KVQ_ASYM_PER_CHANNEL)
  KVQ_MHA(8, KVQ_ASYM_PER_CHANNEL)
  KVQ_MHA(4, KVQ_ASYM_PER_TOKEN)
  KVQ_MHA(8, KVQ_ASYM_PER_TOKEN)
#undef KVQ_MHA
  return cudaErrorNotSupported;
}

}  // namespace kvq
