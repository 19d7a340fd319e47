// GQA decode-kernel instantiations (2, 4 or 8 query heads per kv-head).
#include "decode_gqa.cuh"

namespace kvq {

bool decode_gqa_supported(const LayerDev& L, int gqa) {
  if (gqa != 2 && gqa != 4 && gqa != 8) return false;
  const TensorDev& k = L.k;
  const TensorDev& v = L.v;
  if (L.outliers > 0) return false;
  if (k.mode == KVQ_CODEBOOK_PER_TOKEN || v.mode == KVQ_CODEBOOK_PER_TOKEN)  // 4-bit, groups of 32 .. 128
    return k.mode == v.mode && k.group >= 32 && v.group >= 32;
  if ((k.bits == 3) != (v.bits == 3)) return false;  // 3-bit keys and values go together
  if (v.mode == KVQ_ASYM_PER_CHANNEL || v.group < 32) return false;
  if (k.mode != KVQ_ASYM_PER_CHANNEL && k.group < 32) return false;
  if ((k.mode == KVQ_SYM_PER_TOKEN) != (v.mode == KVQ_SYM_PER_TOKEN)) return false;
  return true;
}

cudaError_t launch_decode_gqa(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  const int kb = L.k.bits, vb = L.v.bits, km = L.k.mode;
  const bool g32 = L.k.group == 32 && L.v.group == 32;  // the q8_0 layout: constant groups of 32
  if (km == KVQ_SYM_PER_TOKEN)
    return g32 ? gqa::launch_t<8, KVQ_SYM_PER_TOKEN, 8, KVQ_SYM_PER_TOKEN, 32>(L, a, st)
               : gqa::launch_t<8, KVQ_SYM_PER_TOKEN, 8, KVQ_SYM_PER_TOKEN>(L, a, st);
  if (km == KVQ_CODEBOOK_PER_TOKEN)
    return g32 ? gqa::launch_t<4, KVQ_CODEBOOK_PER_TOKEN, 4, KVQ_CODEBOOK_PER_TOKEN, 32>(L, a, st)
               : gqa::launch_t<4, KVQ_CODEBOOK_PER_TOKEN, 4, KVQ_CODEBOOK_PER_TOKEN>(L, a, st);
#define KVQ_GQA(KB_, KM_)                                                          \
  if (kb == KB_ && km == KM_) {                                                    \
    if (vb == 4) return gqa::launch_t<KB_, KM_, 4, KVQ_ASYM_PER_TOKEN>(L, a, st);  \
    return gqa::launch_t<KB_, KM_, 8, KVQ_ASYM_PER_TOKEN>(L, a, st);               \
  }
  if (kb == 3 && vb == 3) {
    if (km == KVQ_ASYM_PER_CHANNEL) return gqa::launch_t<3, KVQ_ASYM_PER_CHANNEL, 3, KVQ_ASYM_PER_TOKEN>(L, a, st);
    return gqa::launch_t<3, KVQ_ASYM_PER_TOKEN, 3, KVQ_ASYM_PER_TOKEN>(L, a, st);
  }
  KVQ_GQA(4, KVQ_ASYM_PER_CHANNEL)
  KVQ_GQA(8, KVQ_ASYM_PER_CHANNEL)
  KVQ_GQA(4, KVQ_ASYM_PER_TOKEN)
  KVQ_GQA(8, KVQ_ASYM_PER_TOKEN)
#undef KVQ_GQA
  return cudaErrorNotSupported;
}

}  // namespace kvq
