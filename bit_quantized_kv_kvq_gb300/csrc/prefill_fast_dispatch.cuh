// Dispatch of the prefill kernels of prefill_fast.cuh for one value codec,
// chosen by the including translation unit through KVQ_PF_VB and
// KVQ_PF_VSYM, with (KVQ_PF_OUTL 1) or without (0) the outlier split.
#pragma once
#include "prefill_fast.cuh"

namespace kvq {

#ifndef KVQ_PF_VB
#error "KVQ_PF_VB (4 or 8) and KVQ_PF_VSYM (0 or 1) select the value codec of this unit"
#endif

#ifndef KVQ_PF_OUTL
#define KVQ_PF_OUTL 0
#endif

#define KVQ_PF_NAME4(a, b, c, d) a##b##c##d
#define KVQ_PF_NAME(b, c, d) KVQ_PF_NAME4(launch_prefill_fast_v, b, c, d)

// launch_prefill_fast_v<bits><sym><outl>
cudaError_t KVQ_PF_NAME(KVQ_PF_VB, KVQ_PF_VSYM, KVQ_PF_OUTL)(const LayerDev& L, const __half* k,
                                                              const __half* v, int seq_len,
                                                              cudaStream_t st) {
  constexpr int VB = KVQ_PF_VB;
  constexpr bool VS = KVQ_PF_VSYM != 0;
  constexpr bool OU = KVQ_PF_OUTL != 0;
  const TensorDev& K = L.k;
#define KVQ_PF_KB(B)                                                                               \
  if (K.bits == B) {                                                                               \
    if (K.mode == KVQ_ASYM_PER_CHANNEL) {                                                          \
      if (K.group == 64) return pfx::launch_fast_t<B, KVQ_ASYM_PER_CHANNEL, 64, VB, VS, OU>(L, k, v, seq_len, st); \
      return pfx::launch_fast_t<B, KVQ_ASYM_PER_CHANNEL, 128, VB, VS, OU>(L, k, v, seq_len, st);     \
    }                                                                                              \
    return pfx::launch_fast_t<B, KVQ_ASYM_PER_TOKEN, 1, VB, VS, OU>(L, k, v, seq_len, st);           \
  }
  if (K.mode == KVQ_SYM_PER_TOKEN) return pfx::launch_fast_t<8, KVQ_SYM_PER_TOKEN, 1, VB, VS, OU>(L, k, v, seq_len, st);
  KVQ_PF_KB(3)
  KVQ_PF_KB(4)
  KVQ_PF_KB(8)
#undef KVQ_PF_KB
  return cudaErrorNotSupported;
}

}  // namespace kvq
