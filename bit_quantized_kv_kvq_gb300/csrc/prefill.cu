// Prefill dispatch: per-token keys and per-channel key blocks of 64 or 128
// tokens run the barrier-light kernel of prefill_fast.cuh; 256-token key
// blocks the kernel of prefill_impl.cuh.
#include "prefill_impl.cuh"

namespace kvq {

cudaError_t launch_prefill_fast_v300(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);
cudaError_t launch_prefill_fast_v301(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);
cudaError_t launch_prefill_fast_v400(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);
cudaError_t launch_prefill_fast_v401(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);
cudaError_t launch_prefill_fast_v800(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);
cudaError_t launch_prefill_fast_v801(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);
cudaError_t launch_prefill_fast_v810(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);
cudaError_t launch_prefill_fast_v811(const LayerDev& L, const __half* k, const __half* v,
                                     int seq_len, cudaStream_t st);

static bool fast_prefill_supported(const LayerDev& L) {
  if (L.k.mode == KVQ_ASYM_PER_CHANNEL && L.k.group != 64 && L.k.group != 128) return false;
  return true;
}

cudaError_t launch_prefill(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                           cudaStream_t st) {
  if (seq_len <= 0) return cudaSuccess;
  if (L.k.mode == KVQ_CODEBOOK_PER_TOKEN) {
    VarPos none;
    none.on = 0;
    none.hkv = 1;
    return launch_codebook_rows(L, k, v, seq_len, L.in_rows > 0 ? L.in_rows : seq_len, none, 0, st);
  }
  if (fast_prefill_supported(L)) {
    const bool o = L.outliers > 0;
    if (L.v.bits == 3)
      return (o ? launch_prefill_fast_v301 : launch_prefill_fast_v300)(L, k, v, seq_len, st);
    if (L.v.bits == 4)
      return (o ? launch_prefill_fast_v401 : launch_prefill_fast_v400)(L, k, v, seq_len, st);
    if (L.v.mode == KVQ_SYM_PER_TOKEN)
      return (o ? launch_prefill_fast_v811 : launch_prefill_fast_v810)(L, k, v, seq_len, st);
    return (o ? launch_prefill_fast_v801 : launch_prefill_fast_v800)(L, k, v, seq_len, st);
  }
  switch (L.v.bits) {
    case 3: return launch_prefill_v3(L, k, v, seq_len, st);
    case 4: return launch_prefill_v4(L, k, v, seq_len, st);
    default: return launch_prefill_v8(L, k, v, seq_len, st);
  }
}

}  // namespace kvq
