// Split-K combine and decode dispatch.
//
// The combine merges per-split partials (m_i, l_i, o_i), with m in log2
// units, by the log-sum-exp rule: M = max m_i, L = sum l_i 2^(m_i - M),
// o = sum o_i 2^(m_i - M) / L.
#include "decode_impl.cuh"

namespace kvq {
namespace {

__global__ void __launch_bounds__(kHeadDim)
    combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                   int splits, void* out, int out_dtype) {
  const int64_t r = blockIdx.x;
  const int c = threadIdx.x;
  const float* ml = part_ml + r * splits * 2;
  float M = -INFINITY;
  for (int i = 0; i < splits; ++i) M = fmaxf(M, ml[2 * i]);
  float lsum = 0.0f, o = 0.0f;
  for (int i = 0; i < splits; ++i) {
    const float w = exp2f(ml[2 * i] - M);
    lsum += w * ml[2 * i + 1];
    o += w * part_o[(r * splits + i) * kHeadDim + c];
  }
  const float res = o / lsum;
  if (out_dtype == KVQ_F32)
    reinterpret_cast<float*>(out)[r * kHeadDim + c] = res;
  else
    reinterpret_cast<__half*>(out)[r * kHeadDim + c] = __float2half_rn(res);
}

}  // namespace

bool decode_supported(const LayerDev& L, int gqa) {
  if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8) return false;
  const int km = L.k.mode, vm = L.v.mode;
  if (km == KVQ_SYM_PER_TOKEN || vm == KVQ_SYM_PER_TOKEN)
    return km == KVQ_SYM_PER_TOKEN && vm == KVQ_SYM_PER_TOKEN;
  return vm == KVQ_ASYM_PER_TOKEN;
}

cudaError_t launch_decode(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e;
  const int rows = (L.n_streams / L.num_kv_heads) * a.num_q_heads;
  bool combine = true;
  if (a.gqa == 1 && decode_mha_supported(L)) {
    e = launch_decode_mha(L, a, st);
    combine = a.splits > 1;  // one split writes the output itself
  } else if (a.gqa > 1 && decode_gqa_supported(L, a.gqa)) {
    e = launch_decode_gqa(L, a, st);
    combine = a.splits > 1;
  } else {
    switch (a.gqa) {
      case 1: e = launch_decode_g1(L, a, st); break;
      case 2: e = launch_decode_g2(L, a, st); break;
      case 4: e = launch_decode_g4(L, a, st); break;
      case 8: e = launch_decode_g8(L, a, st); break;
      default: return cudaErrorNotSupported;
    }
  }
  if (e != cudaSuccess || a.occupancy_out) return e;
  count_launches(1);
  if (!combine) return cudaSuccess;
  combine_kernel<<<rows, kHeadDim, 0, st>>>(a.part_o, a.part_ml, a.splits, a.out, a.out_dtype);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace kvq
