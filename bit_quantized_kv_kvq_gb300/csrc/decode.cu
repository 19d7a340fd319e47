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

cudaError_t launch_decode_tc_k33(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_tc_k44(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_tc_k48(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_tc_k84(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_tc_k88(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);

// Per-channel keys and asymmetric per-token values with 3/3, 4/4, 4/8, 8/4
// or 8/8 bits (value groups of 64 or 128 channels; 128 at 3 bits): the
// tensor-core kernels of decode_tc.cuh, for every query-group size.
static bool decode_tc_supported(const LayerDev& L, int gqa) {
  if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8) return false;
  if (L.k.mode != KVQ_ASYM_PER_CHANNEL || L.v.mode != KVQ_ASYM_PER_TOKEN) return false;
  const int kb = L.k.bits, vb = L.v.bits;
  if ((kb == 3) != (vb == 3)) return false;
  if (vb == 3) return L.v.group == 128;
  return L.v.group == 64 || L.v.group == 128;
}

static cudaError_t launch_decode_tc(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  switch (L.k.bits * 10 + L.v.bits) {
    case 33: return launch_decode_tc_k33(L, a, st);
    case 44: return launch_decode_tc_k44(L, a, st);
    case 48: return launch_decode_tc_k48(L, a, st);
    case 84: return launch_decode_tc_k84(L, a, st);
    default: return launch_decode_tc_k88(L, a, st);
  }
}

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
  if (decode_tc_supported(L, a.gqa)) {
    e = launch_decode_tc(L, a, st);
    combine = a.splits > 1;  // one split writes the output itself
  } else if (a.gqa == 1 && decode_mha_supported(L)) {
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
