// Split-K combine and decode dispatch.
//
// The combine merges per-split partials (m_i, l_i, o_i), with m in log2
// units, by the log-sum-exp rule: M = max m_i, L = sum l_i 2^(m_i - M),
// o = sum o_i 2^(m_i - M) / L.
#include <cstring>

#include "decode_impl.cuh"
#include "decode_merge.cuh"
#include "decode_pipe.cuh"

namespace kvq {
namespace {

__global__ void __launch_bounds__(kHeadDim)
    combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                   int splits, void* out, int out_dtype, const float* sink_part) {
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
  const float res = finish_row(sink_part, r, c, o, M, lsum);
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

cudaError_t launch_decode_pipe_k33(const LayerDev& L, const pipe::Args& a, cudaStream_t st);
cudaError_t launch_decode_pipe_k44(const LayerDev& L, const pipe::Args& a, cudaStream_t st);
cudaError_t launch_decode_pipe_k48(const LayerDev& L, const pipe::Args& a, cudaStream_t st);
cudaError_t launch_decode_pipe_k84(const LayerDev& L, const pipe::Args& a, cudaStream_t st);
cudaError_t launch_decode_pipe_k88(const LayerDev& L, const pipe::Args& a, cudaStream_t st);

// The stream-K kernel puts the query heads of a kv-head on the mma rows
// (heads x hi/lo): with 8 heads every row and lane is used and P leaves QK^T
// in PV's operand layout. With fewer heads most rows and softmax lanes would
// idle, so 1, 2 and 4 heads per kv-head use the token-row kernels of
// decode_tc.cuh instead.
bool decode_pipe_supported(const LayerDev& L, int gqa) {
  if (gqa != 8) return false;
  if (L.k.mode != KVQ_ASYM_PER_CHANNEL || L.v.mode != KVQ_ASYM_PER_TOKEN) return false;
  if (L.k.group != 64 && L.k.group != 128 && L.k.group != 256) return false;
  switch (L.k.bits * 10 + L.v.bits) {
    case 33: return L.v.group == 128;
    case 44: case 48: case 84: case 88: return L.v.group == 64 || L.v.group == 128;
    default: return false;
  }
}

// Partition of the key blocks of all streams over `ctas` CTAs. Each stream
// of cps blocks is followed by `vex` empty places worth the cost of a stream
// switch (finishing a stream, loading the next query, its first rebuild),
// and the virtual space of streams * (cps + vex) places is cut evenly: CTA c
// takes the blocks in [c V / P, (c + 1) V / P). A stream meets at most
// ceil(P / streams) + 1 CTAs, which bounds the partial rows per stream.
// Measured on 152 SMs: with 32 streams of 257 blocks of 128 tokens, a switch
// weighed as 640 tokens brings the slowest CTAs (those crossing a stream
// boundary) in: 76.3 -> 72.4 us; with 8 streams of 2049 blocks of 64 tokens
// any weight was slower (84.0 -> 86.0 us), so fewer than 16 streams get none.
PipePlan plan_decode_pipe(const LayerDev& L, int len, int gqa, int sm_count, int ctas_override) {
  PipePlan p;
  const int T = L.k.group;
  p.cps = (len + T - 1) / T;
  p.n_chunks = (long long)L.n_streams * p.cps;
  p.vex = L.n_streams >= 16 ? (640 + T - 1) / T : 0;
  p.n_virtual = (long long)L.n_streams * (p.cps + p.vex);
  int P = sm_count > 0 ? sm_count : 1;
  if (ctas_override > 0 && ctas_override < P) P = ctas_override;
  if ((long long)P > p.n_chunks) P = (int)p.n_chunks;
  if (P < 1) P = 1;
  p.ctas = P;
  p.jmax = (P + L.n_streams - 1) / L.n_streams + 1;
  p.ws_bytes = (size_t)L.n_streams * p.jmax * gqa * pipe::kPartRow * 4;
  return p;
}

size_t decode_pipe_workspace_max(const LayerDev& L, int gqa, int sm_count) {
  const int P = sm_count > 0 ? sm_count : 1;
  const int jmax = (P + L.n_streams - 1) / L.n_streams + 1;
  return (size_t)L.n_streams * jmax * gqa * pipe::kPartRow * 4;
}

cudaError_t launch_decode_pipe(const LayerDev& L, const DecodeArgs& d, const PipePlan& p, cudaStream_t st) {
  pipe::Args a;
  std::memset(&a, 0, sizeof a);
  a.q = d.q;
  a.sink_part = d.sink_part;
  a.out = d.out;
  a.part = d.part_o;
  a.counters = L.counters;
  a.out_dtype = d.out_dtype;
  a.num_q_heads = d.num_q_heads;
  a.H = d.gqa;
  a.scale_log2 = d.scale_log2;
  a.length = d.length;
  a.kq = d.k_quant_len;
  a.T = L.k.group;
  a.cps = p.cps;
  a.n_chunks = p.n_chunks;
  a.vex = p.vex;
  a.n_virtual = p.n_virtual;
  a.P = p.ctas;
  a.jmax = p.jmax;
  a.kout = L.outliers;
  cudaError_t e;
  switch (L.k.bits * 10 + L.v.bits) {
    case 33: e = launch_decode_pipe_k33(L, a, st); break;
    case 44: e = launch_decode_pipe_k44(L, a, st); break;
    case 48: e = launch_decode_pipe_k48(L, a, st); break;
    case 84: e = launch_decode_pipe_k84(L, a, st); break;
    default: e = launch_decode_pipe_k88(L, a, st); break;
  }
  if (e == cudaSuccess) count_launches(1);
  return e;
}

bool decode_supported(const LayerDev& L, int gqa) {
  if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8) return false;
  const int km = L.k.mode, vm = L.v.mode;
  if (km == KVQ_CODEBOOK_PER_TOKEN || vm == KVQ_CODEBOOK_PER_TOKEN)
    return km == KVQ_CODEBOOK_PER_TOKEN && vm == KVQ_CODEBOOK_PER_TOKEN;
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
    combine = false;  // one split writes the output itself; the last CTA of a stream merges the splits
  } else if (a.gqa == 1 && !a.varlen && decode_mha_supported(L)) {
    e = launch_decode_mha(L, a, st);
    combine = false;  // as above
  } else if (a.gqa > 1 && decode_gqa_supported(L, a.gqa)) {
    e = launch_decode_gqa(L, a, st);
    combine = false;  // as above
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
  combine_kernel<<<rows, kHeadDim, 0, st>>>(a.part_o, a.part_ml, a.splits, a.out, a.out_dtype, a.sink_part);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace kvq
