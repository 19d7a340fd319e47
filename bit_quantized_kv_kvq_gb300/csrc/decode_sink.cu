// Attention over the attention-sink tokens: the first tokens of every stream
// kept in fp16 for keys and values (KVQuant page, cf-1.com/news/2306543,
// §4.1: the first 5-10 tokens draw a large share of the attention, so they
// are kept at full precision). One CTA per (batch, kv-head) stream; warp w
// takes the stream's query heads w, w + 4, ...; a lane owns four channels.
// The scores are in log2 units, e_t = scale_log2 * <q, k_t>; the result is
// the unnormalised o = sum_t 2^(e_t - m) v_t with m = max_t e_t and
// l = sum_t 2^(e_t - m), which the decode kernels merge into their output
// (or, when no token is quantized yet, the normalised output itself).
#include <cstdint>

#include "common.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kSinkWarps = 4;

__global__ void __launch_bounds__(32 * kSinkWarps)
    sink_attention_kernel(LayerDev L, const __half* __restrict__ q, int num_q_heads, float scale_log2,
                          int sink_len, float* __restrict__ part, void* final_out, int out_dtype) {
  const int n = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = L.num_kv_heads;
  const int G = num_q_heads / Hkv;
  const int b = n / Hkv, kvh = n - b * Hkv;
  const __half* ks = L.sink_k + (int64_t)n * L.sink_tokens * kHeadDim;
  const __half* vs = L.sink_v + (int64_t)n * L.sink_tokens * kHeadDim;
  __shared__ float e[kSinkWarps][kMaxSinkTokens];
  for (int h = warp; h < G; h += kSinkWarps) {
    const int64_t row = (int64_t)b * num_q_heads + kvh * G + h;
    const uint2 qr = *reinterpret_cast<const uint2*>(q + row * kHeadDim + 4 * lane);
    const float2 q01 = __half22float2(*reinterpret_cast<const __half2*>(&qr.x));
    const float2 q23 = __half22float2(*reinterpret_cast<const __half2*>(&qr.y));
    float m = -INFINITY;
    for (int t = 0; t < sink_len; ++t) {
      const uint2 kr = *reinterpret_cast<const uint2*>(ks + (int64_t)t * kHeadDim + 4 * lane);
      const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kr.x));
      const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kr.y));
      float d = fmaf(q01.x, k01.x, fmaf(q01.y, k01.y, fmaf(q23.x, k23.x, q23.y * k23.y)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      const float et = d * scale_log2;
      if (lane == 0) e[warp][t] = et;
      m = fmaxf(m, et);
    }
    __syncwarp();
    float l = 0.0f;
    float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int t = 0; t < sink_len; ++t) {
      const float w = exp2f(e[warp][t] - m);
      const uint2 vr = *reinterpret_cast<const uint2*>(vs + (int64_t)t * kHeadDim + 4 * lane);
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vr.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vr.y));
      l += w;
      o.x = fmaf(w, v01.x, o.x);
      o.y = fmaf(w, v01.y, o.y);
      o.z = fmaf(w, v23.x, o.z);
      o.w = fmaf(w, v23.y, o.w);
    }
    __syncwarp();
    if (final_out) {
      const float il = 1.0f / l;
      if (out_dtype == KVQ_F32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(final_out) + row * kHeadDim + 4 * lane) =
            make_float4(o.x * il, o.y * il, o.z * il, o.w * il);
      } else {
        const __half2 h01 = __floats2half2_rn(o.x * il, o.y * il), h23 = __floats2half2_rn(o.z * il, o.w * il);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&h01);
        u.y = *reinterpret_cast<const uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(final_out) + row * kHeadDim + 4 * lane) = u;
      }
    } else {
      float* pr = part + row * kSinkPartRow;
      *reinterpret_cast<float4*>(pr + 4 * lane) = o;
      if (lane == 0) {
        pr[kHeadDim] = m;
        pr[kHeadDim + 1] = l;
      }
    }
  }
}

}  // namespace

cudaError_t launch_sink_attention(const LayerDev& L, const __half* q, int num_q_heads, float scale_log2,
                                  int sink_len, float* part, void* final_out, int out_dtype,
                                  cudaStream_t stream) {
  if (sink_len <= 0 || sink_len > L.sink_tokens || sink_len > kMaxSinkTokens) return cudaErrorInvalidValue;
  sink_attention_kernel<<<L.n_streams, 32 * kSinkWarps, 0, stream>>>(L, q, num_q_heads, scale_log2, sink_len,
                                                                       part, final_out, out_dtype);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace kvq
