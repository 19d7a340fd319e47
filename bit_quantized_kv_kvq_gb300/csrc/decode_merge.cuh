// Split-K merge fused into the end of a split decode kernel (grid: splits x
// streams), instead of a second launch that combines the partials.
#pragma once

#include "common.cuh"
#include "kvq_internal.h"

namespace kvq {

// The output value of channel c of (batch, query head) row `row` from the
// decode's unnormalised sum o = sum_t 2^(s_t - M) v_t, its maximum M (log2
// units) and its weight sum lsum, merged by the log-sum-exp rule with the
// row's attention over the fp16 sink tokens when there is one (sink_part:
// [rows][kSinkPartRow] = o_s[128], m_s, l_s; NULL when the layer has none).
__device__ __forceinline__ float finish_row(const float* sink_part, int64_t row, int c, float o, float M,
                                            float lsum) {
  if (!sink_part) return o / lsum;
  const float* sp = sink_part + row * kSinkPartRow;
  const float ms = __ldcg(sp + kHeadDim), ls = __ldcg(sp + kHeadDim + 1);
  const float Mx = fmaxf(M, ms);
  const float wa = M == -INFINITY ? 0.0f : exp2f(M - Mx);
  const float wb = ms == -INFINITY ? 0.0f : exp2f(ms - Mx);
  return fmaf(o, wa, __ldcg(sp + c) * wb) / fmaf(lsum, wa, ls * wb);
}

__device__ __forceinline__ float4 finish_row4(const float* sink_part, int64_t row, int c0, float4 o, float M,
                                              float lsum) {
  return make_float4(finish_row(sink_part, row, c0, o.x, M, lsum), finish_row(sink_part, row, c0 + 1, o.y, M, lsum),
                     finish_row(sink_part, row, c0 + 2, o.z, M, lsum), finish_row(sink_part, row, c0 + 3, o.w, M, lsum));
}

// Split-K merge at the end of the kernel. Every CTA of a stream, once its
// partials are written and fenced, adds one to the stream's arrival counter;
// the CTA that arrives last merges the partials of the stream's G query rows
// (row0 .. row0 + G - 1) by the log-sum-exp rule, M = max m_i,
// L = sum l_i 2^(m_i - M), o = sum o_i 2^(m_i - M) / L, writes the output
// and clears the counter for the next call. Warp w merges rows w, w + WARPS,
// ...; a lane owns four channels and keeps 16 partials' loads in flight,
// with a running maximum so the partials are read in a single pass.
template <int WARPS>
__device__ __forceinline__ void merge_splits_if_last(uint32_t* counter, const DecodeArgs& a,
                                                     int64_t row0, int G) {
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(counter, 1u) == (uint32_t)(a.splits - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = a.splits;
  constexpr int kBatch = 16;
  for (int h = warp; h < G; h += WARPS) {
    const int64_t prow = row0 + h;
    const float* pm = a.part_ml + prow * S * 2;
    const float* po = a.part_o + prow * S * kHeadDim + 4 * lane;
    // one pass with a running maximum: every lane walks the same partials,
    // so M, the rescale factors and lsum are the same in every lane
    float M = -INFINITY, lsum = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int i0 = 0; i0 < S; i0 += kBatch) {
      float4 v[kBatch];
      float2 ml[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (i0 + j < S) {
          v[j] = __ldcg(reinterpret_cast<const float4*>(po + (int64_t)(i0 + j) * kHeadDim));
          ml[j] = __ldcg(reinterpret_cast<const float2*>(pm + 2 * (i0 + j)));
        } else {
          v[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          ml[j] = make_float2(-INFINITY, 0.0f);
        }
      }
      float Mb = M;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) Mb = fmaxf(Mb, ml[j].x);
      if (Mb > M) {  // the same in every lane
        const float f = M == -INFINITY ? 0.0f : exp2f(M - Mb);
        lsum *= f;
        acc.x *= f;
        acc.y *= f;
        acc.z *= f;
        acc.w *= f;
        M = Mb;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float w = ml[j].x == -INFINITY ? 0.0f : exp2f(ml[j].x - M);
        lsum = fmaf(w, ml[j].y, lsum);
        acc.x = fmaf(w, v[j].x, acc.x);
        acc.y = fmaf(w, v[j].y, acc.y);
        acc.z = fmaf(w, v[j].z, acc.z);
        acc.w = fmaf(w, v[j].w, acc.w);
      }
    }
    const int64_t o = prow * kHeadDim + 4 * lane;
    const float4 r = finish_row4(a.sink_part, prow, 4 * lane, acc, M, lsum);
    if (a.out_dtype == KVQ_F32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + o) = r;
    } else {
      const __half2 h01 = __floats2half2_rn(r.x, r.y);
      const __half2 h23 = __floats2half2_rn(r.z, r.w);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&h01);
      u.y = *reinterpret_cast<const uint32_t*>(&h23);
      *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.out) + o) = u;
    }
  }
  if (threadIdx.x == 0) atomicExch(counter, 0u);
}

}  // namespace kvq
