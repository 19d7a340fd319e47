// Codebook (non-uniform) quantization of keys and values, per token over
// groups of channels (KVQuant page, cf-1.com/news/2306543, §2.2 item 2:
// levels placed where the values are dense; TurboQuant 3-bit KV-cache page,
// dpshk.com/news/6341316, §3.3: the 4-bit minifloat `1 sign | 2 exponent |
// 1 mantissa` is one such codebook). One fp16 scale per group,
// s = absmax / max_i |cb_i|; each value x takes the index of the level
// nearest to x / s16 (computed in fp32, the lowest index on ties); a group
// whose scale is 0 stores code 0. Codes are 4 bits, eight per word, code j
// of a row at bit 4 (j mod 8) of word j / 8.
//
// One warp per (stream, row, tensor); lane l holds channels 4l .. 4l + 3.
#include <cstdint>

#include "common.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kRowsPerCta = 8;

__global__ void __launch_bounds__(32 * kRowsPerCta)
    codebook_rows_kernel(LayerDev L, const __half* __restrict__ k, const __half* __restrict__ v, int rows,
                         int in_rows, int row0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = blockIdx.x * kRowsPerCta + warp;  // input row
  const int n = blockIdx.y;
  const bool is_k = blockIdx.z == 0;
  if (i >= rows) return;
  const TensorDev& T = is_k ? L.k : L.v;
  const __half* src = (is_k ? k : v) + ((int64_t)n * in_rows + i) * kHeadDim + 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2*>(src);
  const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  const float x[4] = {x01.x, x01.y, x23.x, x23.y};

  float cb[16], cbmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    cb[j] = __half2float(__ushort_as_half(L.codebook[j]));
    cbmax = fmaxf(cbmax, fabsf(cb[j]));
  }
  // group absmax over the group's lanes (G / 4 of them, G in 16 .. 128)
  float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  const int lpg = T.group / 4;
  for (int off = 1; off < lpg; off <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
  const __half s16 = __float2half_rn(__fdiv_rn(am, cbmax));
  const float s = __half2float(s16);

  uint32_t nib = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    int best = 0;
    if (s > 0.0f) {
      const float y = __fdiv_rn(x[c], s);
      float bd = fabsf(y - cb[0]);
#pragma unroll
      for (int j = 1; j < 16; ++j) {
        const float d = fabsf(y - cb[j]);
        if (d < bd) {
          bd = d;
          best = j;
        }
      }
    }
    nib |= (uint32_t)best << (4 * c);
  }
  // word w of the row holds channels 8w .. 8w + 7: lanes 2w (low half) and 2w + 1
  const uint32_t other = __shfl_xor_sync(0xffffffffu, nib, 1);
  const int r = row0 + i;
  if ((lane & 1) == 0)
    T.codes[(int64_t)n * T.codes_sstride + (int64_t)r * T.words + (lane >> 1)] = nib | (other << 16);
  if ((lane & (lpg - 1)) == 0) {
    __half* meta = reinterpret_cast<__half*>(T.meta + (int64_t)n * T.meta_sstride);
    meta[(int64_t)r * (kHeadDim / T.group) + (4 * lane) / T.group] = s16;
  }
}

}  // namespace

cudaError_t launch_codebook_rows(const LayerDev& L, const __half* k, const __half* v, int rows, int in_rows,
                                 int row0, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((rows + kRowsPerCta - 1) / kRowsPerCta, L.n_streams, 2);
  codebook_rows_kernel<<<grid, 32 * kRowsPerCta, 0, stream>>>(L, k, v, rows, in_rows, row0);
  return cudaGetLastError();
}

}  // namespace kvq
