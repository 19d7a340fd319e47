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
// The nearest level is found by a search, not a scan: with distinct levels
// v_0 < ... < v_{n-1} at least max|v| / 65536 apart, the level nearest to y
// after fp32 rounding of |y - v_i| is always v_k or v_{k+1} for v_k <= y <=
// v_{k+1} (a level further out is further away by more than one fp32 ulp of
// any reachable distance, |y| <= 1.5 max|v|), and the choice between the two
// switches once, at a threshold the host finds exactly by bisection over the
// fp32 values in [v_k, v_{k+1}] with the same rounding and tie rule. So the
// code is cb_code[#{k : cb_thr[k] <= y}], four compares per value.
//
// One warp per (stream, row, tensor); lane l holds channels 4l .. 4l + 3.
#include <cstdint>
#include <algorithm>
#include <cstring>

#include "codebook.cuh"
#include "common.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kRowsPerCta = 8;

// Codes and scale of row i of stream n into cache row row0 + i.
__device__ __forceinline__ void code_row(const TensorDev& T, int n, int r, uint2 raw, int lane, float cbmax,
                                         float rcb, const float* thr, const uint32_t* code) {
  const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  const float x[4] = {x01.x, x01.y, x23.x, x23.y};
  // group absmax over the group's lanes (G / 4 of them, G in 16 .. 128)
  float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  const int lpg = T.group / 4;
  for (int off = 1; off < lpg; off <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
  const __half s16 = __float2half_rn(cb::quotient(am, cbmax, rcb));
  const float s = __half2float(s16);

  uint32_t nib = 0;
  if (s > 0.0f) {
    // an infinite scale (absmax / max|level| beyond fp16) makes every y zero
    const float rs = __frcp_rn(s);
    const bool finite = rs != 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float y = finite ? cb::quotient(x[c], s, rs) : 0.0f;
      int p = y >= thr[7] ? 8 : 0;
      p += y >= thr[p + 3] ? 4 : 0;
      p += y >= thr[p + 1] ? 2 : 0;
      p += y >= thr[p] ? 1 : 0;
      nib |= code[p] << (4 * c);
    }
  }
  // word w of the row holds channels 8w .. 8w + 7: lanes 2w (low half) and 2w + 1
  const uint32_t other = __shfl_xor_sync(0xffffffffu, nib, 1);
  if ((lane & 1) == 0)
    T.codes[(int64_t)n * T.codes_sstride + (int64_t)r * T.words + (lane >> 1)] = nib | (other << 16);
  if ((lane & (lpg - 1)) == 0) {
    __half* meta = reinterpret_cast<__half*>(T.meta + (int64_t)n * T.meta_sstride);
    meta[(int64_t)r * (kHeadDim / T.group) + (4 * lane) / T.group] = s16;
  }
}

// Grid (x, stream, tensor); the warps of all x-blocks stride over the rows,
// two rows in flight per warp.
__global__ void __launch_bounds__(32 * kRowsPerCta)
    codebook_rows_kernel(LayerDev L, const __half* __restrict__ k, const __half* __restrict__ v, int rows,
                         int in_rows, const VarPos vp, int row0_all) {
  __shared__ float thr[16];
  __shared__ uint32_t code[16];
  if (threadIdx.x < 16) {
    thr[threadIdx.x] = L.cb_thr[threadIdx.x];
    code[threadIdx.x] = L.cb_code[threadIdx.x];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = blockIdx.y;
  const bool is_k = blockIdx.z == 0;
  const int row0 = vp.on ? vp.pos[n / vp.hkv] : row0_all;  // per batch row with variable lengths
  const TensorDev& T = is_k ? L.k : L.v;
  const __half* src = (is_k ? k : v) + (int64_t)n * in_rows * kHeadDim + 4 * lane;
  float cbmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) cbmax = fmaxf(cbmax, fabsf(__half2float(__ushort_as_half(L.codebook[j]))));
  const float rcb = __frcp_rn(cbmax);
  const int stride = gridDim.x * kRowsPerCta;
  int i = blockIdx.x * kRowsPerCta + warp;
  for (; i + stride < rows; i += 2 * stride) {
    const uint2 r0 = __ldcs(reinterpret_cast<const uint2*>(src + (int64_t)i * kHeadDim));
    const uint2 r1 = __ldcs(reinterpret_cast<const uint2*>(src + (int64_t)(i + stride) * kHeadDim));
    code_row(T, n, row0 + i, r0, lane, cbmax, rcb, thr, code);
    code_row(T, n, row0 + i + stride, r1, lane, cbmax, rcb, thr, code);
  }
  if (i < rows)
    code_row(T, n, row0 + i, __ldcs(reinterpret_cast<const uint2*>(src + (int64_t)i * kHeadDim)), lane, cbmax,
             rcb, thr, code);
}

}  // namespace

void codebook_search_table(const uint16_t levels[16], float thr[16], uint8_t code[16]) {
  struct Level {
    float v;
    int idx;
  };
  Level lv[16];
  for (int i = 0; i < 16; ++i) {
    __half_raw hr;
    hr.x = levels[i];
    lv[i] = {__half2float(__half(hr)), i};
  }
  std::sort(lv, lv + 16, [](const Level& a, const Level& b) { return a.v < b.v || (a.v == b.v && a.idx < b.idx); });
  int n = 0;  // distinct levels, each with the lowest index among its equals (-0 == +0)
  for (int i = 0; i < 16; ++i)
    if (n == 0 || lv[i].v != lv[n - 1].v) lv[n++] = lv[i];
  // fp32 values in order as integers (-0 and +0 both 0)
  auto ord = [](float f) -> int64_t {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (u >> 31) ? -(int64_t)(u & 0x7FFFFFFFu) : (int64_t)u;
  };
  auto from_ord = [](int64_t o) -> float {
    const uint32_t u = o >= 0 ? (uint32_t)o : (0x80000000u | (uint32_t)(-o));
    float f;
    std::memcpy(&f, &u, 4);
    return f;
  };
  for (int k = 0; k < 16; ++k) {
    thr[k] = INFINITY;
    code[k] = (uint8_t)lv[k < n ? k : n - 1].idx;
  }
  for (int k = 0; k + 1 < n; ++k) {
    const float a = lv[k].v, b = lv[k + 1].v;
    const int ia = lv[k].idx, ib = lv[k + 1].idx;
    // level k + 1 is chosen at y in [a, b] when its fp32 distance is smaller,
    // or equal with the lower index
    auto upper_wins = [&](float y) {
      const float da = y - a, db = b - y;
      return db < da || (db == da && ib < ia);
    };
    int64_t lo = ord(a), hi = ord(b);  // upper_wins(a) is false, upper_wins(b) true
    while (hi - lo > 1) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (upper_wins(from_ord(mid)))
        hi = mid;
      else
        lo = mid;
    }
    thr[k] = from_ord(hi);
  }
}

cudaError_t launch_codebook_rows(const LayerDev& L, const __half* k, const __half* v, int rows, int in_rows,
                                 const VarPos& vp, int row0, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  // about 1216 CTAs of 8 warps in all (eight per SM), more when few streams
  int gx = (rows + kRowsPerCta - 1) / kRowsPerCta;
  const int cap = 1216 / (2 * L.n_streams) > 1 ? 1216 / (2 * L.n_streams) : 1;
  if (gx > cap) gx = cap;
  const dim3 grid(gx, L.n_streams, 2);
  codebook_rows_kernel<<<grid, 32 * kRowsPerCta, 0, stream>>>(L, k, v, rows, in_rows, vp, row0);
  return cudaGetLastError();
}

}  // namespace kvq
