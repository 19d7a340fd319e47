// Append quantize: one new token per stream (the prefill kernel is in
// prefill_impl.cuh).
//
// Codec (pages cited by short name, address and section):
//  - asymmetric min/max groups, offset = group minimum, codes clamped to
//    [0, 2^b - 1]: TurboQuant 3-bit KV quantization (dpshk.com/news/6341316)
//    §3.1; scale = (max - min) / (2^b - 1), stored as fp16, codes computed
//    from the stored fp16 scale and zero point.
//  - symmetric int8 groups with zero point 0: NIAH q8_0 KV-cache write-up
//    (cf-1.com/news/5482713) §1.2; scale = absmax / 127.
//  - per-channel keys over blocks of T tokens, per-token values in groups of
//    G channels: KVQuant (cf-1.com/news/2306543) §2.2 item 1; W4A8/FA3 page
//    (discosf.com/news/4854722) §2.4 (groups of 64 positions).
//  - dense-and-sparse split: the k largest-|x| entries of each (token, head)
//    row are kept as fp16 CSR outliers, left out of the group statistics and
//    stored with dense code 0: KVQuant §2.2 item 3, §3.3.
//  - append quantizes only the new row: NIAH q8_0 write-up §2.2.
//
// Every floating-point step that decides a code uses explicit round-to-
// nearest intrinsics, so no FMA contraction can change a code.
#include "common.cuh"

namespace kvq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Warp top-k over one 128-channel row (lane l holds channels 4l .. 4l+3).
// Ranking: |x| descending, ties to the lower channel. Returns this lane's
// 4-bit slot mask; sel[0..k) receives the chosen channels in ascending order
// (identical in every lane).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t warp_topk(const float (&x)[4], int k, int lane,
                                              int (&sel)[kMaxOutliers]) {
  uint32_t m = 0;
  for (int it = 0; it < k; ++it) {
    float bm = -1.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!((m >> i) & 1u)) {
        float a = fabsf(x[i]);
        if (a > bm) {
          bm = a;
          bi = lane * 4 + i;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float om = __shfl_xor_sync(kFull, bm, off);
      int oi = __shfl_xor_sync(kFull, bi, off);
      if (om > bm || (om == bm && oi < bi)) {
        bm = om;
        bi = oi;
      }
    }
    if ((bi >> 2) == lane) m |= 1u << (bi & 3);
    sel[it] = bi;
  }
  for (int i = 1; i < k; ++i) {
    int v = sel[i];
    int j = i - 1;
    while (j >= 0 && sel[j] > v) {
      sel[j + 1] = sel[j];
      --j;
    }
    sel[j + 1] = v;
  }
  return m;
}

__device__ __forceinline__ float pick4(const float (&x)[4], int i) {
  return i == 0 ? x[0] : i == 1 ? x[1] : i == 2 ? x[2] : x[3];
}

// Writes the CSR entries of one row (all lanes call; lane 0 stores).
__device__ __forceinline__ void store_outliers(const TensorDev& T, int n, int row, int k,
                                               const float (&x)[4], const int (&sel)[kMaxOutliers],
                                               int lane) {
  int32_t* rp = T.rowptr + (int64_t)n * T.rowptr_sstride;
  int64_t base = (int64_t)n * T.out_sstride + (int64_t)row * k;
  for (int i = 0; i < k; ++i) {
    int c = sel[i];
    float v = __shfl_sync(kFull, pick4(x, c & 3), c >> 2);
    if (lane == 0) {
      T.col[base + i] = (uint16_t)c;
      T.val[base + i] = __float2half_rn(v);  // exact: v came from an fp16
    }
  }
  if (lane == 0) {
    rp[row + 1] = (row + 1) * k;
    if (row == 0) rp[0] = 0;
  }
}

__device__ __forceinline__ void load_row4(const __half* src, int lane, float (&x)[4]) {
  uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
  __half2 a = *reinterpret_cast<__half2*>(&raw.x);
  __half2 b = *reinterpret_cast<__half2*>(&raw.y);
  x[0] = __low2float(a);
  x[1] = __high2float(a);
  x[2] = __low2float(b);
  x[3] = __high2float(b);
}

// ---------------------------------------------------------------------------
// One (token, head) row quantized per token by one warp: outliers, group
// statistics (warp shuffles), fp16 scale/zero, codes, packed stores.
// ---------------------------------------------------------------------------
template <int BITS, bool SYM>
__device__ void quant_row_warp(const __half* __restrict__ src, const TensorDev& T, int n,
                               int row, int kout, int lane, uint8_t* scratch) {
  using P = Pack<BITS>;
  float x[4];
  load_row4(src, lane, x);
  uint32_t om = 0;
  if (kout > 0) {
    int sel[kMaxOutliers];
    om = warp_topk(x, kout, lane, sel);
    store_outliers(T, n, row, kout, x, sel, lane);
  }
  const int lg = T.group >> 2;  // lanes per group
  int code[4];
  __half s16, z16;
  if (SYM) {
    constexpr int qmax = (1 << (BITS - 1)) - 1;
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!((om >> i) & 1u)) am = fmaxf(am, fabsf(x[i]));
    for (int off = 1; off < lg; off <<= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, off));
    s16 = __float2half_rn(__fdiv_rn(am, (float)qmax));
    z16 = __float2half_rn(0.0f);
    const float s = __half2float(s16);
    const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int c = 0;
      if (s > 0.0f && !((om >> i) & 1u)) c = min(max(quant_step(x[i], s, r), -qmax), qmax);
      code[i] = c & (int)P::kMask;
    }
  } else {
    constexpr int levels = (1 << BITS) - 1;
    float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!((om >> i) & 1u)) {
        mn = fminf(mn, x[i]);
        mx = fmaxf(mx, x[i]);
      }
    for (int off = 1; off < lg; off <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(kFull, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    }
    if (mn > mx) {  // every member an outlier
      mn = 0.0f;
      mx = 0.0f;
    }
    mn = __fadd_rn(mn, 0.0f);  // zero extremes are taken as +0
    mx = __fadd_rn(mx, 0.0f);
    s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)levels));
    z16 = __float2half_rn(mn);
    const float s = __half2float(s16);
    const float z = __half2float(z16);
    const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int c = 0;
      if (s > 0.0f && !((om >> i) & 1u))
        c = min(max(quant_step(__fsub_rn(x[i], z), s, r), 0), levels);
      code[i] = c;
    }
  }
  // metadata: one entry per group, written by the group's first lane
  if ((lane & (lg - 1)) == 0) {
    const int g = lane / lg;
    const int per_row = kHeadDim / T.group;
    unsigned char* mb = T.meta + (int64_t)n * T.meta_sstride;
    if (SYM) {
      reinterpret_cast<__half*>(mb)[(int64_t)row * per_row + g] = s16;
    } else {
      reinterpret_cast<__half2*>(mb)[(int64_t)row * per_row + g] = __halves2half2(s16, z16);
    }
  }
  // packed codes
  uint32_t* dst = T.codes + (int64_t)n * T.codes_sstride + (int64_t)row * P::kWords;
  if (BITS == 8) {
    dst[lane] = (uint32_t)code[0] | ((uint32_t)code[1] << 8) | ((uint32_t)code[2] << 16) |
                ((uint32_t)code[3] << 24);
  } else if (BITS == 4) {
    uint32_t nib = (uint32_t)code[0] | ((uint32_t)code[1] << 4) | ((uint32_t)code[2] << 8) |
                   ((uint32_t)code[3] << 12);
    uint32_t hi = __shfl_down_sync(kFull, nib, 1);
    if (!(lane & 1)) dst[lane >> 1] = nib | (hi << 16);
  } else {
    *reinterpret_cast<uint32_t*>(scratch + 4 * lane) =
        (uint32_t)code[0] | ((uint32_t)code[1] << 8) | ((uint32_t)code[2] << 16) |
        ((uint32_t)code[3] << 24);
    __syncwarp();
    if (lane < P::kWords) {
      uint32_t w = 0;
#pragma unroll
      for (int k = 0; k < P::kCpw; ++k) {
        const int c = lane * P::kCpw + k;
        if (c < kHeadDim) w |= (uint32_t)scratch[c] << (k * BITS);
      }
      dst[lane] = w;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// One per-channel key block (T tokens x 128 channels, staged in shared
// memory) quantized by a whole CTA.
// ---------------------------------------------------------------------------
struct BlockSmem {
  __half* tile;    // [T][128]
  uint32_t* mask;  // [T][4] outlier bits
  float* s;        // [128]
  float* z;        // [128]
  float* r;        // [128]
  float* red;      // [4][128]
};

__device__ __forceinline__ BlockSmem carve_block_smem(unsigned char* base, int T) {
  BlockSmem b;
  b.tile = reinterpret_cast<__half*>(base);
  b.mask = reinterpret_cast<uint32_t*>(base + (size_t)T * kHeadDim * 2);
  b.s = reinterpret_cast<float*>(base + (size_t)T * kHeadDim * 2 + (size_t)T * 16);
  b.z = b.s + kHeadDim;
  b.r = b.z + kHeadDim;
  b.red = b.r + kHeadDim;
  return b;
}

inline size_t block_smem_bytes(int T) {
  return (size_t)T * kHeadDim * 2 + (size_t)T * 16 + 7 * kHeadDim * sizeof(float);
}

template <int BITS>
__device__ void quant_kblock(const BlockSmem& sm, int T, int t0, int blk, const TensorDev& K,
                             int n, int kout) {
  using P = Pack<BITS>;
  constexpr int levels = (1 << BITS) - 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = blockDim.x >> 5;
  // 1. per-row outliers
  if (kout > 0) {
    for (int row = warp; row < T; row += nwarp) {
      float x[4];
      load_row4(sm.tile + (size_t)row * kHeadDim, lane, x);
      int sel[kMaxOutliers];
      uint32_t om = warp_topk(x, kout, lane, sel);
      uint32_t part = om << (4 * (lane & 7));
      part |= __shfl_xor_sync(kFull, part, 1);
      part |= __shfl_xor_sync(kFull, part, 2);
      part |= __shfl_xor_sync(kFull, part, 4);
      if ((lane & 7) == 0) sm.mask[row * 4 + (lane >> 3)] = part;
      store_outliers(K, n, t0 + row, kout, x, sel, lane);
    }
    __syncthreads();
  }
  // 2. per-channel statistics over the T tokens (two threads per channel)
  {
    const int c = tid & (kHeadDim - 1);
    const int h = tid >> 7;  // 0 or 1
    const int half_rows = T >> 1;
    float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
    for (int row = h * half_rows; row < (h + 1) * half_rows; ++row) {
      bool masked = kout > 0 && ((sm.mask[row * 4 + (c >> 5)] >> (c & 31)) & 1u);
      if (!masked) {
        float v = __half2float(sm.tile[(size_t)row * kHeadDim + c]);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
    }
    sm.red[h * kHeadDim + c] = mn;
    sm.red[(2 + h) * kHeadDim + c] = mx;
  }
  __syncthreads();
  if (tid < kHeadDim) {
    const int c = tid;
    float mn = fminf(sm.red[c], sm.red[kHeadDim + c]);
    float mx = fmaxf(sm.red[2 * kHeadDim + c], sm.red[3 * kHeadDim + c]);
    if (mn > mx) {
      mn = 0.0f;
      mx = 0.0f;
    }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)levels));
    __half z16 = __float2half_rn(mn);
    reinterpret_cast<__half2*>(K.meta + (int64_t)n * K.meta_sstride)[(int64_t)blk * kHeadDim + c] =
        __halves2half2(s16, z16);
    float s = __half2float(s16);
    sm.s[c] = s;
    sm.z[c] = __half2float(z16);
    sm.r[c] = s > 0.0f ? __frcp_rn(s) : 0.0f;
  }
  __syncthreads();
  // 3. codes and packed rows
  uint32_t* dst = K.codes + (int64_t)n * K.codes_sstride + (int64_t)t0 * P::kWords;
  for (int item = tid; item < T * P::kWords; item += blockDim.x) {
    const int row = item / P::kWords;
    const int w = item - row * P::kWords;
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < P::kCpw; ++k) {
      const int c = w * P::kCpw + k;
      if (c < kHeadDim) {
        bool masked = kout > 0 && ((sm.mask[row * 4 + (c >> 5)] >> (c & 31)) & 1u);
        const float s = sm.s[c];
        int code = 0;
        if (!masked && s > 0.0f) {
          float x = __half2float(sm.tile[(size_t)row * kHeadDim + c]);
          code = min(max(quant_step(__fsub_rn(x, sm.z[c]), s, sm.r[c]), 0), levels);
        }
        word |= (uint32_t)code << (k * BITS);
      }
    }
    dst[item] = word;
  }
}

// ---------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------
template <int KB, int KMODE, int VB, bool VSYM>
__global__ void __launch_bounds__(256)
    append_kernel(LayerDev L, const __half* __restrict__ k1, const __half* __restrict__ v1,
                  int pos_all, const VarPos vp) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ __align__(16) uint8_t scratch[2][kHeadDim];
  const int n = blockIdx.x;
  // the stream's row: its batch row's own length with variable lengths (per-token keys)
  const int pos = vp.on ? vp.pos[n / vp.hkv] : pos_all;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const __half* kn = k1 + (int64_t)n * kHeadDim;
  if (warp == 0) quant_row_warp<VB, VSYM>(v1 + (int64_t)n * kHeadDim, L.v, n, pos, L.outliers,
                                          lane, scratch[0]);
  if (KMODE != KVQ_ASYM_PER_CHANNEL) {
    if (warp == 1)
      quant_row_warp<KB, KMODE == KVQ_SYM_PER_TOKEN>(kn, L.k, n, pos, L.outliers, lane,
                                                     scratch[1]);
  } else {
    const int T = L.k.group;
    const int r = pos % T;
    __half* res = L.k.resid + (int64_t)n * L.k.resid_sstride;
    if (warp == 1) {
      reinterpret_cast<uint2*>(res + (size_t)r * kHeadDim)[lane] =
          reinterpret_cast<const uint2*>(kn)[lane];
    }
    if (r == T - 1) {  // the residual is full: quantize the block
      BlockSmem sm = carve_block_smem(smem_raw, T);
      uint4* d4 = reinterpret_cast<uint4*>(sm.tile);
      const uint4* r4 = reinterpret_cast<const uint4*>(res);
      const uint4* k4 = reinterpret_cast<const uint4*>(kn);
      for (int i = threadIdx.x; i < T * (kHeadDim / 8); i += blockDim.x) {
        const int row = i / (kHeadDim / 8);
        d4[i] = row == T - 1 ? k4[i - row * (kHeadDim / 8)] : r4[i];
      }
      __syncthreads();
      quant_kblock<KB>(sm, T, pos - r, pos / T, L.k, n, L.outliers);
    }
  }
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
template <typename F>
cudaError_t ensure_smem(F* kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int KB, int KMODE, int VB, bool VSYM>
cudaError_t launch_append_t(const LayerDev& L, const __half* k1, const __half* v1, int pos, const VarPos& vp,
                            cudaStream_t st) {
  size_t sm = 0;
  if (KMODE == KVQ_ASYM_PER_CHANNEL) {  // a key block fills (in some row, with variable lengths)
    bool flush = (pos % L.k.group) == L.k.group - 1;
    if (vp.on) {
      flush = false;
      for (int b = 0; b < vp.rows; ++b) flush = flush || (vp.pos[b] % L.k.group) == L.k.group - 1;
    }
    if (flush) sm = block_smem_bytes(L.k.group);
  }
  cudaError_t e = ensure_smem(append_kernel<KB, KMODE, VB, VSYM>, sm);
  if (e != cudaSuccess) return e;
  append_kernel<KB, KMODE, VB, VSYM><<<L.n_streams, 256, sm, st>>>(L, k1, v1, pos, vp);
  return cudaGetLastError();
}

template <int KB, int KMODE>
cudaError_t launch_append_v(const LayerDev& L, const __half* k1, const __half* v1, int pos, const VarPos& vp,
                            cudaStream_t st) {
  if (L.v.mode == KVQ_SYM_PER_TOKEN) return launch_append_t<KB, KMODE, 8, true>(L, k1, v1, pos, vp, st);
  switch (L.v.bits) {
    case 3: return launch_append_t<KB, KMODE, 3, false>(L, k1, v1, pos, vp, st);
    case 4: return launch_append_t<KB, KMODE, 4, false>(L, k1, v1, pos, vp, st);
    default: return launch_append_t<KB, KMODE, 8, false>(L, k1, v1, pos, vp, st);
  }
}

}  // namespace

cudaError_t launch_append(const LayerDev& L, const __half* k1, const __half* v1, int pos, const VarPos& vp,
                          cudaStream_t st) {
  if (L.k.mode == KVQ_CODEBOOK_PER_TOKEN) return launch_codebook_rows(L, k1, v1, 1, 1, vp, pos, st);
  if (L.k.mode == KVQ_SYM_PER_TOKEN) return launch_append_v<8, KVQ_SYM_PER_TOKEN>(L, k1, v1, pos, vp, st);
  if (L.k.mode == KVQ_ASYM_PER_TOKEN) {
    switch (L.k.bits) {
      case 3: return launch_append_v<3, KVQ_ASYM_PER_TOKEN>(L, k1, v1, pos, vp, st);
      case 4: return launch_append_v<4, KVQ_ASYM_PER_TOKEN>(L, k1, v1, pos, vp, st);
      default: return launch_append_v<8, KVQ_ASYM_PER_TOKEN>(L, k1, v1, pos, vp, st);
    }
  }
  switch (L.k.bits) {
    case 3: return launch_append_v<3, KVQ_ASYM_PER_CHANNEL>(L, k1, v1, pos, vp, st);
    case 4: return launch_append_v<4, KVQ_ASYM_PER_CHANNEL>(L, k1, v1, pos, vp, st);
    default: return launch_append_v<8, KVQ_ASYM_PER_CHANNEL>(L, k1, v1, pos, vp, st);
  }
}

}  // namespace kvq
