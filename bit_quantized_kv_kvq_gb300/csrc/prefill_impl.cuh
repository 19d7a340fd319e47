// Prefill quantize: one launch quantizes a whole prompt of one layer.
//
// Grid: x = key CTAs then value CTAs of one stream, y = stream (batch,
// kv-head). A row CTA (256 threads) quantizes 64 consecutive (token, head)
// rows per token: a half-warp owns a row, a lane 8 channels (one 16-byte
// load). A key-block CTA quantizes one per-channel block of T tokens: a
// thread owns 8 channels of T/16 rows, kept in registers between the
// statistics and the code pass.
//
// Codec (TurboQuant 3-bit KV quantization page, dpshk.com/news/6341316,
// §3.1; KVQuant page, cf-1.com/news/2306543, §2.2; NIAH q8_0 write-up,
// cf-1.com/news/5482713, §1.2): group min/max (or absmax), fp16 scale and
// zero point from fp32 arithmetic with explicit round-to-nearest steps,
// code = clamp(rne((x - z) / s)). Outliers (the k largest |x| of a row, ties
// to the lower channel) are stored as fp16 CSR entries, left out of the
// group statistics and coded 0.
#pragma once

#include "common.cuh"

namespace kvq {
namespace pf {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;
constexpr int kRowsPerCta = 64;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: x + kMagic holds rne(x) in its low bits
constexpr uint32_t kMagicBits = 0x4B400000u;

__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Codes: rne(d / s) for |d / s| < 2^21. r approximates 1/s within one ulp,
// so d*r is within a few ulp of the IEEE quotient and both round to the same
// integer unless d*r lies within 2^-12 of a half-integer; only those rare
// elements are redone by quot_exact with the IEEE quotient (behind a warp
// vote, so the division is a real branch, not predicated code). Rounding to
// an integer adds and subtracts 1.5 * 2^23.
static __device__ __noinline__ int quot_exact(float d, float s) {
  return (int)(__float_as_uint(__fadd_rn(__fdiv_rn(d, s), kMagic)) - kMagicBits);
}

constexpr float kNear = 0.5f - 0x1p-12f;

// Eight codes of one lane, asymmetric: c_i = min(rne((x_i - z) / s), LEVELS)
// for live slots (bit i of `dead` clear and s > 0), else 0. The fp32 steps
// run on packed pairs (f32x2, each element rounded to nearest even exactly as
// the scalar operation): d = x - z, q = d * r, min, q + 1.5*2^23 (rounding to
// an integer) and the distance to it; the rare near-half elements are redone
// with the IEEE quotient behind a warp vote.
template <int LEVELS>
__device__ __forceinline__ void codes8_asym(const float (&x)[8], float z, float s, float r,
                                            uint32_t dead, int (&c)[8]) {
  const uint64_t NZ = f2_pack(-z, -z), R = f2_pack(r, r);
  const uint64_t MG = f2_pack(kMagic, kMagic), NMG = f2_pack(-kMagic, -kMagic);
  const uint64_t NEG1 = f2_pack(-1.0f, -1.0f);
  const bool sok = s > 0.0f;
  uint32_t need = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float q0, q1;
    f2_unpack(f2_mul(f2_add(f2_pack(x[2 * p], x[2 * p + 1]), NZ), R), q0, q1);
    q0 = fminf(q0, (float)LEVELS);
    q1 = fminf(q1, (float)LEVELS);
    const uint64_t Q = f2_pack(q0, q1);
    const uint64_t CF = f2_add(Q, MG);
    float d0, d1, c0, c1;
    f2_unpack(f2_fma(f2_add(CF, NMG), NEG1, Q), d0, d1);
    f2_unpack(CF, c0, c1);
    const bool on0 = sok && !((dead >> (2 * p)) & 1u);
    const bool on1 = sok && !((dead >> (2 * p + 1)) & 1u);
    c[2 * p] = on0 ? (int)(__float_as_uint(c0) - kMagicBits) : 0;
    c[2 * p + 1] = on1 ? (int)(__float_as_uint(c1) - kMagicBits) : 0;
    need |= (on0 && fabsf(d0) >= kNear) ? 1u << (2 * p) : 0u;
    need |= (on1 && fabsf(d1) >= kNear) ? 1u << (2 * p + 1) : 0u;
  }
  if (__any_sync(kFull, need != 0)) {
    for (int i = 0; i < 8; ++i)
      if ((need >> i) & 1u) c[i] = min(quot_exact(__fsub_rn(x[i], z), s), LEVELS);
  }
}

// Symmetric: c_i = clamp(rne(x_i / s), -QMAX, QMAX) (two's complement later).
template <int QMAX>
__device__ __forceinline__ void codes8_sym(const float (&x)[8], float s, float r, uint32_t dead,
                                           int (&c)[8]) {
  const uint64_t R = f2_pack(r, r);
  const uint64_t MG = f2_pack(kMagic, kMagic), NMG = f2_pack(-kMagic, -kMagic);
  const uint64_t NEG1 = f2_pack(-1.0f, -1.0f);
  const bool sok = s > 0.0f;
  uint32_t need = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float q0, q1;
    f2_unpack(f2_mul(f2_pack(x[2 * p], x[2 * p + 1]), R), q0, q1);
    q0 = fmaxf(fminf(q0, (float)QMAX), -(float)QMAX);
    q1 = fmaxf(fminf(q1, (float)QMAX), -(float)QMAX);
    const uint64_t Q = f2_pack(q0, q1);
    const uint64_t CF = f2_add(Q, MG);
    float d0, d1, c0, c1;
    f2_unpack(f2_fma(f2_add(CF, NMG), NEG1, Q), d0, d1);
    f2_unpack(CF, c0, c1);
    const bool on0 = sok && !((dead >> (2 * p)) & 1u);
    const bool on1 = sok && !((dead >> (2 * p + 1)) & 1u);
    c[2 * p] = on0 ? (int)(__float_as_uint(c0) - kMagicBits) : 0;
    c[2 * p + 1] = on1 ? (int)(__float_as_uint(c1) - kMagicBits) : 0;
    need |= (on0 && fabsf(d0) >= kNear) ? 1u << (2 * p) : 0u;
    need |= (on1 && fabsf(d1) >= kNear) ? 1u << (2 * p + 1) : 0u;
  }
  if (__any_sync(kFull, need != 0)) {
    for (int i = 0; i < 8; ++i)
      if ((need >> i) & 1u) c[i] = min(max(quot_exact(x[i], s), -QMAX), QMAX);
  }
}


// Per-channel keys: as codes8_asym with a scale, zero point and reciprocal
// per element (one per channel).
template <int LEVELS>
__device__ __forceinline__ void codes8_kblock(const float (&x)[8], const float (&z)[8],
                                              const float (&s)[8], const float (&r)[8],
                                              uint32_t dead, int (&c)[8]) {
  const uint64_t MG = f2_pack(kMagic, kMagic), NMG = f2_pack(-kMagic, -kMagic);
  const uint64_t NEG1 = f2_pack(-1.0f, -1.0f);
  uint32_t need = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float q0, q1;
    const uint64_t D = f2_add(f2_pack(x[2 * p], x[2 * p + 1]), f2_pack(-z[2 * p], -z[2 * p + 1]));
    f2_unpack(f2_mul(D, f2_pack(r[2 * p], r[2 * p + 1])), q0, q1);
    q0 = fminf(q0, (float)LEVELS);
    q1 = fminf(q1, (float)LEVELS);
    const uint64_t Q = f2_pack(q0, q1);
    const uint64_t CF = f2_add(Q, MG);
    float d0, d1, c0, c1;
    f2_unpack(f2_fma(f2_add(CF, NMG), NEG1, Q), d0, d1);
    f2_unpack(CF, c0, c1);
    const bool on0 = s[2 * p] > 0.0f && !((dead >> (2 * p)) & 1u);
    const bool on1 = s[2 * p + 1] > 0.0f && !((dead >> (2 * p + 1)) & 1u);
    c[2 * p] = on0 ? (int)(__float_as_uint(c0) - kMagicBits) : 0;
    c[2 * p + 1] = on1 ? (int)(__float_as_uint(c1) - kMagicBits) : 0;
    need |= (on0 && fabsf(d0) >= kNear) ? 1u << (2 * p) : 0u;
    need |= (on1 && fabsf(d1) >= kNear) ? 1u << (2 * p + 1) : 0u;
  }
  if (__any_sync(kFull, need != 0)) {
    for (int i = 0; i < 8; ++i)
      if ((need >> i) & 1u) c[i] = min(quot_exact(__fsub_rn(x[i], z[i]), s[i]), LEVELS);
  }
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void unpack8(const uint4& raw, float (&x)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __low2float(h[i]);
    x[2 * i + 1] = __high2float(h[i]);
  }
}

__device__ __forceinline__ float pick8(const float (&x)[8], int i) {
  float v = x[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) v = (i == k) ? x[k] : v;
  return v;
}

// Top-k of a 128-channel row held by one half-warp (lane l16 holds channels
// 8*l16 .. 8*l16+7): |x| descending, ties to the lower channel. Returns the
// lane's 8-bit slot mask; sel[0..k) gets the channels in ascending order.
__device__ __forceinline__ uint32_t half_topk(const float (&x)[8], int k, int l16,
                                              int (&sel)[kMaxOutliers]) {
  uint32_t m = 0;
  for (int it = 0; it < k; ++it) {
    float bm = -1.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (!((m >> i) & 1u)) {
        const float a = fabsf(x[i]);
        if (a > bm) {
          bm = a;
          bi = l16 * 8 + i;
        }
      }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
      const float om = __shfl_xor_sync(kFull, bm, off);
      const int oi = __shfl_xor_sync(kFull, bi, off);
      if (om > bm || (om == bm && oi < bi)) {
        bm = om;
        bi = oi;
      }
    }
    if ((bi >> 3) == l16) m |= 1u << (bi & 7);
    sel[it] = bi;
  }
  for (int i = 1; i < k; ++i) {
    const int v = sel[i];
    int j = i - 1;
    while (j >= 0 && sel[j] > v) {
      sel[j + 1] = sel[j];
      --j;
    }
    sel[j + 1] = v;
  }
  return m;
}

// CSR entries of one row (every lane of the half-warp calls; lane 0 stores).
__device__ __forceinline__ void store_row_outliers(const TensorDev& T, int n, int row, int k,
                                                   const float (&x)[8],
                                                   const int (&sel)[kMaxOutliers], int lane,
                                                   bool live) {
  const int l16 = lane & 15;
  const int hb = lane & 16;
  const int64_t base = (int64_t)n * T.out_sstride + (int64_t)row * k;
  for (int i = 0; i < k; ++i) {
    const int c = sel[i];
    const float v = __shfl_sync(kFull, pick8(x, c & 7), hb | (c >> 3));
    if (live && l16 == 0) {
      T.col[base + i] = (uint16_t)c;
      T.val[base + i] = __float2half_rn(v);  // exact: v came from an fp16
    }
  }
  if (live && l16 == 0) {
    int32_t* rp = T.rowptr + (int64_t)n * T.rowptr_sstride;
    rp[row + 1] = (row + 1) * k;
    if (row == 0) rp[0] = 0;
  }
}

template <int BITS>
__device__ __forceinline__ void store_packed8(uint32_t* rowdst, const int (&c)[8], int l16,
                                              uint8_t* scratch, bool live) {
  if (BITS == 4) {
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) w |= (uint32_t)c[k] << (4 * k);
    if (live) rowdst[l16] = w;
  } else if (BITS == 8) {
    uint2 w;
    w.x = (uint32_t)(c[0] & 0xFF) | ((uint32_t)(c[1] & 0xFF) << 8) | ((uint32_t)(c[2] & 0xFF) << 16) |
          ((uint32_t)(c[3] & 0xFF) << 24);
    w.y = (uint32_t)(c[4] & 0xFF) | ((uint32_t)(c[5] & 0xFF) << 8) | ((uint32_t)(c[6] & 0xFF) << 16) |
          ((uint32_t)(c[7] & 0xFF) << 24);
    if (live) reinterpret_cast<uint2*>(rowdst)[l16] = w;
  } else {
    uint2 b;
    b.x = (uint32_t)c[0] | ((uint32_t)c[1] << 8) | ((uint32_t)c[2] << 16) | ((uint32_t)c[3] << 24);
    b.y = (uint32_t)c[4] | ((uint32_t)c[5] << 8) | ((uint32_t)c[6] << 16) | ((uint32_t)c[7] << 24);
    reinterpret_cast<uint2*>(scratch)[l16] = b;
    __syncwarp();
    if (l16 < Pack<3>::kWords) {
      uint32_t w = 0;
#pragma unroll
      for (int k = 0; k < 10; ++k) {
        const int ch = l16 * 10 + k;
        if (ch < kHeadDim) w |= (uint32_t)scratch[ch] << (3 * k);
      }
      if (live) rowdst[l16] = w;
    }
    __syncwarp();
  }
}

// One per-token row on a half-warp.
template <int BITS, bool SYM>
__device__ __forceinline__ void quant_row16(const uint4& raw, bool live, const TensorDev& T,
                                            int n, int row, int kout, int lane,
                                            uint8_t* scratch) {
  const int l16 = lane & 15;
  float x[8];
  unpack8(raw, x);
  uint32_t om = 0;
  if (kout > 0) {
    int sel[kMaxOutliers];
    om = half_topk(x, kout, l16, sel);
    store_row_outliers(T, n, row, kout, x, sel, lane, live);
  }
  const int lpg = T.group >> 3;  // lanes per group
  int c[8];
  __half s16, z16;
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
  const __half2 pinf2 = bits_h2(0x7C007C00u);
  if (SYM) {
    constexpr int qmax = (1 << (BITS - 1)) - 1;
    __half2 a2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a2[j] = __habs2(h[j]);
      if (kout > 0)
        a2[j] = __halves2half2(((om >> (2 * j)) & 1u) ? __float2half_rn(0.0f) : __low2half(a2[j]),
                               ((om >> (2 * j + 1)) & 1u) ? __float2half_rn(0.0f) : __high2half(a2[j]));
    }
    __half2 m = __hmax2(__hmax2(a2[0], a2[1]), __hmax2(a2[2], a2[3]));
    m = __hmax2(m, __lowhigh2highlow(m));
    for (int off = 1; off < lpg; off <<= 1) m = __hmax2(m, bits_h2(__shfl_xor_sync(kFull, h2_bits(m), off)));
    const float am = __low2float(m);
    s16 = __float2half_rn(__fdiv_rn(am, (float)qmax));
    z16 = __float2half_rn(0.0f);
    const float sc = __half2float(s16);
    codes8_sym<qmax>(x, sc, rcp_approx(sc), om, c);
  } else {
    constexpr int levels = (1 << BITS) - 1;
    __half2 lo2[4], hi2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      lo2[j] = h[j];
      hi2[j] = __hneg2(h[j]);  // max through min of the negation
      if (kout > 0) {
        const bool a = (om >> (2 * j)) & 1u, b2 = (om >> (2 * j + 1)) & 1u;
        lo2[j] = __halves2half2(a ? __low2half(pinf2) : __low2half(lo2[j]), b2 ? __low2half(pinf2) : __high2half(lo2[j]));
        hi2[j] = __halves2half2(a ? __low2half(pinf2) : __low2half(hi2[j]), b2 ? __low2half(pinf2) : __high2half(hi2[j]));
      }
    }
    const __half2 mn2 = __hmin2(__hmin2(lo2[0], lo2[1]), __hmin2(lo2[2], lo2[3]));
    const __half2 nx2 = __hmin2(__hmin2(hi2[0], hi2[1]), __hmin2(hi2[2], hi2[3]));
    // (min, -max) of the lane in one half2, then one shuffle per level
    __half2 pr = __hmin2(__halves2half2(__low2half(mn2), __low2half(nx2)),
                         __halves2half2(__high2half(mn2), __high2half(nx2)));
    for (int off = 1; off < lpg; off <<= 1) pr = __hmin2(pr, bits_h2(__shfl_xor_sync(kFull, h2_bits(pr), off)));
    float mn = __low2float(pr), mx = -__high2float(pr);
    if (mn > mx) {  // every member an outlier
      mn = 0.0f;
      mx = 0.0f;
    }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)levels));
    z16 = __float2half_rn(mn);
    const float sc = __half2float(s16);
    codes8_asym<levels>(x, __half2float(z16), sc, rcp_approx(sc), om, c);
  }
  if (live && (l16 & (lpg - 1)) == 0) {
    const int g = l16 / lpg;
    const int per_row = kHeadDim / T.group;
    unsigned char* mb = T.meta + (int64_t)n * T.meta_sstride;
    if (SYM)
      reinterpret_cast<__half*>(mb)[(int64_t)row * per_row + g] = s16;
    else
      reinterpret_cast<__half2*>(mb)[(int64_t)row * per_row + g] = __halves2half2(s16, z16);
  }
  uint32_t* rowdst = T.codes + (int64_t)n * T.codes_sstride + (int64_t)row * Pack<BITS>::kWords;
  store_packed8<BITS>(rowdst, c, l16, scratch, live);
}

template <int BITS, bool SYM>
__device__ __forceinline__ void rows_cta(const TensorDev& T, const __half* __restrict__ src, int n,
                                         int row0, int seq_len, int kout, uint8_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const __half* base = src + (int64_t)n * seq_len * kHeadDim;
  uint4 raw[4];
  int rows[4];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = row0 + warp * 8 + it * 2 + (lane >> 4);
    rows[it] = r;
    raw[it] = r < seq_len
                  ? __ldcs(reinterpret_cast<const uint4*>(base + (int64_t)r * kHeadDim) + (lane & 15))
                  : make_uint4(0, 0, 0, 0);
  }
  uint8_t* my = scratch + (warp * 2 + (lane >> 4)) * kHeadDim;
#pragma unroll
  for (int it = 0; it < 4; ++it)
    quant_row16<BITS, SYM>(raw[it], rows[it] < seq_len, T, n, rows[it], kout, lane, my);
}

// Shared memory of a key-block CTA.
template <int BITS, int R>
struct KBlockSmem {
  __half2 mn[8][64];
  __half2 mx[8][64];
  float s[kHeadDim], z[kHeadDim], r[kHeadDim];
  uint8_t stage3[BITS == 3 ? 16 * R * kHeadDim : 16];
};

template <int BITS, int R>
__device__ __forceinline__ void kblock_cta(const TensorDev& K, const __half* __restrict__ src,
                                           int n, int blk, int seq_len, int kout,
                                           KBlockSmem<BITS, R>& sm) {
  constexpr int T = 16 * R;
  constexpr int levels = (1 << BITS) - 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int w16 = tid & 15, rg = tid >> 4;
  const int t0 = blk * T;
  const __half* base = src + ((int64_t)n * seq_len + t0) * kHeadDim;
  uint4 raw[R];
#pragma unroll
  for (int i = 0; i < R; ++i)
    raw[i] = __ldcs(reinterpret_cast<const uint4*>(base + (int64_t)(rg + 16 * i) * kHeadDim) + w16);
  uint32_t om[R];
#pragma unroll
  for (int i = 0; i < R; ++i) om[i] = 0;
  if (kout > 0) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      float x[8];
      unpack8(raw[i], x);
      int sel[kMaxOutliers];
      om[i] = half_topk(x, kout, w16, sel);
      store_row_outliers(K, n, t0 + rg + 16 * i, kout, x, sel, lane, true);
    }
  }
  // per-channel min / max over the block (fp16 compares are exact)
  const __half2 pinf = __halves2half2(__ushort_as_half(0x7C00), __ushort_as_half(0x7C00));
  const __half2 ninf = __halves2half2(__ushort_as_half(0xFC00), __ushort_as_half(0xFC00));
  __half2 mn2[4], mx2[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mn2[j] = pinf;
    mx2[j] = ninf;
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const __half2* h = reinterpret_cast<const __half2*>(&raw[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 vmin = h[j], vmax = h[j];
      if (kout > 0) {
        const bool mlo = (om[i] >> (2 * j)) & 1u, mhi = (om[i] >> (2 * j + 1)) & 1u;
        vmin = __halves2half2(mlo ? __low2half(pinf) : __low2half(h[j]),
                              mhi ? __low2half(pinf) : __high2half(h[j]));
        vmax = __halves2half2(mlo ? __low2half(ninf) : __low2half(h[j]),
                              mhi ? __low2half(ninf) : __high2half(h[j]));
      }
      mn2[j] = __hmin2(mn2[j], vmin);
      mx2[j] = __hmax2(mx2[j], vmax);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a = *reinterpret_cast<uint32_t*>(&mn2[j]);
    uint32_t b = *reinterpret_cast<uint32_t*>(&mx2[j]);
    uint32_t oa = __shfl_xor_sync(kFull, a, 16), ob = __shfl_xor_sync(kFull, b, 16);
    mn2[j] = __hmin2(mn2[j], *reinterpret_cast<__half2*>(&oa));
    mx2[j] = __hmax2(mx2[j], *reinterpret_cast<__half2*>(&ob));
  }
  if (lane < 16) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sm.mn[warp][4 * w16 + j] = mn2[j];
      sm.mx[warp][4 * w16 + j] = mx2[j];
    }
  }
  __syncthreads();
  if (tid < 64) {
    __half2 a = sm.mn[0][tid], b = sm.mx[0][tid];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      a = __hmin2(a, sm.mn[w][tid]);
      b = __hmax2(b, sm.mx[w][tid]);
    }
    __half2 meta[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mn = __half2float(e ? __high2half(a) : __low2half(a));
      float mx = __half2float(e ? __high2half(b) : __low2half(b));
      if (mn > mx) {  // every member an outlier
        mn = 0.0f;
        mx = 0.0f;
      }
      mn = __fadd_rn(mn, 0.0f);
      mx = __fadd_rn(mx, 0.0f);
      const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)levels));
      const __half z16 = __float2half_rn(mn);
      meta[e] = __halves2half2(s16, z16);
      const int c = 2 * tid + e;
      const float s = __half2float(s16);
      sm.s[c] = s;
      sm.z[c] = __half2float(z16);
      sm.r[c] = rcp_approx(s);
    }
    unsigned char* mb = K.meta + (int64_t)n * K.meta_sstride;
    reinterpret_cast<uint2*>(mb)[(int64_t)blk * (kHeadDim / 2) + tid] =
        make_uint2(*reinterpret_cast<uint32_t*>(&meta[0]), *reinterpret_cast<uint32_t*>(&meta[1]));
  }
  __syncthreads();
  float s[8], z[8], r[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    s[k] = sm.s[8 * w16 + k];
    z[k] = sm.z[8 * w16 + k];
    r[k] = sm.r[8 * w16 + k];
  }
  uint32_t* kdst = K.codes + (int64_t)n * K.codes_sstride + (int64_t)t0 * Pack<BITS>::kWords;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    float x[8];
    unpack8(raw[i], x);
    int c[8];
    codes8_kblock<levels>(x, z, s, r, om[i], c);
    const int row = rg + 16 * i;
    if (BITS == 3) {
      uint2 b;
      b.x = (uint32_t)c[0] | ((uint32_t)c[1] << 8) | ((uint32_t)c[2] << 16) | ((uint32_t)c[3] << 24);
      b.y = (uint32_t)c[4] | ((uint32_t)c[5] << 8) | ((uint32_t)c[6] << 16) | ((uint32_t)c[7] << 24);
      reinterpret_cast<uint2*>(sm.stage3 + row * kHeadDim)[w16] = b;
    } else {
      store_packed8<BITS>(kdst + (int64_t)row * Pack<BITS>::kWords, c, w16, nullptr, true);
    }
  }
  if (BITS == 3) {
    __syncthreads();
    constexpr int W3 = Pack<3>::kWords;
    for (int item = tid; item < T * W3; item += kThreads) {
      const int row = item / W3;
      const int w = item - row * W3;
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 10; ++k) {
        const int ch = w * 10 + k;
        if (ch < kHeadDim) word |= (uint32_t)sm.stage3[row * kHeadDim + ch] << (3 * k);
      }
      kdst[item] = word;
    }
  }
}

__device__ __forceinline__ void resid_copy(const TensorDev& K, const __half* __restrict__ src,
                                           int n, int t0, int seq_len) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src + ((int64_t)n * seq_len + t0) * kHeadDim);
  uint4* d4 = reinterpret_cast<uint4*>(K.resid + (int64_t)n * K.resid_sstride);
  const int count = (seq_len - t0) * (kHeadDim / 8);
  for (int i = threadIdx.x; i < count; i += kThreads) d4[i] = s4[i];
}

struct PrefillArgs {
  TensorDev k, v;
  const __half* ksrc;
  const __half* vsrc;
  int seq_len;
  int kout;
  int k_ctas;   // key CTAs per stream
  int k_nfull;  // whole per-channel key blocks per stream
};

template <int KB, int KMODE, int KR, int VB, bool VSYM>
struct PrefillSmem {
  static constexpr size_t kKB = KMODE == KVQ_ASYM_PER_CHANNEL ? sizeof(KBlockSmem<KB, KR>) : 0;
  static constexpr size_t kRows = 16 * kHeadDim;
  static constexpr size_t bytes = kKB > kRows ? kKB : kRows;
};

template <int KB, int KMODE, int KR, int VB, bool VSYM>
__global__ void __launch_bounds__(kThreads) prefill_kernel(PrefillArgs a) {
  using SM = PrefillSmem<KB, KMODE, KR, VB, VSYM>;
  __shared__ __align__(16) unsigned char smem[SM::bytes];
  const int n = blockIdx.y;
  const int x = blockIdx.x;
  if (x < a.k_ctas) {
    if (KMODE == KVQ_ASYM_PER_CHANNEL) {
      if (x < a.k_nfull)
        kblock_cta<KB, KR>(a.k, a.ksrc, n, x, a.seq_len, a.kout,
                           *reinterpret_cast<KBlockSmem<KB, KR>*>(smem));
      else
        resid_copy(a.k, a.ksrc, n, a.k_nfull * 16 * KR, a.seq_len);
    } else {
      rows_cta<KB, KMODE == KVQ_SYM_PER_TOKEN>(a.k, a.ksrc, n, x * kRowsPerCta, a.seq_len, a.kout,
                                               smem);
    }
  } else {
    rows_cta<VB, VSYM>(a.v, a.vsrc, n, (x - a.k_ctas) * kRowsPerCta, a.seq_len, a.kout, smem);
  }
}

template <int KB, int KMODE, int KR, int VB, bool VSYM>
cudaError_t launch_prefill_t(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                             cudaStream_t st) {
  PrefillArgs a;
  a.k = L.k;
  a.v = L.v;
  a.ksrc = k;
  a.vsrc = v;
  a.seq_len = seq_len;
  a.kout = L.outliers;
  const int row_ctas = (seq_len + kRowsPerCta - 1) / kRowsPerCta;
  if (KMODE == KVQ_ASYM_PER_CHANNEL) {
    a.k_nfull = seq_len / L.k.group;
    a.k_ctas = a.k_nfull + (seq_len % L.k.group ? 1 : 0);
  } else {
    a.k_nfull = 0;
    a.k_ctas = row_ctas;
  }
  dim3 grid(a.k_ctas + row_ctas, L.n_streams);
  prefill_kernel<KB, KMODE, KR, VB, VSYM><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

// Dispatch over key codecs for one value codec.
template <int VB, bool VSYM>
cudaError_t launch_prefill_v(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                             cudaStream_t st) {
  if (VSYM) {
    if (L.k.mode != KVQ_SYM_PER_TOKEN) return cudaErrorNotSupported;
    return launch_prefill_t<8, KVQ_SYM_PER_TOKEN, 1, VB, VSYM>(L, k, v, seq_len, st);
  }
  if (L.k.mode == KVQ_ASYM_PER_CHANNEL) {
    const int R = L.k.group / 16;
#define KVQ_KB(B)                                                                          \
  if (L.k.bits == B) {                                                                     \
    if (R == 4) return launch_prefill_t<B, KVQ_ASYM_PER_CHANNEL, 4, VB, VSYM>(L, k, v, seq_len, st); \
    if (R == 8) return launch_prefill_t<B, KVQ_ASYM_PER_CHANNEL, 8, VB, VSYM>(L, k, v, seq_len, st); \
    return launch_prefill_t<B, KVQ_ASYM_PER_CHANNEL, 16, VB, VSYM>(L, k, v, seq_len, st);  \
  }
    KVQ_KB(3)
    KVQ_KB(4)
    KVQ_KB(8)
#undef KVQ_KB
    return cudaErrorNotSupported;
  }
  if (L.k.mode == KVQ_ASYM_PER_TOKEN) {
    if (L.k.bits == 3) return launch_prefill_t<3, KVQ_ASYM_PER_TOKEN, 1, VB, VSYM>(L, k, v, seq_len, st);
    if (L.k.bits == 4) return launch_prefill_t<4, KVQ_ASYM_PER_TOKEN, 1, VB, VSYM>(L, k, v, seq_len, st);
    return launch_prefill_t<8, KVQ_ASYM_PER_TOKEN, 1, VB, VSYM>(L, k, v, seq_len, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace pf

cudaError_t launch_prefill_v3(const LayerDev& L, const __half* k, const __half* v, int s, cudaStream_t st);
cudaError_t launch_prefill_v4(const LayerDev& L, const __half* k, const __half* v, int s, cudaStream_t st);
cudaError_t launch_prefill_v8(const LayerDev& L, const __half* k, const __half* v, int s, cudaStream_t st);

}  // namespace kvq
