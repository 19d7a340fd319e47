// Prefill quantize: one launch quantizes a whole prompt of one layer.
//
// Grid: x = key CTAs then value CTAs of one stream, y = stream (batch,
// kv-head). A row CTA (256 threads) quantizes 128 consecutive (token, head)
// rows per token: 8 lanes own a row, a lane 16 channels (two 16-byte
// loads; all of a lane's loads are issued before the first row is coded). A key-block CTA quantizes one per-channel block of T tokens: a
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
constexpr int kRowsPerCta = 128;
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

// x + c in fp32 with x an fp16 value: one mixed-precision instruction,
// the same value as widening x and adding in fp32.
__device__ __forceinline__ float add_h_f(uint16_t xh, float c) {
  float r;
  asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(r) : "h"(xh), "f"(c));
  return r;
}

__device__ __forceinline__ void unpack16(const uint4 (&raw)[2], float (&x)[16]) {
#pragma unroll
  for (int v = 0; v < 2; ++v) {
    const __half2* h = reinterpret_cast<const __half2*>(&raw[v]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[8 * v + 2 * i] = __low2float(h[i]);
      x[8 * v + 2 * i + 1] = __high2float(h[i]);
    }
  }
}

// Fast path of 16 asymmetric codes (no outliers, s > 0 everywhere):
// cb[i] = bits of rne(min(RN(x_i - z) * r, LEVELS)) + 1.5*2^23, and the
// largest distance of an approximate quotient to its integer in *maxd.
template <int LEVELS>
__device__ __forceinline__ void codes16_fast_asym(const uint4 (&raw)[2], float z, float r,
                                                  uint32_t (&cb)[16], float& maxd) {
  const uint64_t R = f2_pack(r, r);
  const uint64_t MG = f2_pack(kMagic, kMagic), NMG = f2_pack(-kMagic, -kMagic);
  const uint64_t NEG1 = f2_pack(-1.0f, -1.0f);
  const uint16_t* hx = reinterpret_cast<const uint16_t*>(&raw[0]);
  const float nz = -z;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const float d0 = add_h_f(hx[2 * p], nz), d1 = add_h_f(hx[2 * p + 1], nz);
    float q0, q1;
    f2_unpack(f2_mul(f2_pack(d0, d1), R), q0, q1);
    const uint64_t Q = f2_pack(fminf(q0, (float)LEVELS), fminf(q1, (float)LEVELS));
    const uint64_t CF = f2_add(Q, MG);
    float e0, e1, c0, c1;
    f2_unpack(f2_fma(f2_add(CF, NMG), NEG1, Q), e0, e1);
    f2_unpack(CF, c0, c1);
    maxd = fmaxf(maxd, fmaxf(fabsf(e0), fabsf(e1)));
    cb[2 * p] = __float_as_uint(c0);
    cb[2 * p + 1] = __float_as_uint(c1);
  }
}

template <int QMAX>
__device__ __forceinline__ void codes16_fast_sym(const uint4 (&raw)[2], float r,
                                                 uint32_t (&cb)[16], float& maxd) {
  const uint64_t R = f2_pack(r, r);
  const uint64_t MG = f2_pack(kMagic, kMagic), NMG = f2_pack(-kMagic, -kMagic);
  const uint64_t NEG1 = f2_pack(-1.0f, -1.0f);
  const __half2* h = reinterpret_cast<const __half2*>(&raw[0]);
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const float2 xv = __half22float2(h[p]);
    float q0, q1;
    f2_unpack(f2_mul(f2_pack(xv.x, xv.y), R), q0, q1);
    const uint64_t Q = f2_pack(fmaxf(fminf(q0, (float)QMAX), -(float)QMAX),
                               fmaxf(fminf(q1, (float)QMAX), -(float)QMAX));
    const uint64_t CF = f2_add(Q, MG);
    float e0, e1, c0, c1;
    f2_unpack(f2_fma(f2_add(CF, NMG), NEG1, Q), e0, e1);
    f2_unpack(CF, c0, c1);
    maxd = fmaxf(maxd, fmaxf(fabsf(e0), fabsf(e1)));
    cb[2 * p] = __float_as_uint(c0);
    cb[2 * p + 1] = __float_as_uint(c1);
  }
}

// Packs codes held as bits of (code + 1.5*2^23): code k of a group of
// 32/BITS goes to bit k*BITS. For unsigned codes the sum of bits << k*BITS
// carries the magic in every slot; it is removed by one subtraction.
template <int BITS>
__device__ __forceinline__ uint32_t pack_word(const uint32_t* cb) {
  constexpr int n = 32 / BITS;
  constexpr uint32_t rep = BITS == 4 ? 0x11111111u : 0x01010101u;
  constexpr uint32_t off = kMagicBits * rep;
  uint32_t w = 0;
#pragma unroll
  for (int k = 0; k < n; ++k) w += cb[k] << (k * BITS);
  return w - off;
}

// Top-k of a 128-channel row held by 8 lanes (16 channels each).
__device__ __forceinline__ uint32_t oct_topk(const float (&x)[16], int k, int l8,
                                             int (&sel)[kMaxOutliers]) {
  uint32_t m = 0;
  for (int it = 0; it < k; ++it) {
    float bm = -1.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (!((m >> i) & 1u)) {
        const float a = fabsf(x[i]);
        if (a > bm) {
          bm = a;
          bi = l8 * 16 + i;
        }
      }
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {
      const float om = __shfl_xor_sync(kFull, bm, off);
      const int oi = __shfl_xor_sync(kFull, bi, off);
      if (om > bm || (om == bm && oi < bi)) {
        bm = om;
        bi = oi;
      }
    }
    if ((bi >> 4) == l8) m |= 1u << (bi & 15);
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

__device__ __forceinline__ float pick16(const float (&x)[16], int i) {
  float v = x[0];
#pragma unroll
  for (int k = 1; k < 16; ++k) v = (i == k) ? x[k] : v;
  return v;
}

// One per-token row on 8 lanes (lane l8 owns channels 16*l8 .. 16*l8+15).
template <int BITS, bool SYM>
__device__ __forceinline__ void quant_row8(const uint4 (&raw)[2], bool live, const TensorDev& T,
                                           int n, int row, int kout, int lane,
                                           uint8_t* scratch) {
  const int l8 = lane & 7;
  const int gb = lane & 24;
  uint32_t om = 0;
  float xf[16];
  if (kout > 0) {
    unpack16(raw, xf);
    int sel[kMaxOutliers];
    om = oct_topk(xf, kout, l8, sel);
    const int64_t base = (int64_t)n * T.out_sstride + (int64_t)row * kout;
    for (int i = 0; i < kout; ++i) {
      const int c = sel[i];
      const float v = __shfl_sync(kFull, pick16(xf, c & 15), gb | (c >> 4));
      if (live && l8 == 0) {
        T.col[base + i] = (uint16_t)c;
        T.val[base + i] = __float2half_rn(v);
      }
    }
    if (live && l8 == 0) {
      int32_t* rp = T.rowptr + (int64_t)n * T.rowptr_sstride;
      rp[row + 1] = (row + 1) * kout;
      if (row == 0) rp[0] = 0;
    }
  }
  const int lpg = T.group >> 4;  // lanes per group (groups of >= 16 channels)
  const __half2* h = reinterpret_cast<const __half2*>(&raw[0]);
  const __half2 pinf2 = bits_h2(0x7C007C00u);
  __half s16, z16;
  float sc, zc = 0.0f;
  if (SYM) {
    constexpr int qmax = (1 << (BITS - 1)) - 1;
    __half2 m = __float2half2_rn(0.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      __half2 a = __habs2(h[j]);
      if (kout > 0)
        a = __halves2half2(((om >> (2 * j)) & 1u) ? __float2half_rn(0.0f) : __low2half(a),
                           ((om >> (2 * j + 1)) & 1u) ? __float2half_rn(0.0f) : __high2half(a));
      m = __hmax2(m, a);
    }
    m = __hmax2(m, __lowhigh2highlow(m));
    for (int off = 1; off < lpg; off <<= 1) m = __hmax2(m, bits_h2(__shfl_xor_sync(kFull, h2_bits(m), off)));
    s16 = __float2half_rn(__fdiv_rn(__low2float(m), (float)qmax));
    z16 = __float2half_rn(0.0f);
    sc = __half2float(s16);
  } else {
    constexpr int levels = (1 << BITS) - 1;
    __half2 mn2 = pinf2, nx2 = pinf2;  // min of x and min of -x
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      __half2 lo = h[j], hi = __hneg2(h[j]);
      if (kout > 0) {
        const bool a = (om >> (2 * j)) & 1u, b2 = (om >> (2 * j + 1)) & 1u;
        lo = __halves2half2(a ? __low2half(pinf2) : __low2half(lo), b2 ? __low2half(pinf2) : __high2half(lo));
        hi = __halves2half2(a ? __low2half(pinf2) : __low2half(hi), b2 ? __low2half(pinf2) : __high2half(hi));
      }
      mn2 = __hmin2(mn2, lo);
      nx2 = __hmin2(nx2, hi);
    }
    __half2 pr = __hmin2(__halves2half2(__low2half(mn2), __low2half(nx2)),
                         __halves2half2(__high2half(mn2), __high2half(nx2)));
    for (int off = 1; off < lpg; off <<= 1) pr = __hmin2(pr, bits_h2(__shfl_xor_sync(kFull, h2_bits(pr), off)));
    float mn = __low2float(pr), mx = -__high2float(pr);
    if (mn > mx) {
      mn = 0.0f;
      mx = 0.0f;
    }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)levels));
    z16 = __float2half_rn(mn);
    sc = __half2float(s16);
    zc = __half2float(z16);
  }
  const float rc = rcp_approx(sc);
  // codes as bits of (code + 1.5*2^23)
  uint32_t cb[16];
  float maxd = 0.0f;
  const bool fast = __all_sync(kFull, sc > 0.0f);
  if (fast) {
    if (SYM) codes16_fast_sym<(1 << (BITS - 1)) - 1>(raw, rc, cb, maxd);
    else codes16_fast_asym<(1 << BITS) - 1>(raw, zc, rc, cb, maxd);
    if (kout > 0) {  // outlier slots store code 0
#pragma unroll
      for (int i = 0; i < 16; ++i) cb[i] = ((om >> i) & 1u) ? kMagicBits : cb[i];
    }
  }
  if (!fast) {  // a zero scale somewhere in the warp: the general path
    if (kout == 0) unpack16(raw, xf);
    int c[8];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float x8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x8[i] = xf[8 * half + i];
      const uint32_t dead = (om >> (8 * half)) & 0xFFu;
      if (SYM) codes8_sym<(1 << (BITS - 1)) - 1>(x8, sc, rc, dead, c);
      else codes8_asym<(1 << BITS) - 1>(x8, zc, sc, rc, dead, c);
#pragma unroll
      for (int i = 0; i < 8; ++i) cb[8 * half + i] = kMagicBits + (uint32_t)c[i];
    }
  } else if (__any_sync(kFull, maxd >= kNear)) {
    // a few quotients lie within 2^-12 of a half-integer: redo just those
    // with the IEEE quotient
    const uint16_t* hx = reinterpret_cast<const uint16_t*>(&raw[0]);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float d, qa;
      if (SYM) {
        constexpr float qm = (float)((1 << (BITS - 1)) - 1);
        d = __half2float(__ushort_as_half(hx[i]));
        qa = fmaxf(fminf(__fmul_rn(d, rc), qm), -qm);
      } else {
        d = add_h_f(hx[i], -zc);
        qa = fminf(__fmul_rn(d, rc), (float)((1 << BITS) - 1));
      }
      const float ci = (float)(int)(cb[i] - kMagicBits);
      if (!((om >> i) & 1u) && fabsf(__fsub_rn(qa, ci)) >= kNear) {
        int q = quot_exact(d, sc);
        q = SYM ? min(max(q, -((1 << (BITS - 1)) - 1)), (1 << (BITS - 1)) - 1) : min(q, (1 << BITS) - 1);
        cb[i] = kMagicBits + (uint32_t)q;
      }
    }
  }
  if (live && (l8 & (lpg - 1)) == 0) {
    const int g = l8 / lpg;
    const int per_row = kHeadDim / T.group;
    unsigned char* mb = T.meta + (int64_t)n * T.meta_sstride;
    if (SYM)
      reinterpret_cast<__half*>(mb)[(int64_t)row * per_row + g] = s16;
    else
      reinterpret_cast<__half2*>(mb)[(int64_t)row * per_row + g] = __halves2half2(s16, z16);
  }
  uint32_t* rowdst = T.codes + (int64_t)n * T.codes_sstride + (int64_t)row * Pack<BITS>::kWords;
  if (BITS == 4) {
    const uint2 w = make_uint2(pack_word<4>(cb), pack_word<4>(cb + 8));
    if (live) reinterpret_cast<uint2*>(rowdst)[l8] = w;
  } else if (BITS == 8) {
    uint4 w;
    if (SYM) {
      w.x = __byte_perm(__byte_perm(cb[0], cb[1], 0x0040u), __byte_perm(cb[2], cb[3], 0x0040u), 0x5410u);
      w.y = __byte_perm(__byte_perm(cb[4], cb[5], 0x0040u), __byte_perm(cb[6], cb[7], 0x0040u), 0x5410u);
      w.z = __byte_perm(__byte_perm(cb[8], cb[9], 0x0040u), __byte_perm(cb[10], cb[11], 0x0040u), 0x5410u);
      w.w = __byte_perm(__byte_perm(cb[12], cb[13], 0x0040u), __byte_perm(cb[14], cb[15], 0x0040u), 0x5410u);
    } else {
      w = make_uint4(pack_word<8>(cb), pack_word<8>(cb + 4), pack_word<8>(cb + 8), pack_word<8>(cb + 12));
    }
    if (live) reinterpret_cast<uint4*>(rowdst)[l8] = w;
  } else {
    // 3-bit: codes through shared memory, ten per word
    uint4 b;
    b.x = __byte_perm(__byte_perm(cb[0], cb[1], 0x0040u), __byte_perm(cb[2], cb[3], 0x0040u), 0x5410u);
    b.y = __byte_perm(__byte_perm(cb[4], cb[5], 0x0040u), __byte_perm(cb[6], cb[7], 0x0040u), 0x5410u);
    b.z = __byte_perm(__byte_perm(cb[8], cb[9], 0x0040u), __byte_perm(cb[10], cb[11], 0x0040u), 0x5410u);
    b.w = __byte_perm(__byte_perm(cb[12], cb[13], 0x0040u), __byte_perm(cb[14], cb[15], 0x0040u), 0x5410u);
    reinterpret_cast<uint4*>(scratch)[l8] = b;
    __syncwarp();
    for (int wi = l8; wi < Pack<3>::kWords; wi += 8) {
      uint32_t w = 0;
#pragma unroll
      for (int k = 0; k < 10; ++k) {
        const int ch = wi * 10 + k;
        if (ch < kHeadDim) w |= (uint32_t)scratch[ch] << (3 * k);
      }
      if (live) rowdst[wi] = w;
    }
    __syncwarp();
  }
}

// 64 per-token rows of one stream, staged in shared memory (`tile`, 256 B per
// row): warp w codes rows 8w .. 8w+7, four at a time (8 lanes per row).
template <int BITS, bool SYM>
__device__ __forceinline__ void rows_item(const uint4* __restrict__ tile, const TensorDev& T,
                                          int n, int row0, int nrows, int kout,
                                          uint8_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t* my = scratch + (warp * 4 + (lane >> 3)) * kHeadDim;
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int lr = warp * 8 + it * 4 + (lane >> 3);
    uint4 raw[2];
    raw[0] = tile[lr * 16 + 2 * (lane & 7)];
    raw[1] = tile[lr * 16 + 2 * (lane & 7) + 1];
    quant_row8<BITS, SYM>(raw, lr < nrows, T, n, row0 + lr, kout, lane, my);
  }
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
__device__ __forceinline__ void kblock_item(const uint4* __restrict__ tile, const TensorDev& K,
                                            int n, int blk, int kout, KBlockSmem<BITS, R>& sm) {
  constexpr int T = 16 * R;
  constexpr int levels = (1 << BITS) - 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int w16 = tid & 15, rg = tid >> 4;
  const int t0 = blk * T;
  uint4 raw[R];
#pragma unroll
  for (int i = 0; i < R; ++i) raw[i] = tile[(rg + 16 * i) * 16 + w16];
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
  // (min, -max) pairs per channel; the two row groups of a warp merge by one
  // shuffle, the eight warps through shared memory
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 plo = __halves2half2(__low2half(mn2[j]), __hneg(__low2half(mx2[j])));
    __half2 phi = __halves2half2(__high2half(mn2[j]), __hneg(__high2half(mx2[j])));
    plo = __hmin2(plo, bits_h2(__shfl_xor_sync(kFull, h2_bits(plo), 16)));
    phi = __hmin2(phi, bits_h2(__shfl_xor_sync(kFull, h2_bits(phi), 16)));
    if (lane < 16) {
      sm.mn[warp][(8 * w16 + 2 * j) >> 1] = plo;       // channel 8*w16 + 2j
      sm.mx[warp][(8 * w16 + 2 * j + 1) >> 1] = phi;   // channel 8*w16 + 2j + 1
    }
  }
  __syncthreads();
  if (tid < kHeadDim) {
    const int c = tid;
    // partials of channel c: even channels in sm.mn, odd in sm.mx (index c / 2)
    __half2 pr = (c & 1) ? sm.mx[0][c >> 1] : sm.mn[0][c >> 1];
#pragma unroll
    for (int w = 1; w < 8; ++w) pr = __hmin2(pr, (c & 1) ? sm.mx[w][c >> 1] : sm.mn[w][c >> 1]);
    float mn = __low2float(pr), mx = -__high2float(pr);
    if (mn > mx) {  // every member an outlier
      mn = 0.0f;
      mx = 0.0f;
    }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)levels));
    const __half z16 = __float2half_rn(mn);
    unsigned char* mb = K.meta + (int64_t)n * K.meta_sstride;
    reinterpret_cast<__half2*>(mb)[(int64_t)blk * kHeadDim + c] = __halves2half2(s16, z16);
    const float sv = __half2float(s16);
    sm.s[c] = sv;
    sm.z[c] = __half2float(z16);
    sm.r[c] = rcp_approx(sv);
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
  bool all_pos = true;
#pragma unroll
  for (int k = 0; k < 8; ++k) all_pos = all_pos && s[k] > 0.0f;
  const bool fast = __all_sync(kFull, all_pos);
  const uint64_t MG = f2_pack(kMagic, kMagic), NMG = f2_pack(-kMagic, -kMagic);
  const uint64_t NEG1 = f2_pack(-1.0f, -1.0f);
#pragma unroll
  for (int i = 0; i < R; ++i) {
    uint32_t cb[8];
    float maxd = 0.0f;
    if (fast) {
      const uint16_t* hx = reinterpret_cast<const uint16_t*>(&raw[i]);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float d0 = add_h_f(hx[2 * p], -z[2 * p]), d1 = add_h_f(hx[2 * p + 1], -z[2 * p + 1]);
        float q0, q1;
        f2_unpack(f2_mul(f2_pack(d0, d1), f2_pack(r[2 * p], r[2 * p + 1])), q0, q1);
        const uint64_t Q = f2_pack(fminf(q0, (float)levels), fminf(q1, (float)levels));
        const uint64_t CF = f2_add(Q, MG);
        float e0, e1, c0, c1;
        f2_unpack(f2_fma(f2_add(CF, NMG), NEG1, Q), e0, e1);
        f2_unpack(CF, c0, c1);
        maxd = fmaxf(maxd, fmaxf(fabsf(e0), fabsf(e1)));
        cb[2 * p] = __float_as_uint(c0);
        cb[2 * p + 1] = __float_as_uint(c1);
      }
      if (kout > 0) {
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) cb[k2] = ((om[i] >> k2) & 1u) ? kMagicBits : cb[k2];
      }
    }
    if (!fast) {
      float x[8];
      unpack8(raw[i], x);
      int c[8];
      codes8_kblock<levels>(x, z, s, r, om[i], c);
#pragma unroll
      for (int k = 0; k < 8; ++k) cb[k] = kMagicBits + (uint32_t)c[k];
    } else if (__any_sync(kFull, maxd >= kNear)) {
      const uint16_t* hx = reinterpret_cast<const uint16_t*>(&raw[i]);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float d = add_h_f(hx[k], -z[k]);
        const float qa = fminf(__fmul_rn(d, r[k]), (float)levels);
        const float ck = (float)(int)(cb[k] - kMagicBits);
        if (!((om[i] >> k) & 1u) && fabsf(__fsub_rn(qa, ck)) >= kNear)
          cb[k] = kMagicBits + (uint32_t)min(quot_exact(d, s[k]), levels);
      }
    }
    const int row = rg + 16 * i;
    if (BITS == 4) {
      kdst[(int64_t)row * Pack<4>::kWords + w16] = pack_word<4>(cb);
    } else if (BITS == 8) {
      reinterpret_cast<uint2*>(kdst + (int64_t)row * Pack<8>::kWords)[w16] =
          make_uint2(pack_word<8>(cb), pack_word<8>(cb + 4));
    } else {
      uint2 b;
      b.x = __byte_perm(__byte_perm(cb[0], cb[1], 0x0040u), __byte_perm(cb[2], cb[3], 0x0040u), 0x5410u);
      b.y = __byte_perm(__byte_perm(cb[4], cb[5], 0x0040u), __byte_perm(cb[6], cb[7], 0x0040u), 0x5410u);
      reinterpret_cast<uint2*>(sm.stage3 + row * kHeadDim)[w16] = b;
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
                                           int n, int t0, int seq_len, int in_rows) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src + ((int64_t)n * in_rows + t0) * kHeadDim);
  uint4* d4 = reinterpret_cast<uint4*>(K.resid + (int64_t)n * K.resid_sstride);
  const int count = (seq_len - t0) * (kHeadDim / 8);
  for (int i = threadIdx.x; i < count; i += kThreads) d4[i] = s4[i];
}

struct PrefillArgs {
  TensorDev k, v;
  const __half* ksrc;
  const __half* vsrc;
  int seq_len;
  int in_rows;  // input rows between streams (>= seq_len)
  int kout;
  int k_items;  // key items per stream: whole blocks (+1 residual copy) or 64-row chunks
  int k_nfull;  // whole per-channel key blocks per stream
  int v_items;  // 64-row value chunks per stream
  int n_streams;
  uint32_t* status;
};

template <int KB, int KMODE, int KR>
struct PfGeom {
  static constexpr int kTileRows = (KMODE == KVQ_ASYM_PER_CHANNEL && 16 * KR > 64) ? 16 * KR : 64;
  static constexpr size_t kStage = (size_t)kTileRows * kHeadDim * 2;
  static constexpr int kStages = kTileRows > 64 ? 2 : 3;  // two items in flight for 16 KB tiles
};

template <int KB, int KMODE, int KR, int VB, bool VSYM>
struct PrefillSmem {
  static constexpr size_t kKB = KMODE == KVQ_ASYM_PER_CHANNEL ? sizeof(KBlockSmem<KB, KR>) : 0;
  static constexpr size_t kRows = 32 * kHeadDim;
  static constexpr size_t kScratch = kKB > kRows ? kKB : kRows;
  static constexpr size_t bytes =
      PfGeom<KB, KMODE, KR>::kStages * (PfGeom<KB, KMODE, KR>::kStage + 8) + kScratch;
};

// Persistent prefill: CTA c takes work items c, c + gridDim.x, ... An item is
// a per-channel key block, a residual copy, or 64 per-token rows of one
// stream. Each item's fp16 input (one contiguous run of rows) is staged by a
// 1-D bulk copy into a 3-deep shared-memory ring, so two items' loads are in
// flight while one is coded.
template <int KB, int KMODE, int KR, int VB, bool VSYM>
__global__ void __launch_bounds__(kThreads, (KR >= 16 ? 1 : 3)) prefill_kernel(PrefillArgs a) {
  using G = PfGeom<KB, KMODE, KR>;
  using SM = PrefillSmem<KB, KMODE, KR, VB, VSYM>;
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kPfStages = G::kStages;
  unsigned char* scratch = smem + kPfStages * G::kStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(scratch + SM::kScratch);
  const int per_stream = a.k_items + a.v_items;
  const int total = a.n_streams * per_stream;
  const int tid = threadIdx.x;
  constexpr int T = 16 * KR;

  struct Item {
    int n, kind, idx, row0, nrows;  // kind: 0 key block, 1 residual copy, 2 key rows, 3 value rows
  };
  auto decode_item = [&](int it) {
    Item r;
    r.n = it / per_stream;
    const int j = it - r.n * per_stream;
    if (j < a.k_items) {
      if (KMODE == KVQ_ASYM_PER_CHANNEL) {
        r.kind = j < a.k_nfull ? 0 : 1;
        r.idx = j;
        r.row0 = j * T;
        r.nrows = r.kind == 0 ? T : 0;
      } else {
        r.kind = 2;
        r.idx = j;
        r.row0 = j * 64;
        r.nrows = min(64, a.seq_len - r.row0);
      }
    } else {
      r.kind = 3;
      r.idx = j - a.k_items;
      r.row0 = r.idx * 64;
      r.nrows = min(64, a.seq_len - r.row0);
    }
    return r;
  };
  auto issue = [&](int it, int s) {
    const Item r = decode_item(it);
    const __half* src = (r.kind == 3) ? a.vsrc : a.ksrc;
    const uint32_t bytes = (uint32_t)r.nrows * kHeadDim * 2;
    mbar_arrive_expect_tx(&bars[s], bytes);
    if (bytes)
      bulk_g2s(smem + (size_t)s * G::kStage, src + ((int64_t)r.n * a.in_rows + r.row0) * kHeadDim,
               bytes, &bars[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();
  const int first = blockIdx.x, stride = gridDim.x;
  if (tid == 0)
    for (int s = 0; s < kPfStages && first + s * stride < total; ++s) issue(first + s * stride, s);

  int k = 0;
  for (int it = first; it < total; it += stride, ++k) {
    const int s = k % kPfStages;
    const uint32_t par = (uint32_t)(k / kPfStages) & 1u;
    const bool ok = mbar_wait_bounded(&bars[s], par);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        raise_status(a.status, kStatusTimeout);
        for (int kk = k; kk < k + kPfStages && first + kk * stride < total; ++kk)
          (void)mbar_wait_bounded(&bars[kk % kPfStages], (uint32_t)(kk / kPfStages) & 1u);
      }
      __syncthreads();
      return;
    }
    const Item r = decode_item(it);
    const uint4* tile = reinterpret_cast<const uint4*>(smem + (size_t)s * G::kStage);
    if (r.kind == 0) {
      if (KMODE == KVQ_ASYM_PER_CHANNEL)
        kblock_item<KB, KR>(tile, a.k, r.n, r.idx, a.kout,
                            *reinterpret_cast<KBlockSmem<KB, KR>*>(scratch));
    } else if (r.kind == 1) {
      resid_copy(a.k, a.ksrc, r.n, a.k_nfull * T, a.seq_len, a.in_rows);
    } else if (r.kind == 2) {
      rows_item<KB, KMODE == KVQ_SYM_PER_TOKEN>(tile, a.k, r.n, r.row0, r.nrows, a.kout, scratch);
    } else {
      rows_item<VB, VSYM>(tile, a.v, r.n, r.row0, r.nrows, a.kout, scratch);
    }
    __syncthreads();
    const int nxt = it + kPfStages * stride;
    if (tid == 0 && nxt < total) {
      fence_proxy_async_smem();
      issue(nxt, s);
    }
  }
}

template <int KB, int KMODE, int KR, int VB, bool VSYM>
cudaError_t launch_prefill_t(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                             cudaStream_t st) {
  using SM = PrefillSmem<KB, KMODE, KR, VB, VSYM>;
  auto kern = prefill_kernel<KB, KMODE, KR, VB, VSYM>;
  static SmemAttr attr;
  static std::atomic<int> occ_cached{0};  // resident CTAs per SM, computed once
  {
    const cudaError_t e = attr.ensure(kern, SM::bytes);
    if (e != cudaSuccess) return e;
  }
  int occ = occ_cached.load(std::memory_order_relaxed);
  if (occ == 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, SM::bytes);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    occ_cached.store(occ, std::memory_order_relaxed);
  }
  PrefillArgs a;
  a.k = L.k;
  a.v = L.v;
  a.ksrc = k;
  a.vsrc = v;
  a.seq_len = seq_len;
  a.in_rows = L.in_rows > 0 ? L.in_rows : seq_len;
  a.kout = L.outliers;
  a.n_streams = L.n_streams;
  a.status = L.status;
  a.v_items = (seq_len + 63) / 64;
  if (KMODE == KVQ_ASYM_PER_CHANNEL) {
    a.k_nfull = seq_len / L.k.group;
    a.k_items = a.k_nfull + (seq_len % L.k.group ? 1 : 0);
  } else {
    a.k_nfull = 0;
    a.k_items = a.v_items;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t total = (int64_t)L.n_streams * (a.k_items + a.v_items);
  if (total > 0x7fffffff) return cudaErrorInvalidValue;  // item index is 32-bit
  const int64_t slots = (int64_t)(sms > 0 ? sms : 1) * occ;
  const int grid = (int)(total < slots ? total : slots);
  kern<<<grid, kThreads, SM::bytes, st>>>(a);
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
