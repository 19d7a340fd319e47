// Prefill quantize (3-, 4- or 8-bit codes; per-token rows and per-channel key
// blocks of 64 or 128 tokens), with or without the dense-and-sparse outlier
// split (template parameter OUTL).
//
// One launch quantizes a whole prompt of one layer. CTAs of four warps are
// persistent and take work items in a fixed order: a per-channel key block
// of T tokens, the copy of the key residual (the last S mod T tokens, kept in
// fp16), or a chunk of per-token rows. Each item's fp16 rows (one contiguous
// run in HBM) are staged by a 1-D bulk copy into a ring of shared-memory
// stages. Warps work on their own rows and release a stage through a
// counter: the last warp done with a stage refills it, so warps never wait
// for one another except at the two points of a key block where the
// per-channel statistics of the four warps' rows are merged.
//
// Codec (TurboQuant 3-bit KV quantization page, dpshk.com/news/6341316,
// §3.1; NIAH q8_0 write-up, cf-1.com/news/5482713, §1.2): group minimum and
// maximum (or absolute maximum), scale = (max - min) / (2^b - 1) (or
// absmax / 127) in fp32 and rounded to fp16, zero point = the minimum in
// fp16, code = clamp(rne(RN32(x - z) / s)) with the IEEE quotient.
//
// How the codes are formed without a division per element: with
// R_lo < 1/s < R_hi a tight bracket of the reciprocal (relative width 2^-20),
// one fused multiply-add per bound gives rne(d * R_lo) and rne(d * R_hi) for
// the exact products. rne is monotone and RN32(d / s) lies strictly between
// the two products, so where they agree the agreed integer is the code.
// Where they differ (the quotient is an exact tie k + 1/2, or lies within
// 2^-20 of one) the code is settled exactly from the residual
// d - (k + 1/2) s, formed without rounding by one fused multiply-add. With a
// normal fp16 scale no code can exceed the range, so no clamp is needed; a
// subnormal nonzero scale takes a per-element IEEE-division path instead.
#pragma once

#include "common.cuh"

namespace kvq {
namespace pfx {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: x + kMagic holds rne(x) in its low bits
constexpr uint32_t kMagicBits = 0x4B400000u;
constexpr float kMinNormal16 = 0x1p-14f;
constexpr int kKeyBarrier = 1;  // named barrier of the four warps at a key block

// x + c in fp32 with x an fp16 value (one mixed-precision instruction; the
// same value as widening x and adding in fp32).
__device__ __forceinline__ float add_h_f(uint16_t xh, float c) {
  float r;
  asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(r) : "h"(xh), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t bfi(uint32_t field, uint32_t base, uint32_t pos, uint32_t len) {
  uint32_t r;
  asm("bfi.b32 %0, %1, %2, %3, %4;" : "=r"(r) : "r"(field), "r"(base), "r"(pos), "r"(len));
  return r;
}

// Barrier of the NTH threads of the CTA that also ANDs a predicate over them.
template <int NTH>
__device__ __forceinline__ bool key_barrier_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kKeyBarrier), "n"(NTH)
      : "memory");
  return r != 0;
}

// RN32(a / L) for 0 <= a <= 2^17 and L in {3, 7, 15, 127, 255}: the product
// a * RN(1/L) corrected once from its exact remainder (a fused multiply-add),
// the correction step of Markstein's division method. For these divisors the
// result equals the IEEE quotient for every fp32 a in that range (checked by
// enumerating all of them).
template <int L>
__device__ __forceinline__ float div_levels(float a) {
  constexpr float c = 1.0f / (float)L;
  const float y = __fmul_rn(a, c);
  const float r = __fmaf_rn(-y, (float)L, a);
  return __fmaf_rn(r, c, y);
}

// Bracket of 1/s for a normal fp32 s > 0: the approximate reciprocal after
// one Newton step (within one ulp of 1/s), widened by 2^-21 each way.
__device__ __forceinline__ void recip_bracket(float s, float& rlo, float& rhi) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  const float e = __fmaf_rn(-s, r, 1.0f);
  r = __fmaf_rn(e, r, r);
  rlo = __fmul_rn(r, 1.0f - 0x1p-21f);
  rhi = __fmul_rn(r, 1.0f + 0x1p-21f);
}

// Bracket for a stored scale: a zero scale gives a zero bracket (every code
// 0, as the codec defines); *slow is set for a subnormal nonzero scale.
__device__ __forceinline__ void scale_bracket(float s, float& rlo, float& rhi, bool& slow) {
  if (s > 0.0f) {
    recip_bracket(s, rlo, rhi);
  } else {
    rlo = 0.0f;
    rhi = 0.0f;
  }
  slow = s > 0.0f && s < kMinNormal16;
}

// rne(d * r) for the exact product, as an integer (|d * r| < 2^22).
__device__ __forceinline__ int rne_prod(float d, float r) {
  return (int)(__float_as_uint(__fmaf_rn(d, r, kMagic)) - kMagicBits);
}

// Exact rne(RN32(d / s)) for d >= 0 and a normal s, given k with d / s
// strictly inside (k, k + 1) and near m = k + 1/2. e = d - m*s is exact
// (m*s has at most 20 significant bits and lies within 2^-20 of d), so
// RN32(d / s) lies above m exactly when e > s * ulp(m) / 2, below m exactly
// when e < -s * ulp(m-) / 2 (ulp(m-) = the spacing below m, half of ulp(m)
// only at m = 1/2), and equals m otherwise; a quotient of exactly m rounds
// to the even one of k and k + 1.
__device__ __forceinline__ int resolve_code(float d, float s, int k) {
  const float m = (float)k + 0.5f;
  const float e = __fmaf_rn(-m, s, d);
  const float h = __uint_as_float((__float_as_uint(m) & 0x7F800000u) - (24u << 23));  // ulp(m) / 2
  const float up = __fmul_rn(s, h);
  const float dn = k == 0 ? __fmul_rn(up, 0.5f) : up;
  if (e > up) return k + 1;
  if (e < -dn) return k;
  return k + (k & 1);
}

// Eight codes held as bits of (code + 1.5 * 2^23) packed into one word of
// 4-bit fields (code i at bits 4i).
__device__ __forceinline__ uint32_t pack8x4(const uint32_t (&c)[8]) {
  const uint32_t t0 = c[0] + (c[1] << 4), t1 = c[2] + (c[3] << 4);
  const uint32_t t2 = c[4] + (c[5] << 4), t3 = c[6] + (c[7] << 4);
  return __byte_perm(__byte_perm(t0, t1, 0x0040u), __byte_perm(t2, t3, 0x0040u), 0x5410u);
}

// Four codes (low bytes, two's complement for signed codes) into one word.
__device__ __forceinline__ uint32_t pack4x8(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  return __byte_perm(__byte_perm(c0, c1, 0x0040u), __byte_perm(c2, c3, 0x0040u), 0x5410u);
}

// Eight codes of eight consecutive channels (one 16-byte chunk of a row):
// wa = rne(d * R_lo) packed, wb = rne(d * R_hi) packed, with d = x - z
// (asymmetric) or x (symmetric). Per-element z / R arrays (per-channel keys)
// or broadcast values (per-token groups) both fit: NZ, RL, RH are indexable.
template <int BITS, bool SYM, class Z, class RLo, class RHi>
__device__ __forceinline__ void chunk_codes(const uint4& raw, const Z& nz, const RLo& rl,
                                            const RHi& rh, uint32_t (&wa)[BITS / 4],
                                            uint32_t (&wb)[BITS / 4]) {
  const uint16_t* hx = reinterpret_cast<const uint16_t*>(&raw);
  const uint64_t MG = f2_pack(kMagic, kMagic);
  uint32_t ca[8], cb[8];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float d0 = SYM ? add_h_f(hx[2 * p], 0.0f) : add_h_f(hx[2 * p], nz[2 * p]);
    const float d1 = SYM ? add_h_f(hx[2 * p + 1], 0.0f) : add_h_f(hx[2 * p + 1], nz[2 * p + 1]);
    const uint64_t D = f2_pack(d0, d1);
    float a0, a1, b0, b1;
    f2_unpack(f2_fma(D, f2_pack(rl[2 * p], rl[2 * p + 1]), MG), a0, a1);
    f2_unpack(f2_fma(D, f2_pack(rh[2 * p], rh[2 * p + 1]), MG), b0, b1);
    ca[2 * p] = __float_as_uint(a0);
    ca[2 * p + 1] = __float_as_uint(a1);
    cb[2 * p] = __float_as_uint(b0);
    cb[2 * p + 1] = __float_as_uint(b1);
  }
  if (BITS == 4) {
    wa[0] = pack8x4(ca);
    wb[0] = pack8x4(cb);
  } else {
    wa[0] = pack4x8(ca[0], ca[1], ca[2], ca[3]);
    wa[BITS / 4 - 1] = pack4x8(ca[4], ca[5], ca[6], ca[7]);
    wb[0] = pack4x8(cb[0], cb[1], cb[2], cb[3]);
    wb[BITS / 4 - 1] = pack4x8(cb[4], cb[5], cb[6], cb[7]);
  }
}

template <class T>
struct Bcast {
  T v;
  __device__ __forceinline__ T operator[](int) const { return v; }
};

// Settles the fields where wa and wb differ, in place in wa. x_at(i) gives
// the fp16 bits of element i of the chunk; the element's z, s and R_lo come
// from nz_at / s_at / rl_at.
template <int BITS, bool SYM, class XAt, class ZAt, class SAt, class RAt>
__device__ __forceinline__ void settle_chunk(uint32_t (&wa)[BITS / 4], const uint32_t (&wb)[BITS / 4],
                                             XAt x_at, ZAt nz_at, SAt s_at, RAt rl_at) {
  constexpr int kPer = 32 / BITS;
  constexpr uint32_t kMask = (1u << BITS) - 1u;
#pragma unroll
  for (int j = 0; j < BITS / 4; ++j) {
    uint32_t f = wa[j] ^ wb[j];
    while (f) {
      const int fld = (__ffs(f) - 1) / BITS;
      const int i = j * kPer + fld;
      const uint16_t xh = x_at(i);
      int code;
      if (SYM) {
        const float x = add_h_f(xh, 0.0f);
        const float ad = fabsf(x);
        const int c = resolve_code(ad, s_at(i), rne_prod(ad, rl_at(i)));
        code = x < 0.0f ? -c : c;
      } else {
        const float d = add_h_f(xh, nz_at(i));
        code = resolve_code(d, s_at(i), rne_prod(d, rl_at(i)));
      }
      wa[j] = bfi((uint32_t)code, wa[j], (uint32_t)(fld * BITS), BITS);
      f &= ~(kMask << (fld * BITS));
    }
  }
}

// Codes of one chunk by the IEEE quotient with the clamp (a subnormal
// nonzero scale somewhere in the warp's rows).
template <int BITS, bool SYM, int LEV, class XAt, class ZAt, class SAt>
__device__ __forceinline__ void slow_chunk(uint32_t (&wa)[BITS / 4], XAt x_at, ZAt nz_at, SAt s_at) {
  constexpr int kPer = 32 / BITS;
  constexpr int kLev = LEV;
#pragma unroll
  for (int j = 0; j < BITS / 4; ++j) {
    uint32_t w = 0;
    for (int f = 0; f < kPer; ++f) {
      const int i = j * kPer + f;
      const float s = s_at(i);
      int code = 0;
      if (s > 0.0f) {
        const float d = add_h_f(x_at(i), SYM ? 0.0f : nz_at(i));
        code = __float2int_rn(__fdiv_rn(d, s));
        code = SYM ? min(max(code, -kLev), kLev) : min(max(code, 0), kLev);
      }
      w = bfi((uint32_t)code, w, (uint32_t)(f * BITS), BITS);
    }
    wa[j] = w;
  }
}

// ---------------------------------------------------------------------------
// Outliers (KVQuant page, cf-1.com/news/2306543, §2.2 item 3): the k largest
// |x| of a (token, head) row, ties to the lower channel, stored as CSR sorted
// by channel; their slots are left out of the group statistics and get code
// 0.
//
// Selection works on packed fp16 magnitudes (sign bits cleared; for
// non-negative halves the fp16 order is the order of |x|). A threshold t
// (the k-th largest |x| of the row, see kth_magnitude) marks the slots with
// |x| >= t; they are the outliers exactly when there are k of them.
// Otherwise a magnitude repeats at the threshold (a tie), and the warp redoes
// the selection with unique keys (|x| bits << 16) | (128 - channel): round r
// takes the largest key below the one round r-1 took.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t hmax2_bits(uint32_t a, uint32_t b) {
  const __half2 r = __hmax2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t ge_mask(uint32_t a, uint32_t b) {
  return __hge2_mask(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
}
__device__ __forceinline__ uint32_t lt_mask(uint32_t a, uint32_t b) {
  return __hlt2_mask(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
}

// Maximum over NP packed pairs of this lane and the NL lanes of its row
// (xor 1 .. NL/2), in both halves of the result.
template <int NP, int NL>
__device__ __forceinline__ uint32_t row_max2(const uint32_t (&v)[NP]) {
  uint32_t m = v[0];
#pragma unroll
  for (int p = 1; p < NP; ++p) m = hmax2_bits(m, v[p]);
  m = hmax2_bits(m, __byte_perm(m, 0u, 0x1032u));
#pragma unroll
  for (int off = 1; off < NL; off <<= 1) m = hmax2_bits(m, __shfl_xor_sync(kFull, m, off));
  return m;
}

__device__ __forceinline__ uint32_t hmin2_bits(uint32_t a, uint32_t b) {
  const __half2 r = __hmin2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// The second largest magnitude of the row, counted with multiplicity (equal
// to the largest when that occurs twice): per half a running (largest,
// second) pair, then pairs merge across the halves and the NL lanes.
template <int NP, int NL>
__device__ __forceinline__ uint32_t row_second2(const uint32_t (&a)[NP]) {
  uint32_t m1 = a[0], m2 = 0u;
#pragma unroll
  for (int p = 1; p < NP; ++p) {
    m2 = hmax2_bits(m2, hmin2_bits(m1, a[p]));
    m1 = hmax2_bits(m1, a[p]);
  }
  auto merge = [](uint32_t& x1, uint32_t& x2, uint32_t y1, uint32_t y2) {
    x2 = hmax2_bits(hmin2_bits(x1, y1), hmax2_bits(x2, y2));
    x1 = hmax2_bits(x1, y1);
  };
  merge(m1, m2, __byte_perm(m1, 0u, 0x1032u), __byte_perm(m2, 0u, 0x1032u));
#pragma unroll
  for (int off = 1; off < NL; off <<= 1) {
    const uint32_t y1 = __shfl_xor_sync(kFull, m1, off), y2 = __shfl_xor_sync(kFull, m2, off);
    merge(m1, m2, y1, y2);
  }
  return m2;
}

// The outlier threshold of the row from the magnitudes a of this lane's
// pairs: k = 1 the largest, k = 2 the second largest with multiplicity,
// k > 2 the k-th largest distinct magnitude M_k. The slots at or above it
// are the outliers when they number k.
template <int NP, int NL>
__device__ __forceinline__ uint32_t kth_magnitude(const uint32_t (&a)[NP], int kout) {
  if (kout == 2) return row_second2<NP, NL>(a);
  uint32_t m = row_max2<NP, NL>(a);
  for (int r = 1; r < kout; ++r) {
    uint32_t b[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) b[p] = a[p] & lt_mask(a[p], m);
    m = row_max2<NP, NL>(b);
  }
  return m;
}

// Bits of NP pair masks (0xFFFF per selected half): element 2p <- bit 2p,
// element 2p + 1 <- bit 2p + 1.
template <int NP>
__device__ __forceinline__ uint32_t mask_bits(const uint32_t (&mk)[NP]) {
  uint32_t b = 0;
#pragma unroll
  for (int p = 0; p < NP; ++p) b |= (mk[p] & 0x00010001u) << (2 * p);
  return (b | (b >> 15)) & ((1u << (2 * NP)) - 1u);
}

// Pair masks of four pairs from eight element bits (the inverse of
// mask_bits): bits 2p and 2p + 1 are moved to the sign bits of bytes 0 and 1
// and replicated by a sign-extending byte permute.
__device__ __forceinline__ void expand_mask4(uint32_t bits, uint32_t (&mk)[4]) {
  const uint32_t t = bits | (bits << 7);  // bit i (i < 8) at i and i + 7
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    // selector nibbles 8, 8, 9, 9: bytes 0 and 1 of the result take the sign
    // of source byte 0, bytes 2 and 3 the sign of source byte 1
    asm("prmt.b32 %0, %1, 0, 0x9988;" : "=r"(mk[p]) : "r"(t << (7 - 2 * p)));
  }
}

__device__ __forceinline__ uint32_t outlier_key(uint16_t xh, int ch) {
  return ((uint32_t)(xh & 0x7FFFu) << 16) | (uint32_t)(kHeadDim - ch);
}

// k rounds of the keyed max over a group of NL lanes (xor 1 .. NL/2);
// returns the key of the k-th largest |x| of the row.
template <int NL, int NE>
__device__ __forceinline__ uint32_t kth_key(const uint32_t (&key)[NE], int kout) {
  uint32_t thr = 0xFFFFFFFFu;
  for (int r = 0; r < kout; ++r) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < NE; ++i) m = max(m, key[i] < thr ? key[i] : 0u);
#pragma unroll
    for (int off = 1; off < NL; off <<= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
    thr = m;
  }
  return thr;
}

// The tie path, kept out of line (it runs for a few rows in a thousand): the
// outlier bits of this lane's chunks by unique keys. Sixteen channels
// (chunks c0, c1, eight lanes a row): returns bits of c0 | bits of c1 << 8.
static __device__ __noinline__ uint32_t exact_bits16(uint4 raw0, uint4 raw1, int c0, int c1, int kout) {
  const uint16_t* hx0 = reinterpret_cast<const uint16_t*>(&raw0);
  const uint16_t* hx1 = reinterpret_cast<const uint16_t*>(&raw1);
  uint32_t key[16];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    key[e] = outlier_key(hx0[e], 8 * c0 + e);
    key[8 + e] = outlier_key(hx1[e], 8 * c1 + e);
  }
  const uint32_t kw = kth_key<8, 16>(key, kout);
  uint32_t om = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e) om |= (key[e] >= kw ? 1u : 0u) << e;
  return om;
}

// Eight channels (chunk o, sixteen lanes a row).
static __device__ __noinline__ uint32_t exact_bits8(uint4 raw, int o, int kout) {
  const uint16_t* hx = reinterpret_cast<const uint16_t*>(&raw);
  uint32_t key[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) key[e] = outlier_key(hx[e], 8 * o + e);
  const uint32_t kw = kth_key<16, 8>(key, kout);
  uint32_t om = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) om |= (key[e] >= kw ? 1u : 0u) << e;
  return om;
}

// CSR entries of this lane's outliers (om: bit i <- channel ch0 + i, in
// channel order) at positions first, first + 1, ... of the row; xs holds the
// row's fp16 values.
__device__ __forceinline__ void write_lane_csr(const TensorDev& T, int n, int row, int kout,
                                               uint32_t om, int ch0, int first,
                                               const uint16_t* xs) {
  const int64_t base = (int64_t)n * T.out_sstride + (int64_t)row * kout + first;
  int i = 0;
  for (uint32_t m = om; m; m &= m - 1, ++i) {
    const int c = ch0 + __ffs(m) - 1;
    T.col[base + i] = (uint16_t)c;
    T.val[base + i] = __ushort_as_half(xs[c]);
  }
}

__device__ __forceinline__ void write_rowptr(const TensorDev& T, int n, int row, int kout) {
  int32_t* rp = T.rowptr + (int64_t)n * T.rowptr_sstride;
  rp[row + 1] = (row + 1) * kout;
  if (row == 0) rp[0] = 0;
}

// Exclusive prefix sum of v over the NL lanes of a row, and the row total.
template <int NL>
__device__ __forceinline__ int row_scan(int v, int li, int& total) {
  int s = v;
#pragma unroll
  for (int d = 1; d < NL; d <<= 1) {
    const int t = __shfl_up_sync(kFull, s, d, NL);
    if (li >= d) s += t;
  }
  total = __shfl_sync(kFull, s, NL - 1, NL);
  return s - v;
}

// Clears field i (of PB bits) of an eight-code chunk packed in w.
template <int PB>
__device__ __forceinline__ void clear_field(uint32_t (&w)[PB / 4], int i) {
  if (PB == 4) {
    w[0] = bfi(0u, w[0], (uint32_t)(4 * i), 4);
  } else if (i < 4) {
    w[0] = bfi(0u, w[0], (uint32_t)(8 * i), 8);
  } else {
    w[PB / 4 - 1] = bfi(0u, w[PB / 4 - 1], (uint32_t)(8 * (i - 4)), 8);
  }
}

// Ten-per-word packing in registers. comb4: the four one-byte codes of a
// word as four 3-bit fields (12 bits). A lane holding the codes of channels
// c0 .. c0 + k - 1 contributes 3k bits at bit 3 c0 of the row's 3-bit
// stream; word w of the row is the stream's bits 30 w .. 30 w + 29, taken
// from at most two neighbouring lanes by shuffles.
__device__ __forceinline__ uint32_t comb4(uint32_t x) {
  return (x & 0x7u) | ((x >> 5) & 0x38u) | ((x >> 10) & 0x1C0u) | ((x >> 15) & 0xE00u);
}

// ---------------------------------------------------------------------------
// Per-token rows. A warp owns kRowsPerItem / 4 rows of the item; eight lanes
// code one row (16 channels each: 16-byte chunks 2q and 2q + 1, read in an
// order that keeps the four rows of a warp instruction on distinct banks).
// ---------------------------------------------------------------------------
template <int BITS, bool SYM, int RPW, bool OUTL>
__device__ __forceinline__ void rows_warp(const unsigned char* tile, const TensorDev& T, int n,
                                          int row0, int nrows, int warp, int lane,
                                          unsigned char* rowbuf, int kout) {
  constexpr int kLev = SYM ? (1 << (BITS - 1)) - 1 : (1 << BITS) - 1;
  constexpr int kWords = Pack<BITS>::kWords;
  constexpr int PB = BITS == 3 ? 8 : BITS;  // field width while coding (3-bit codes go one per byte)
  const int q = lane & 7, rr = lane >> 3;
  const int sw = q >> 2;
  const int lpg = T.group >> 4;  // lanes per group (groups of 16 .. 128 channels)
  const int per_row = kHeadDim / T.group;
#pragma unroll(OUTL ? 1 : 2)  // with outliers the body is long: code size matters more
  for (int it = 0; it < RPW / 4; ++it) {
    const int lr = warp * RPW + it * 4 + rr;
    const bool live = lr < nrows;
    const uint4* rowp = reinterpret_cast<const uint4*>(tile + (size_t)lr * (kHeadDim * 2));
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(rowp);
    const int c0 = 2 * q + sw, c1 = 2 * q + 1 - sw;  // chunk indices of raw0, raw1
    // outliers: om0 / om1 bit e <- element e of chunk c0 / c1; mk[p] the
    // mask of pair p (pairs 0-3 of raw0, 4-7 of raw1); first: entries of
    // the row before this lane's
    uint32_t om0 = 0, om1 = 0, mk[8];
    int first = 0;
    __half s16, z16;
    uint32_t wa0[PB / 4], wa1[PB / 4];
    // Pass 0 selects by threshold; a tie in any row of the warp (found
    // only after the codes, so that the count's shuffles overlap them)
    // sends the warp through pass 1 with unique keys.
    for (int pass = 0;; ++pass) {
      uint4 raw0 = rowp[c0], raw1 = rowp[c1];
      int total = kout;
      if (OUTL) {
        const uint32_t wv[8] = {raw0.x, raw0.y, raw0.z, raw0.w, raw1.x, raw1.y, raw1.z, raw1.w};
        if (pass == 0) {
          uint32_t a[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) a[p] = wv[p] & 0x7FFF7FFFu;
          const uint32_t th = kth_magnitude<8, 8>(a, kout);
#pragma unroll
          for (int p = 0; p < 8; ++p) mk[p] = ge_mask(a[p], th);
          om0 = mask_bits<4>(*reinterpret_cast<const uint32_t(*)[4]>(&mk[0]));
          om1 = mask_bits<4>(*reinterpret_cast<const uint32_t(*)[4]>(&mk[4]));
        } else {
          const uint32_t ob = exact_bits16(raw0, raw1, c0, c1, kout);
          om0 = ob & 0xFFu;
          om1 = ob >> 8;
          expand_mask4(om0, *reinterpret_cast<uint32_t(*)[4]>(&mk[0]));
          expand_mask4(om1, *reinterpret_cast<uint32_t(*)[4]>(&mk[4]));
        }
        first = row_scan<8>(__popc(om0) + __popc(om1), q, total);
        if (SYM) {
          // an outlier slot reads +0: the absolute maximum of the rest
          // stays, and the slot codes 0
          raw0 = make_uint4(wv[0] & ~mk[0], wv[1] & ~mk[1], wv[2] & ~mk[2], wv[3] & ~mk[3]);
          raw1 = make_uint4(wv[4] & ~mk[4], wv[5] & ~mk[5], wv[6] & ~mk[6], wv[7] & ~mk[7]);
        }
      }
      const __half2* h0 = reinterpret_cast<const __half2*>(&raw0);
      const __half2* h1 = reinterpret_cast<const __half2*>(&raw1);
      float nz = 0.0f, rlo, rhi;
      bool slow;
      if (SYM) {
        __half2 m = __habs2(h0[0]);
#pragma unroll
        for (int j = 1; j < 4; ++j) m = __hmax2(m, __habs2(h0[j]));
#pragma unroll
        for (int j = 0; j < 4; ++j) m = __hmax2(m, __habs2(h1[j]));
        m = __hmax2(m, __lowhigh2highlow(m));
        for (int off = 1; off < lpg; off <<= 1) {
          const uint32_t o = __shfl_xor_sync(kFull, *reinterpret_cast<uint32_t*>(&m), off);
          m = __hmax2(m, *reinterpret_cast<const __half2*>(&o));
        }
        const float am = __low2float(m);  // |x| >= 0, canonical +0
        s16 = __float2half_rn(div_levels<kLev>(am));
        z16 = __ushort_as_half(0);
      } else {
        __half2 vn[8], vx[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const __half2 h = p < 4 ? h0[p] : h1[p - 4];
          if (OUTL) {
            // outlier slots read +inf for the minimum and -inf for the maximum
            const uint32_t w = *reinterpret_cast<const uint32_t*>(&h);
            const uint32_t wn = (w & ~mk[p]) | (0x7C007C00u & mk[p]);
            const uint32_t wx = (w & ~mk[p]) | (0xFC00FC00u & mk[p]);
            vn[p] = *reinterpret_cast<const __half2*>(&wn);
            vx[p] = *reinterpret_cast<const __half2*>(&wx);
          } else {
            vn[p] = h;
            vx[p] = h;
          }
        }
        __half2 mn = __hmin2(vn[0], vn[1]), mx = __hmax2(vx[0], vx[1]);
        mn = __hmin2(mn, __hmin2(vn[2], vn[3]));
        mx = __hmax2(mx, __hmax2(vx[2], vx[3]));
        mn = __hmin2(mn, __hmin2(__hmin2(vn[4], vn[5]), __hmin2(vn[6], vn[7])));
        mx = __hmax2(mx, __hmax2(__hmax2(vx[4], vx[5]), __hmax2(vx[6], vx[7])));
        const __half2 nmx = __hneg2(mx);
        __half2 pr = __hmin2(__lows2half2(mn, nmx), __highs2half2(mn, nmx));  // (min, -max)
        for (int off = 1; off < lpg; off <<= 1) {
          const uint32_t o = __shfl_xor_sync(kFull, *reinterpret_cast<uint32_t*>(&pr), off);
          pr = __hmin2(pr, *reinterpret_cast<const __half2*>(&o));
        }
        // zero extremes are taken as +0
        const float mnv = __fadd_rn(__low2float(pr), 0.0f);
        const float mxv = __fadd_rn(-__high2float(pr), 0.0f);
        s16 = __float2half_rn(div_levels<kLev>(__fsub_rn(mxv, mnv)));
        z16 = __float2half_rn(mnv);
        nz = -mnv;
        if (OUTL) {
          // an outlier slot codes the zero point: d = 0, code 0
          const uint32_t z2 = (uint32_t)__half_as_ushort(z16) * 0x10001u;
          uint32_t* r0 = reinterpret_cast<uint32_t*>(&raw0);
          uint32_t* r1 = reinterpret_cast<uint32_t*>(&raw1);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            r0[p] = (r0[p] & ~mk[p]) | (z2 & mk[p]);
            r1[p] = (r1[p] & ~mk[4 + p]) | (z2 & mk[4 + p]);
          }
        }
      }
      const float s = __half2float(s16);
      scale_bracket(s, rlo, rhi, slow);
      uint32_t wb0[PB / 4], wb1[PB / 4];
      const Bcast<float> NZ{nz}, RL{rlo};
      auto xat0 = [&](int i) { return xs[8 * c0 + i]; };
      auto xat1 = [&](int i) { return xs[8 * c1 + i]; };
      auto zat = [&](int) { return nz; };
      auto sat = [&](int) { return s; };
      auto rat = [&](int) { return rlo; };
      if (!__any_sync(kFull, slow)) {
        chunk_codes<PB, SYM>(raw0, NZ, RL, Bcast<float>{rhi}, wa0, wb0);
        chunk_codes<PB, SYM>(raw1, NZ, RL, Bcast<float>{rhi}, wa1, wb1);
        uint32_t diff = 0;
#pragma unroll
        for (int j = 0; j < PB / 4; ++j) diff |= (wa0[j] ^ wb0[j]) | (wa1[j] ^ wb1[j]);
        if (__any_sync(kFull, diff != 0)) {
          settle_chunk<PB, SYM>(wa0, wb0, xat0, zat, sat, rat);
          settle_chunk<PB, SYM>(wa1, wb1, xat1, zat, sat, rat);
        }
      } else {
        slow_chunk<PB, SYM, kLev>(wa0, xat0, zat, sat);
        slow_chunk<PB, SYM, kLev>(wa1, xat1, zat, sat);
        if (OUTL) {  // the IEEE path coded the outliers' own values
          for (uint32_t m = om0; m; m &= m - 1) clear_field<PB>(wa0, __ffs(m) - 1);
          for (uint32_t m = om1; m; m &= m - 1) clear_field<PB>(wa1, __ffs(m) - 1);
        }
      }
      if (!OUTL || pass > 0 || !__any_sync(kFull, total != kout)) break;
    }
    if (live && (q & (lpg - 1)) == 0) {
      unsigned char* mb = T.meta + (int64_t)n * T.meta_sstride;
      const int64_t at = (int64_t)(row0 + lr) * per_row + q / lpg;
      if (SYM)
        reinterpret_cast<__half*>(mb)[at] = s16;
      else
        reinterpret_cast<__half2*>(mb)[at] = __halves2half2(s16, z16);
    }
    if (OUTL && live) {
      const uint32_t om16 = sw ? (om1 | (om0 << 8)) : (om0 | (om1 << 8));  // channel order
      write_lane_csr(T, n, row0 + lr, kout, om16, 16 * q, first, xs);
      if (q == 0) write_rowptr(T, n, row0 + lr, kout);
    }
    if (BITS == 3) {
      // ten codes per word: the lane's 16 codes (channels 16 q ..) are 48 bits
      // at bit 48 q of the row's stream; it writes words q and q + 8
      const uint32_t* lo = sw ? wa1 : wa0;  // chunk 2q
      const uint32_t* hi = sw ? wa0 : wa1;  // chunk 2q + 1
      const uint32_t f0 = comb4(lo[0]), f1 = comb4(lo[PB / 4 - 1]);
      const uint32_t f2 = comb4(hi[0]), f3 = comb4(hi[PB / 4 - 1]);
      const uint32_t p_lo = f0 | (f1 << 12) | (f2 << 24), p_hi = (f2 >> 8) | (f3 << 4);
      const int rbase = lane & ~7;
      uint32_t word[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int w = min(q + 8 * k, kWords - 1);
        const int A = (5 * w) >> 3, oA = 30 * w - 48 * A;  // first source lane, bit offset in it
        const uint32_t alo = __shfl_sync(kFull, p_lo, rbase + A), ahi = __shfl_sync(kFull, p_hi, rbase + A);
        const uint32_t blo = __shfl_sync(kFull, p_lo, rbase + min(A + 1, 7));
        const uint64_t pa = (uint64_t)alo | ((uint64_t)ahi << 32);
        const uint64_t pb = A + 1 < 8 ? (uint64_t)blo << (48 - oA) : 0ull;
        word[k] = (uint32_t)((pa >> oA) | pb) & 0x3FFFFFFFu;
      }
      if (live) {
        uint32_t* rowdst = T.codes + (int64_t)n * T.codes_sstride + (int64_t)(row0 + lr) * kWords;
        rowdst[q] = word[0];
        if (q + 8 < kWords) rowdst[q + 8] = word[1];
      }
    } else if (live) {
      uint32_t* rowdst = T.codes + (int64_t)n * T.codes_sstride + (int64_t)(row0 + lr) * kWords;
      if (BITS == 4) {
        reinterpret_cast<uint2*>(rowdst)[q] = sw ? make_uint2(wa1[0], wa0[0]) : make_uint2(wa0[0], wa1[0]);
      } else {
        reinterpret_cast<uint4*>(rowdst)[q] = sw ? make_uint4(wa1[0], wa1[1], wa0[0], wa0[1])
                                                 : make_uint4(wa0[0], wa0[1], wa1[0], wa1[1]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Per-channel key block of T tokens, W warps: warp w owns rows
// [w T/W, (w+1) T/W); sixteen lanes cover one row (8 channels each), two rows
// per instruction. The warps' per-channel minima and maxima meet in shared
// memory; one thread per channel then forms the scale, zero point and bracket.
// ---------------------------------------------------------------------------
template <int W>
struct KeyScratch {
  __half mn[W][kHeadDim];
  __half mx[W][kHeadDim];
  float nz[kHeadDim], rlo[kHeadDim], rhi[kHeadDim], s[kHeadDim];
};

template <int BITS, int TB, bool OUTL, int W>
__device__ __forceinline__ bool key_block(const unsigned char* tile, const TensorDev& K, int n,
                                          int blk, bool ok, KeyScratch<W>& ks, int warp, int lane,
                                          unsigned char* rowbuf, int kout, uint16_t* ombuf) {
  constexpr int kLev = (1 << BITS) - 1;
  constexpr int kRW = TB / W;  // rows of this warp
  constexpr int kIt = kRW / 2;      // rows per lane
  constexpr int kWords = Pack<BITS>::kWords;
  constexpr int PB = BITS == 3 ? 8 : BITS;
  const int o = lane & 15, p = lane >> 4;
  const uint4* t4 = reinterpret_cast<const uint4*>(tile);
  const __half2 pinf = __half2half2(__ushort_as_half(0x7C00));
  const __half2 ninf = __half2half2(__ushort_as_half(0xFC00));
  __half2 mn[4], mx[4];
  // Pass 1: per-channel minima and maxima of the block. With outliers each
  // token row (sixteen lanes hold it) first selects its outliers, which the
  // statistics leave out; ombuf keeps the lane's bits and its first CSR
  // position for the code pass. A tie in any row of the warp (a repeated
  // magnitude at the threshold) repeats the pass with unique keys.
  for (int pass = 0; pass < (OUTL ? 2 : 1); ++pass) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mn[j] = pinf;
      mx[j] = ninf;
    }
    bool tie = false;
#pragma unroll(OUTL ? 1 : 4)  // with outliers the body is long; code size matters more
    for (int i = 0; i < kIt; ++i) {
      const int row = warp * kRW + 2 * i + p;
      const uint4 raw = t4[row * 16 + o];
      const __half2* h = reinterpret_cast<const __half2*>(&raw);
      if (OUTL) {
        const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t mk[4], om;
        if (pass == 0) {
          uint32_t a[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) a[j] = wv[j] & 0x7FFF7FFFu;
          const uint32_t th = kth_magnitude<4, 16>(a, kout);
#pragma unroll
          for (int j = 0; j < 4; ++j) mk[j] = ge_mask(a[j], th);
          om = mask_bits<4>(mk);
        } else {
          om = exact_bits8(raw, o, kout);
          expand_mask4(om, mk);
        }
        int total;
        const int first = row_scan<16>(__popc(om), o, total);
        tie |= total != kout;
        ombuf[i * 32 + lane] = (uint16_t)(om | ((uint32_t)first << 8));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t wn = (wv[j] & ~mk[j]) | (0x7C007C00u & mk[j]);  // +inf
          const uint32_t wx = (wv[j] & ~mk[j]) | (0xFC00FC00u & mk[j]);  // -inf
          mn[j] = __hmin2(mn[j], *reinterpret_cast<const __half2*>(&wn));
          mx[j] = __hmax2(mx[j], *reinterpret_cast<const __half2*>(&wx));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mn[j] = __hmin2(mn[j], h[j]);
          mx[j] = __hmax2(mx[j], h[j]);
        }
      }
    }
    if (!OUTL || !__any_sync(kFull, tie)) break;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a = __shfl_xor_sync(kFull, *reinterpret_cast<uint32_t*>(&mn[j]), 16);
    uint32_t b = __shfl_xor_sync(kFull, *reinterpret_cast<uint32_t*>(&mx[j]), 16);
    mn[j] = __hmin2(mn[j], *reinterpret_cast<const __half2*>(&a));
    mx[j] = __hmax2(mx[j], *reinterpret_cast<const __half2*>(&b));
  }
  if (p == 0) {
    auto bits = [](__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); };
    *reinterpret_cast<uint4*>(&ks.mn[warp][8 * o]) = make_uint4(bits(mn[0]), bits(mn[1]), bits(mn[2]), bits(mn[3]));
    *reinterpret_cast<uint4*>(&ks.mx[warp][8 * o]) = make_uint4(bits(mx[0]), bits(mx[1]), bits(mx[2]), bits(mx[3]));
  }
  const bool all_ok = key_barrier_and<32 * W>(ok);
  bool fast = true;
  if (all_ok && threadIdx.x < kHeadDim) {
    const int c = threadIdx.x;  // one channel per thread
    __half m0 = ks.mn[0][c], m1 = ks.mx[0][c];
#pragma unroll
    for (int w = 1; w < W; ++w) {
      m0 = __hmin(m0, ks.mn[w][c]);
      m1 = __hmax(m1, ks.mx[w][c]);
    }
    float mnv = __fadd_rn(__half2float(m0), 0.0f);
    float mxv = __fadd_rn(__half2float(m1), 0.0f);
    if (OUTL && mnv > mxv) {  // every member of the channel's block is an outlier
      mnv = 0.0f;
      mxv = 0.0f;
    }
    const __half s16 = __float2half_rn(div_levels<kLev>(__fsub_rn(mxv, mnv)));
    const __half z16 = __float2half_rn(mnv);
    reinterpret_cast<__half2*>(K.meta + (int64_t)n * K.meta_sstride)[(int64_t)blk * kHeadDim + c] =
        __halves2half2(s16, z16);
    const float s = __half2float(s16);
    float rl, rh;
    bool slow;
    scale_bracket(s, rl, rh, slow);
    fast = !slow;
    ks.nz[c] = -mnv;
    ks.rlo[c] = rl;
    ks.rhi[c] = rh;
    ks.s[c] = s;
  }
  const bool all_fast = key_barrier_and<32 * W>(fast);
  if (!all_ok) return false;
  float nz[8], rl[8], rh[8];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float4 a = *reinterpret_cast<const float4*>(&ks.nz[8 * o + 4 * j]);
    const float4 b = *reinterpret_cast<const float4*>(&ks.rlo[8 * o + 4 * j]);
    const float4 c = *reinterpret_cast<const float4*>(&ks.rhi[8 * o + 4 * j]);
    nz[4 * j] = a.x; nz[4 * j + 1] = a.y; nz[4 * j + 2] = a.z; nz[4 * j + 3] = a.w;
    rl[4 * j] = b.x; rl[4 * j + 1] = b.y; rl[4 * j + 2] = b.z; rl[4 * j + 3] = b.w;
    rh[4 * j] = c.x; rh[4 * j + 1] = c.y; rh[4 * j + 2] = c.z; rh[4 * j + 3] = c.w;
  }
  uint32_t zh[4];  // the zero points of this lane's channel pairs, fp16 (exact)
#pragma unroll
  for (int j = 0; j < 4; ++j)
    zh[j] = (uint32_t)__half_as_ushort(__float2half_rn(-nz[2 * j])) |
            ((uint32_t)__half_as_ushort(__float2half_rn(-nz[2 * j + 1])) << 16);
  uint32_t* kdst = K.codes + (int64_t)n * K.codes_sstride + (int64_t)blk * TB * kWords;
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(tile);
  auto zat = [&](int i) { return ks.nz[8 * o + i]; };
  auto sat = [&](int i) { return ks.s[8 * o + i]; };
  auto rat = [&](int i) { return ks.rlo[8 * o + i]; };
#pragma unroll(OUTL ? 1 : 2)
  for (int i = 0; i < kIt; ++i) {
    const int row = warp * kRW + 2 * i + p;
    uint4 raw = t4[row * 16 + o];
    auto xat = [&](int e) { return xs[row * kHeadDim + 8 * o + e]; };
    uint32_t wa[PB / 4], wb[PB / 4];
    const uint32_t oe = OUTL ? ombuf[i * 32 + lane] : 0u;
    const uint32_t om = oe & 0xFFu;
    if (OUTL) {
      write_lane_csr(K, n, blk * TB + row, kout, om, 8 * o, (int)(oe >> 8), xs + row * kHeadDim);
      if (o == 0) write_rowptr(K, n, blk * TB + row, kout);
      // an outlier slot codes its channel's zero point (code 0 in both
      // brackets): its own value may lie outside the range, and a field out
      // of range would carry into its neighbours when the fields are summed
      uint32_t mk[4];
      expand_mask4(om, mk);
      raw.x = (raw.x & ~mk[0]) | (zh[0] & mk[0]);
      raw.y = (raw.y & ~mk[1]) | (zh[1] & mk[1]);
      raw.z = (raw.z & ~mk[2]) | (zh[2] & mk[2]);
      raw.w = (raw.w & ~mk[3]) | (zh[3] & mk[3]);
    }
    if (all_fast) {
      chunk_codes<PB, false>(raw, nz, rl, rh, wa, wb);
      uint32_t diff = 0;
#pragma unroll
      for (int j = 0; j < PB / 4; ++j) diff |= wa[j] ^ wb[j];
      if (__any_sync(kFull, diff != 0)) settle_chunk<PB, false>(wa, wb, xat, zat, sat, rat);
    } else {
      slow_chunk<PB, false, kLev>(wa, xat, zat, sat);
      if (OUTL)
        for (uint32_t m = om; m; m &= m - 1) clear_field<PB>(wa, __ffs(m) - 1);
    }
    if (BITS == 3) {
      // ten codes per word: the lane's 8 codes (channels 8 o ..) are 24 bits at
      // bit 24 o of the row's stream; lane o writes word o
      const uint32_t pw = comb4(wa[0]) | (comb4(wa[PB / 4 - 1]) << 12);
      const int w = min(o, kWords - 1);
      const int A = (5 * w) >> 2, oA = 30 * w - 24 * A;  // first source lane (0 .. 15), bit offset in it
      const int hbase = lane & 16;
      const uint32_t pa = __shfl_sync(kFull, pw, hbase + A);
      const uint32_t pb = __shfl_sync(kFull, pw, hbase + min(A + 1, 15));
      const uint32_t word = ((pa >> oA) | (A + 1 < 16 ? pb << (24 - oA) : 0u)) & 0x3FFFFFFFu;
      if (o < kWords) kdst[(int64_t)row * kWords + o] = word;
    } else if (BITS == 4)
      kdst[(int64_t)row * kWords + o] = wa[0];
    else
      reinterpret_cast<uint2*>(kdst + (int64_t)row * kWords)[o] = make_uint2(wa[0], wa[1]);
  }
  return true;
}

// ---------------------------------------------------------------------------
// The persistent kernel.
// ---------------------------------------------------------------------------
struct Args {
  TensorDev k, v;
  const __half* ksrc;
  const __half* vsrc;
  int seq_len;
  int in_rows;  // input rows between streams (>= seq_len)
  int k_items;  // key items per stream: whole blocks (+1 residual copy) or row chunks
  int k_nfull;  // whole per-channel key blocks per stream
  int v_items;  // value row chunks per stream
  int n_streams;
  int kout;  // outliers per row (0: none)
  uint32_t* status;
};

template <int KB, int KMODE, int TB, int VB, bool OUTL>
struct Geo {
  static constexpr bool kPerChannel = KMODE == KVQ_ASYM_PER_CHANNEL;
  static constexpr int kRows = (kPerChannel && TB > 64) ? TB : 64;  // rows per item
  static constexpr int kStageBytes = kRows * kHeadDim * 2;
  // Warps per CTA: eight where a stage is a 128-token key block (32 KB; at
  // most three CTAs fit an SM), four otherwise.
  static constexpr int kW = kRows == 128 ? 8 : 4;
  // Two stages per CTA and at least five CTAs per SM (at most 102 registers
  // a thread) where the stages are 16 KB: the same bytes in flight per SM as
  // three stages at four CTAs, with a quarter more warps to cover the
  // quantizer's dependency latencies (measured 0.604 -> 0.529 ms on a 2.75 GB
  // prefill). 32 KB stages (128-token key blocks) keep the register budget
  // of four CTAs.
  static constexpr int kStages = 2;
  static constexpr int kMinBlocks = kStageBytes <= 16384 ? 5 : 3;
  static constexpr size_t kScratch = kPerChannel ? sizeof(KeyScratch<kW>) : 0;
  static constexpr size_t kRowBuf = 0;  // per warp (the 3-bit codes are packed in registers)
  // per warp, the outlier masks of its key-block rows between the two passes
  static constexpr size_t kOmBuf = (kPerChannel && OUTL) ? (size_t)TB / kW / 2 * 32 * 2 : 0;
  static constexpr size_t kCtl = 64;  // counters and barriers
  static constexpr size_t kBytes =
      (size_t)kStages * kStageBytes + kScratch + kW * (kRowBuf + kOmBuf) + kCtl;
};

template <int KB, int KMODE, int TB, int VB, bool VSYM, bool OUTL>
__global__ void __launch_bounds__(32 * Geo<KB, KMODE, TB, VB, OUTL>::kW, (Geo<KB, KMODE, TB, VB, OUTL>::kMinBlocks))
    prefill_fast_kernel(Args a) {
  using G = Geo<KB, KMODE, TB, VB, OUTL>;
  constexpr int S = G::kStages;
  constexpr int W = G::kW;
  constexpr int RPW = G::kRows / W;
  extern __shared__ __align__(128) unsigned char smem[];
  KeyScratch<W>& ks = *reinterpret_cast<KeyScratch<W>*>(smem + S * G::kStageBytes);
  unsigned char* rowbuf = smem + S * G::kStageBytes + G::kScratch + (size_t)(threadIdx.x >> 5) * G::kRowBuf;
  uint16_t* ombuf = reinterpret_cast<uint16_t*>(smem + S * G::kStageBytes + G::kScratch + W * G::kRowBuf +
                                                (size_t)(threadIdx.x >> 5) * G::kOmBuf);
  unsigned char* ctl = smem + S * G::kStageBytes + G::kScratch + W * (G::kRowBuf + G::kOmBuf);
  int* cnt = reinterpret_cast<int*>(ctl);           // [S] warps done with a stage
  int* issued = reinterpret_cast<int*>(ctl + 16);   // [S] copies issued into a stage
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl + 32);  // [S]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_stream = a.k_items + a.v_items;
  const int total = a.n_streams * per_stream;

  struct Item {
    int n, kind, idx, row0, nrows;  // kind: 0 key block, 1 key residual, 2 key rows, 3 value rows
  };
  auto item = [&](int it) {
    Item r;
    r.n = it / per_stream;
    const int j = it - r.n * per_stream;
    if (j < a.k_items) {
      if (G::kPerChannel) {
        r.kind = j < a.k_nfull ? 0 : 1;
        r.idx = j;
        r.row0 = j * TB;
        r.nrows = r.kind == 0 ? TB : 0;
      } else {
        r.kind = 2;
        r.idx = j;
        r.row0 = j * G::kRows;
        r.nrows = min(G::kRows, a.seq_len - r.row0);
      }
    } else {
      r.kind = 3;
      r.idx = j - a.k_items;
      r.row0 = r.idx * G::kRows;
      r.nrows = min(G::kRows, a.seq_len - r.row0);
    }
    return r;
  };
  auto issue = [&](int it, int s) {
    const Item r = item(it);
    const __half* src = r.kind == 3 ? a.vsrc : a.ksrc;
    const uint32_t bytes = (uint32_t)r.nrows * kHeadDim * 2;
    issued[s] += 1;
    mbar_arrive_expect_tx(&full[s], bytes);
    if (bytes)
      bulk_g2s(smem + (size_t)s * G::kStageBytes,
               src + ((int64_t)r.n * a.in_rows + r.row0) * kHeadDim, bytes, &full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      cnt[s] = 0;
      issued[s] = 0;
    }
    mbar_fence_init();
  }
  __syncthreads();
  const int first = blockIdx.x, stride = gridDim.x;
  if (tid == 0)
    for (int s = 0; s < S && first + s * stride < total; ++s) issue(first + s * stride, s);

  bool dead = false;
  int k = 0;
  for (int it = first; it < total; it += stride, ++k) {
    const int s = k % S;
    const Item r = item(it);
    bool ok = !dead && mbar_wait_bounded(&full[s], (uint32_t)(k / S) & 1u);
    if (!ok && !dead) {
      dead = true;
      if (lane == 0) raise_status(a.status, kStatusTimeout);
    }
    const unsigned char* tile = smem + (size_t)s * G::kStageBytes;
    if (r.kind == 0) {
      if constexpr (G::kPerChannel) {
        if (!key_block<KB, TB, OUTL, W>(tile, a.k, r.n, r.idx, ok, ks, warp, lane, rowbuf, a.kout, ombuf))
          dead = true;
      }
    } else if (!dead) {
      if (r.kind == 1) {
        // key residual: the last S mod T tokens stay fp16
        const int t0 = a.k_nfull * TB;
        const uint4* s4 = reinterpret_cast<const uint4*>(a.ksrc + ((int64_t)r.n * a.in_rows + t0) * kHeadDim);
        uint4* d4 = reinterpret_cast<uint4*>(a.k.resid + (int64_t)r.n * a.k.resid_sstride);
        const int count = (a.seq_len - t0) * (kHeadDim / 8);
        for (int i = tid; i < count; i += 32 * W) d4[i] = s4[i];
      } else if (r.kind == 2) {
        rows_warp<KB, KMODE == KVQ_SYM_PER_TOKEN, RPW, OUTL>(tile, a.k, r.n, r.row0, r.nrows, warp, lane,
                                                             rowbuf, a.kout);
      } else {
        rows_warp<VB, VSYM, RPW, OUTL>(tile, a.v, r.n, r.row0, r.nrows, warp, lane, rowbuf, a.kout);
      }
    }
    if (!dead) {
      // release the stage; the last of the four warps refills it
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(&cnt[s], 1) == W - 1) {
          cnt[s] = 0;
          __threadfence_block();
          const int nxt = it + S * stride;
          if (nxt < total) {
            fence_proxy_async_smem();
            issue(nxt, s);
          }
        }
      }
    }
  }
  // No copy may still be landing in shared memory when the CTA exits (after a
  // timeout some were issued and never waited for).
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < S; ++s)
      if (issued[s] > 0) (void)mbar_wait_bounded(&full[s], (uint32_t)(issued[s] - 1) & 1u);
}

template <int KB, int KMODE, int TB, int VB, bool VSYM, bool OUTL>
cudaError_t launch_fast_t(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                          cudaStream_t st) {
  using G = Geo<KB, KMODE, TB, VB, OUTL>;
  auto kern = prefill_fast_kernel<KB, KMODE, TB, VB, VSYM, OUTL>;
  static SmemAttr attr;
  static std::atomic<int> occ_cached{0};  // resident CTAs per SM, computed once
  {
    const cudaError_t e = attr.ensure(kern, G::kBytes);
    if (e != cudaSuccess) return e;
  }
  int occ = occ_cached.load(std::memory_order_relaxed);
  if (occ == 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 32 * G::kW, G::kBytes);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    occ_cached.store(occ, std::memory_order_relaxed);
  }
  Args a;
  a.k = L.k;
  a.v = L.v;
  a.ksrc = k;
  a.vsrc = v;
  a.seq_len = seq_len;
  a.in_rows = L.in_rows > 0 ? L.in_rows : seq_len;
  a.n_streams = L.n_streams;
  a.kout = OUTL ? L.outliers : 0;
  a.status = L.status;
  a.v_items = (seq_len + G::kRows - 1) / G::kRows;
  if (G::kPerChannel) {
    a.k_nfull = seq_len / TB;
    a.k_items = a.k_nfull + (seq_len % TB ? 1 : 0);
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
  kern<<<grid, 32 * G::kW, G::kBytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace pfx
}  // namespace kvq
