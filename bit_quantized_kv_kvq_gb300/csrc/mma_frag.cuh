// Fragment-level helpers of the tensor-core decode kernels: the fp16 mma,
// fp16 hi/lo splitting of fp32 operands, and the map from a thread's key
// k-slots to the channels whose packed codes it extracts.
//
// m16n8k16 fragments (fp16 inputs, fp32 accumulators), lane = 4 g + t4:
//   A (16 x 16, row): a0 = A[g][2t4, 2t4+1], a1 = A[g+8][2t4, 2t4+1],
//                     a2 = A[g][2t4+8, 2t4+9], a3 = A[g+8][2t4+8, 2t4+9]
//   B (16 x 8, col):  b0 = B[2t4, 2t4+1][g], b1 = B[2t4+8, 2t4+9][g]
//   C (16 x 8):       c0 = C[g][2t4], c1 = C[g][2t4+1], c2 = C[g+8][2t4], c3 = C[g+8][2t4+1]
// Within each k-chunk of 16 a thread's k-slots s0..s3 are 2t4, 2t4+1, 2t4+8
// and 2t4+9.
#pragma once

#include "common.cuh"

namespace kvq {
namespace tc {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                    uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (lo, hi) -> fp16x2 with lo in the low half.
__device__ __forceinline__ uint32_t f2h2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// hi + lo split of a float pair: returns the hi pair, *lo_out the lo pair.
__device__ __forceinline__ uint32_t split_pair(float v0, float v1, uint32_t& lo_out) {
  const uint32_t hi = f2h2(v0, v1);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  lo_out = f2h2(__fsub_rn(v0, hf.x), __fsub_rn(v1, hf.y));
  return hi;
}

// ---------------------------------------------------------------------------
// Keys: which channel each k-slot of a thread carries, and how many bits up
// its code sits in the fp16 half (the slot's Q'' is scaled by 2^-shift).
// Slots of thread t4 in chunk kc: s0 = 2t4, s1 = 2t4+1, s2 = 2t4+8, s3 = 2t4+9.
// ---------------------------------------------------------------------------
//  4-bit: word w = 4 t4 + kc/2 of the row, h = kc & 1; the halves of
//         (w >> 8h) & 0x000F000F are nibbles 2h, 2h+4 (s0, s1) and of
//         (w >> 8h) & 0x00F000F0 nibbles 2h+1, 2h+5 (s2, s3; 4 bits up).
//  8-bit: word w = 8 t4 + kc; w & 0x00FF00FF = bytes 0, 2 (s0, s1),
//         (w >> 8) & 0x00FF00FF = bytes 1, 3 (s2, s3).
//  3-bit: words A = t4, B = t4+4, C = t4+8 and D = 12 of the row; sixteen
//         code pairs p (kc uses p = 2kc for s0/s1 and 2kc+1 for s2/s3):
//         p = 4i+m of word X = t4+4i: m=0 X & 0x001C0007 (codes 0, 6),
//         m=1 X & 0x00E00038 (1, 7), m=2 (X>>6) & 0x001C0007 (2, 8),
//         m=3 (X>>9) & 0x001C0007 (3, 9); p = 12, 13: codes 4 and 5 of A and
//         B (a byte permute of A>>12 and B>>12, masks 7 and 7<<3); p = 14, 15:
//         codes 4, 5 of C with codes 2t4, 2t4+1 of D.
__host__ __device__ constexpr int key3_shift_of_code(int j) {
  return j == 1 || j == 5 ? 3 : j == 7 ? 5 : (j == 6 || j == 8 || j == 9) ? 2 : 0;
}

template <int KB>
__device__ __forceinline__ void key_slot(int t4, int kc, int s, int& ch, int& shift) {
  if (KB == 4) {
    const int w = 4 * t4 + (kc >> 1), h = kc & 1;
    const int nib = 2 * h + (s == 0 ? 0 : s == 1 ? 4 : s == 2 ? 1 : 5);
    ch = 8 * w + nib;
    shift = (s >= 2) ? 4 : 0;
  } else if (KB == 8) {
    const int w = 8 * t4 + kc;
    ch = 4 * w + (s == 0 ? 0 : s == 1 ? 2 : s == 2 ? 1 : 3);
    shift = 0;
  } else {
    const int p = 2 * kc + (s >> 1), half = s & 1;
    if (p < 12) {
      const int wx = t4 + 4 * (p >> 2), m = p & 3;
      const int j = half ? m + 6 : m;
      ch = 10 * wx + j;
      shift = key3_shift_of_code(j);
    } else if (p == 12 || p == 13) {
      const int j = p == 12 ? 4 : 5;
      ch = 10 * (half ? t4 + 4 : t4) + j;
      shift = key3_shift_of_code(j);
    } else {
      const int j = p == 14 ? 4 : 5;
      ch = half ? 120 + 2 * t4 + (p - 14) : 10 * (t4 + 8) + j;
      shift = p == 14 ? 0 : 3;
    }
  }
}

// shift of a key channel (a function of the channel alone)
template <int KB>
__host__ __device__ constexpr int key_shift(int c) {
  return KB == 4 ? ((c & 1) ? 4 : 0)
                 : KB == 8 ? 0 : (c >= 120 ? ((c & 1) ? 3 : 0) : key3_shift_of_code(c % 10));
}

// 2^e as a float for -126 <= e <= 127.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

}  // namespace tc
}  // namespace kvq
