// Decode attention for 2, 4 or 8 query heads per kv-head (GQA) on the
// tensor cores (mma.sync m16n8k16, fp16 inputs, fp32 accumulation).
//
// The g query heads that share a kv-head read each K/V tile once, so QK^T and
// PV are small dense contractions over a tile:
//   S[t][h]   = sum_c n[t][c] Q''[c][h]      M = 16 tokens, N = 8 heads, K = 16 channels
//   O^T[c][h] = sum_t n[t][c] P'[h][t]       M = 16 channels, N = 8 heads, K = 16 tokens
// with n the integer codes (exact in fp16: the code is placed in the mantissa
// of 1024 by a byte permute and 1024 is subtracted exactly), Q'' = q * s for
// per-channel keys (bias sum_c q_c z_c added in fp32) and P' = p * s_t for the
// value scales (sum_t p_t z_t added in fp32) -- dequantization folded into the
// attention products (TurboQuant KV-cache page, demingchina.com/news/57821,
// §2.3). Q'' and P' are fp32 values carried as an fp16 pair hi + lo, so the
// products keep about 22 bits. Within one mma the channel <-> k-slot
// assignment is free as long as both operands use it; it is chosen so that a
// thread builds two code pairs from two words with one permute.
//
// Pipeline, warp-local softmax with a lazily moved max and the final
// log-sum-exp merge of the 4 warps follow the MHA kernel (decode_mha.cuh).
#pragma once

#include "common.cuh"
#include "decode_merge.cuh"

namespace kvq {
namespace gqa {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kRows = 32;  // tokens per warp tile (two m16 tiles)
constexpr float kLazy = 8.0f;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2u(uint32_t x, uint32_t y) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&y));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t h2u(__half lo, __half hi) {
  __half2 r = __halves2half2(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

// fp32 v = hi + lo (+ O(2^-22 |v|)) with hi, lo fp16.
__device__ __forceinline__ void split2(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t x, uint32_t y, uint32_t z) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&y),
                      *reinterpret_cast<__half2*>(&z));
  return *reinterpret_cast<uint32_t*>(&r);
}

// fp16 code pair (1024 + n) in the two halves -> exact (n, n').
constexpr uint32_t kH1024 = 0x64006400u;  // (1024, 1024)
constexpr uint32_t kH1152 = 0x64806480u;  // (1152, 1152): offset-binary int8
// (1024 + n, 1024 + 4 n') * (1, 1/4) + (-1024, -256) = (n, n') exactly
constexpr uint32_t kH1Quarter = 0x34003C00u;     // (1.0, 0.25)
constexpr uint32_t kHNeg1024_256 = 0xDC00E400u;  // (-1024, -256)

template <int KB, int KMODE, int VB, int VMODE>
struct Cfg {
  static constexpr bool KCH = KMODE == KVQ_ASYM_PER_CHANNEL;
  static constexpr bool KSYM = KMODE == KVQ_SYM_PER_TOKEN;
  static constexpr bool VSYM = VMODE == KVQ_SYM_PER_TOKEN;
  // codebook codes: a 4-bit code indexes 16 fp16 levels (one table lookup
  // per pair of codes); like symmetric codes their groups have a scale only
  static constexpr bool KCB = KMODE == KVQ_CODEBOOK_PER_TOKEN;
  static constexpr bool VCB = VMODE == KVQ_CODEBOOK_PER_TOKEN;
  static constexpr bool KSC = KSYM || KCB;  // scale-only key groups
  static constexpr bool VSC = VSYM || VCB;
  static constexpr int KW = Pack<KB>::kWords, VW = Pack<VB>::kWords;
  static constexpr int KC_BYTES = kRows * KW * 4;
  static constexpr int VC_BYTES = kRows * VW * 4;
  static constexpr int META = 512;
  static constexpr int STAGE = KC_BYTES + VC_BYTES + 2 * META;
  static constexpr int kStagesPerWarp = STAGE <= 5 * 1024 ? 3 : 2;
  static constexpr size_t stage_bytes() { return (size_t)kWarps * kStagesPerWarp * STAGE; }
  static constexpr size_t merge_bytes() { return (size_t)kWarps * 8 * kHeadDim * 4; }
  static constexpr size_t smem_bytes() {
    return (stage_bytes() > merge_bytes() ? stage_bytes() : merge_bytes()) +
           8 * kHeadDim * 4 /*q*/ + kWarps * 8 * 2 * 4 /*m, l*/ +
           kWarps * 3 * 8 /*bars*/;
  }
};

// Channel of k-slot `slot` (0..15) in key chunk kc for a thread with t4.
// 4-bit keys: chunk kc = words 2kc, 2kc+1; slot 2t4 <-> 2t4, 2t4+1 <-> 8+2t4,
// 2t4+8 <-> 2t4+1, 2t4+9 <-> 9+2t4 (offsets inside the chunk).
// 8-bit keys: chunk kc (group q, local l) uses word q*(Gp/4) + t4*(Gp/16) + l;
// slots 2t4, 2t4+1, 2t4+8, 2t4+9 <-> bytes 0, 2, 1, 3 of that word.
// 3-bit keys (ten codes per word, thirteen words per row): a thread with t4
// reads words t4, t4+4, t4+8 and the last word; its 16 code pairs are
//   p = 0..11: codes (j, j+6) of word t4 + 4*(p/4), j = p mod 4,
//   p = 12, 13: code 4 / code 5 of words t4 and t4+4,
//   p = 14, 15: code 4 / code 5 of word t4+8 with codes 2t4 / 2t4+1 of word 12;
// chunk kc uses pairs 2kc (slots 2t4, 2t4+1) and 2kc+1 (slots 2t4+8, 2t4+9).
__device__ __forceinline__ int key3_pair_channel(int p, int t4, int second) {
  if (p < 12) {
    const int w = t4 + 4 * (p >> 2), j = p & 3;
    return 10 * w + j + (second ? 6 : 0);
  }
  if (p == 12) return second ? 10 * (t4 + 4) + 4 : 10 * t4 + 4;
  if (p == 13) return second ? 10 * (t4 + 4) + 5 : 10 * t4 + 5;
  if (p == 14) return second ? 120 + 2 * t4 : 10 * (t4 + 8) + 4;
  return second ? 121 + 2 * t4 : 10 * (t4 + 8) + 5;
}

template <int KB>
__device__ __forceinline__ int key_channel(int kc, int t4, int which, int gp) {
  if (KB == 3) return key3_pair_channel(2 * kc + (which >> 1), t4, which & 1);
  if (KB == 4) {
    const int base = 16 * kc;
    return which == 0 ? base + 2 * t4 : which == 1 ? base + 8 + 2 * t4
           : which == 2 ? base + 2 * t4 + 1 : base + 9 + 2 * t4;
  } else {
    const int per = gp / 16;
    const int q = kc / per, l = kc - q * per;
    const int w = q * (gp / 4) + t4 * per + l;
    return 4 * w + (which == 0 ? 0 : which == 1 ? 2 : which == 2 ? 1 : 3);
  }
}

// FG: 0, or the group size of per-token keys and of values when both are
// fixed at compile time (then every per-group loop unrolls with constant
// group indices).
template <int KB, int KMODE, int VB, int VMODE, int FG>
__global__ void __launch_bounds__(kThreads, 3)
    decode_gqa_kernel(LayerDev L, DecodeArgs a) {
  using C = Cfg<KB, KMODE, VB, VMODE>;
  constexpr int kStagesPerWarp = C::kStagesPerWarp;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int split = blockIdx.x, n = blockIdx.y;
  const int b = n / L.num_kv_heads;
  const int kvh = n - b * L.num_kv_heads;
  const int G = a.gqa;
  const int hq0 = kvh * G;

  const size_t big = C::stage_bytes() > C::merge_bytes() ? C::stage_bytes() : C::merge_bytes();
  unsigned char* stages = smem;
  float* mo = reinterpret_cast<float*>(smem);  // reused after the main loop: [warps][8][128]
  float* qf = reinterpret_cast<float*>(smem + big);  // [8][128], heads >= G are zero
  float* ml = qf + 8 * kHeadDim;                     // [warps][8][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ml + kWarps * 16);

  const int len = a.varlen ? a.lens[b] : a.length, kq = a.k_quant_len;  // this batch row's tokens
  const int row_begin = split * a.tiles_per_split * kTile;
  const int row_end = max(row_begin, min(row_begin + a.tiles_per_split * kTile, len));  // empty past a short row
  const int ntiles = (row_end - row_begin + kRows - 1) / kRows;
  const int per_warp = (ntiles + kWarps - 1) / kWarps;
  const int w_first = min(warp * per_warp, ntiles);
  const int w_count = min(per_warp, ntiles - w_first);
  const int Gk = FG ? FG : L.k.group, Gv = FG ? FG : L.v.group;
  const int kgpr = C::KCH ? 1 : kHeadDim / Gk;
  const int vgpr = kHeadDim / Gv;
  const int gp = C::KCH ? kHeadDim : Gk;  // key group that chunks must not straddle
  const int mpg = Gv / 16;                 // m16 value-channel tiles per value group (2, 4, 8)
  const int mpg_log2 = mpg == 8 ? 3 : mpg == 4 ? 2 : 1;

  const uint32_t* kcodes = L.k.codes + (int64_t)n * L.k.codes_sstride;
  const uint32_t* vcodes = L.v.codes + (int64_t)n * L.v.codes_sstride;
  const unsigned char* kmeta = L.k.meta + (int64_t)n * L.k.meta_sstride;
  const unsigned char* vmeta = L.v.meta + (int64_t)n * L.v.meta_sstride;

  uint64_t* wb = bars + warp * kStagesPerWarp;
  auto stage_ptr = [&](int s) { return stages + (size_t)(warp * kStagesPerWarp + s) * C::STAGE; };
  auto issue = [&](int ti, int s) {
    unsigned char* base = stage_ptr(s);
    const int t0 = row_begin + (w_first + ti) * kRows;
    const bool rt = C::KCH && t0 >= kq;
    const uint32_t kmb = C::KCH ? (uint32_t)(kHeadDim * 4) : (uint32_t)(kRows * kgpr * (C::KSC ? 2 : 4));
    const uint32_t vmb = (uint32_t)(kRows * vgpr * (C::VSC ? 2 : 4));
    mbar_arrive_expect_tx(&wb[s], C::VC_BYTES + vmb + (rt ? 0u : C::KC_BYTES + kmb));
    if (!rt) {
      bulk_g2s(base, kcodes + (int64_t)t0 * C::KW, C::KC_BYTES, &wb[s]);
      const unsigned char* ks = C::KCH ? kmeta + (int64_t)(t0 / Gk) * kHeadDim * 4
                                       : kmeta + (int64_t)t0 * kgpr * (C::KSC ? 2 : 4);
      bulk_g2s(base + C::KC_BYTES + C::VC_BYTES, ks, kmb, &wb[s]);
    }
    bulk_g2s(base + C::KC_BYTES, vcodes + (int64_t)t0 * C::VW, C::VC_BYTES, &wb[s]);
    bulk_g2s(base + C::KC_BYTES + C::VC_BYTES + C::META,
             vmeta + (int64_t)t0 * vgpr * (C::VSC ? 2 : 4), vmb, &wb[s]);
  };
  // lane 0 of each warp: its barriers and its first copies, before the
  // query load, so that the two latencies overlap
  if (lane == 0) {
    for (int s = 0; s < kStagesPerWarp; ++s) mbar_init(&wb[s], 1);
    mbar_fence_init();
    for (int s = 0; s < kStagesPerWarp && s < w_count; ++s) issue(s, s);
  }

  for (int i = tid; i < 8 * kHeadDim; i += kThreads) {
    const int h = i >> 7, c = i & 127;
    qf[i] = h < G ? __half2float(a.q[((int64_t)b * a.num_q_heads + hq0 + h) * kHeadDim + c]) *
                        a.scale_log2
                  : 0.0f;
  }
  // codebook codes: entry i holds the fp16 pair (level[i & 15], level[i >> 4])
  __shared__ uint32_t cbl[(C::KCB || C::VCB) ? 256 : 1];
  if (C::KCB || C::VCB)
    for (int i = tid; i < 256; i += kThreads)
      cbl[i] = (uint32_t)L.codebook[i & 15] | ((uint32_t)L.codebook[i >> 4] << 16);
  __syncthreads();

  // ---- query fragments (B operand of QK^T), head = g ---------------------------
  // per-token keys: fixed; per-channel keys: rebuilt per key block with q*s.
  uint32_t bqh[8][2], bql[8][2];
  float qsum_g[4];  // per key group: sum_c q[g][c] (per-token keys)
  auto build_q = [&](const __half2* ksz) {
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      __half hi[4], lo[4];
#pragma unroll
      for (int wh = 0; wh < 4; ++wh) {
        const int c = key_channel<KB>(kc, t4, wh, gp);
        float v = qf[g * kHeadDim + c];
        if (C::KCH) v *= __low2float(ksz[c]);
        split2(v, hi[wh], lo[wh]);
      }
      bqh[kc][0] = h2u(hi[0], hi[1]);
      bqh[kc][1] = h2u(hi[2], hi[3]);
      bql[kc][0] = h2u(lo[0], lo[1]);
      bql[kc][1] = h2u(lo[2], lo[3]);
    }
  };
  if (!C::KCH) {
    build_q(nullptr);
#pragma unroll
    for (int q = 0; q < 4; ++q) qsum_g[q] = 0.0f;
    if (!C::KSC) {  // scale-only keys have no zero point: the sums are not used
      // lane t4 of row g sums channels t4, t4 + 4, ... of head g per key group
      // (groups of 32, 64 or 128 channels), then the row's four lanes combine
      const int gshift = __ffs(Gk) - 1;
      for (int c = t4; c < kHeadDim; c += 4) {
        const float x = qf[g * kHeadDim + c];
        const int q = c >> gshift;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq)
          if (qq == q) qsum_g[qq] += x;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        qsum_g[q] += __shfl_xor_sync(kFull, qsum_g[q], 1);
        qsum_g[q] += __shfl_xor_sync(kFull, qsum_g[q], 2);
      }
    }
  }
  // bias of the current key block for the thread's two heads (2t4, 2t4+1)
  float kb0 = 0.0f, kb1 = 0.0f;
  int cur_blk = -1;

  // ---- state -----------------------------------------------------------------
  float m0 = -INFINITY, m1 = -INFINITY;  // running max of heads 2t4, 2t4+1
  float l0 = 0.0f, l1 = 0.0f;            // partial sums over this thread's rows
  float z0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, z1[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // sum p z per value group
  float o[8][4];
#pragma unroll
  for (int mv = 0; mv < 8; ++mv)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mv][e] = 0.0f;

  bool failed = false;
  int ti = 0;
  for (; ti < w_count; ++ti) {
    const int s = ti % kStagesPerWarp;
    const uint32_t par = (uint32_t)(ti / kStagesPerWarp) & 1u;
    const int t0 = row_begin + (w_first + ti) * kRows;
    const bool rt = C::KCH && t0 >= kq;
    unsigned char* base = stage_ptr(s);
    const uint32_t* kc_s = reinterpret_cast<const uint32_t*>(base);
    const uint32_t* vc_s = reinterpret_cast<const uint32_t*>(base + C::KC_BYTES);
    const unsigned char* km = base + C::KC_BYTES + C::VC_BYTES;
    const unsigned char* vm = km + C::META;
    if (!mbar_wait_bounded(&wb[s], par)) {
      failed = true;
      break;
    }
    __syncwarp();

    // ---- scores: S[mt] in mma C layout (rows g, g+8; heads 2t4, 2t4+1) -------
    float S[2][4];
    if (!rt) {
      if (C::KCH && (t0 / Gk) != cur_blk) {
        cur_blk = t0 / Gk;
        const __half2* ksz = reinterpret_cast<const __half2*>(km);
        build_q(ksz);
        float part = 0.0f;
#pragma unroll
        for (int kc = 0; kc < 8; ++kc)
#pragma unroll
          for (int wh = 0; wh < 4; ++wh) {
            const int c = key_channel<KB>(kc, t4, wh, gp);
            part = fmaf(qf[g * kHeadDim + c], __high2float(ksz[c]), part);
          }
        part += __shfl_xor_sync(kFull, part, 1);
        part += __shfl_xor_sync(kFull, part, 2);  // bias of head g in lanes 4g..4g+3
        kb0 = __shfl_sync(kFull, part, 4 * (2 * t4));
        kb1 = __shfl_sync(kFull, part, 4 * (2 * t4 + 1));
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int r0 = 16 * mt + g, r1 = r0 + 8;
        float acc[4][4];  // per key group (per-token keys) or [0] only
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[q][e] = 0.0f;
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
          uint32_t af[4];
          if (KB == 3) {
            // rows r0 / r1: pairs 2kc (-> a0 / a1) and 2kc+1 (-> a2 / a3)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t* rw = kc_s + (half ? r1 : r0) * C::KW;
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int p = 2 * kc + e;
                uint32_t v;
                if (p < 12) {
                  const uint32_t w = rw[t4 + 4 * (p >> 2)];
                  v = ((w >> (3 * (p & 3))) & 0x001C0007u) | kH1024;
                  v = hfma2u(v, kH1Quarter, kHNeg1024_256);  // (n_j, n_{j+6})
                } else {
                  uint32_t lo, hi;
                  if (p == 12) { lo = rw[t4] >> 12; hi = rw[t4 + 4] >> 12; }
                  else if (p == 13) { lo = rw[t4] >> 15; hi = rw[t4 + 4] >> 15; }
                  else if (p == 14) { lo = rw[t4 + 8] >> 12; hi = rw[12] >> (6 * t4); }
                  else { lo = rw[t4 + 8] >> 15; hi = rw[12] >> (6 * t4 + 3); }
                  v = hsub2u((__byte_perm(lo, hi, 0x5410u) & 0x00070007u) | kH1024, kH1024);
                }
                af[2 * e + half] = v;
              }
            }
          } else if (KB == 4) {
            const uint2 w0 = *reinterpret_cast<const uint2*>(kc_s + r0 * C::KW + 2 * kc);
            const uint2 w1 = *reinterpret_cast<const uint2*>(kc_s + r1 * C::KW + 2 * kc);
            const uint32_t sel = (uint32_t)(t4 | (t4 << 4) | ((4 + t4) << 8) | ((4 + t4) << 12));
            const uint32_t x0 = __byte_perm(w0.x, w0.y, sel);
            const uint32_t x1 = __byte_perm(w1.x, w1.y, sel);
            if (C::KCB) {  // the two codes of each half pair index the level-pair table
              af[0] = cbl[(x0 & 0xFu) | ((x0 >> 12) & 0xF0u)];
              af[2] = cbl[((x0 >> 4) & 0xFu) | ((x0 >> 16) & 0xF0u)];
              af[1] = cbl[(x1 & 0xFu) | ((x1 >> 12) & 0xF0u)];
              af[3] = cbl[((x1 >> 4) & 0xFu) | ((x1 >> 16) & 0xF0u)];
            } else {
              af[0] = hsub2u((x0 & 0x000F000Fu) | kH1024, kH1024);
              af[2] = hsub2u(((x0 >> 4) & 0x000F000Fu) | kH1024, kH1024);
              af[1] = hsub2u((x1 & 0x000F000Fu) | kH1024, kH1024);
              af[3] = hsub2u(((x1 >> 4) & 0x000F000Fu) | kH1024, kH1024);
            }
          } else {
            const int per = gp / 16;
            const int q = kc / per, l = kc - q * per;
            const int wi = q * (gp / 4) + t4 * per + l;
            uint32_t w0 = kc_s[r0 * C::KW + wi], w1 = kc_s[r1 * C::KW + wi];
            const uint32_t bias = C::KSYM ? kH1152 : kH1024;
            if (C::KSYM) {
              w0 ^= 0x80808080u;
              w1 ^= 0x80808080u;
            }
            af[0] = hsub2u(__byte_perm(w0, 0x64646464u, 0x4240u), bias);
            af[2] = hsub2u(__byte_perm(w0, 0x64646464u, 0x4341u), bias);
            af[1] = hsub2u(__byte_perm(w1, 0x64646464u, 0x4240u), bias);
            af[3] = hsub2u(__byte_perm(w1, 0x64646464u, 0x4341u), bias);
          }
          if (C::KCH) {
            mma16816(acc[0], af, bqh[kc][0], bqh[kc][1]);
            mma16816(acc[0], af, bql[kc][0], bql[kc][1]);
          } else {
            const int q = key_channel<KB>(kc, 0, 0, gp) / Gk;  // warp-uniform
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              if (qq == q) {
                mma16816(acc[qq], af, bqh[kc][0], bqh[kc][1]);
                mma16816(acc[qq], af, bql[kc][0], bql[kc][1]);
              }
          }
        }
        if (C::KCH) {
          S[mt][0] = acc[0][0] + kb0;
          S[mt][1] = acc[0][1] + kb1;
          S[mt][2] = acc[0][2] + kb0;
          S[mt][3] = acc[0][3] + kb1;
        } else {
          // per-token keys: S = sum_q s[t][q] acc_q + z[t][q] qsum_q(h)
          float sA = 0.0f, sB = 0.0f, sC = 0.0f, sD = 0.0f;
          for (int q = 0; q < kgpr; ++q) {
            float s_r0, s_r1, z_r0 = 0.0f, z_r1 = 0.0f;
            if (C::KSC) {
              s_r0 = __half2float(reinterpret_cast<const __half*>(km)[r0 * kgpr + q]);
              s_r1 = __half2float(reinterpret_cast<const __half*>(km)[r1 * kgpr + q]);
            } else {
              const float2 a0 = __half22float2(reinterpret_cast<const __half2*>(km)[r0 * kgpr + q]);
              const float2 a1 = __half22float2(reinterpret_cast<const __half2*>(km)[r1 * kgpr + q]);
              s_r0 = a0.x; z_r0 = a0.y; s_r1 = a1.x; z_r1 = a1.y;
            }
            float accq0 = 0, accq1 = 0, accq2 = 0, accq3 = 0;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              if (qq == q) {
                accq0 = acc[qq][0]; accq1 = acc[qq][1]; accq2 = acc[qq][2]; accq3 = acc[qq][3];
              }
            // qsum of head (2t4) / (2t4+1) for group q lives in lanes 4*(2t4) / 4*(2t4+1)
            float qs_mine = 0.0f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              if (qq == q) qs_mine = qsum_g[qq];
            const float qs0 = __shfl_sync(kFull, qs_mine, 4 * (2 * t4));
            const float qs1 = __shfl_sync(kFull, qs_mine, 4 * (2 * t4 + 1));
            sA = fmaf(s_r0, accq0, fmaf(z_r0, qs0, sA));
            sB = fmaf(s_r0, accq1, fmaf(z_r0, qs1, sB));
            sC = fmaf(s_r1, accq2, fmaf(z_r1, qs0, sC));
            sD = fmaf(s_r1, accq3, fmaf(z_r1, qs1, sD));
          }
          S[mt][0] = sA;
          S[mt][1] = sB;
          S[mt][2] = sC;
          S[mt][3] = sD;
        }
      }
    } else {
      // fp16 residual keys on the CUDA cores: rows g, g+8 of each m16 tile
      const __half* res =
          L.k.resid + (int64_t)n * L.k.resid_sstride + (int64_t)(t0 - kq) * kHeadDim;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int row = 16 * mt + g + 8 * half;
          float d0 = 0.0f, d1 = 0.0f;
          if (t0 + row < row_end) {
            const __half* kr = res + (size_t)row * kHeadDim;
            for (int c = 0; c < kHeadDim; c += 2) {
              const float2 x = __half22float2(*reinterpret_cast<const __half2*>(kr + c));
              d0 = fmaf(qf[(2 * t4) * kHeadDim + c], x.x, fmaf(qf[(2 * t4) * kHeadDim + c + 1], x.y, d0));
              d1 = fmaf(qf[(2 * t4 + 1) * kHeadDim + c], x.x, fmaf(qf[(2 * t4 + 1) * kHeadDim + c + 1], x.y, d1));
            }
          }
          S[mt][2 * half] = d0;
          S[mt][2 * half + 1] = d1;
        }
      }
    }
    // mask rows past the end of the split
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      if (t0 + 16 * mt + g >= row_end) {
        S[mt][0] = -INFINITY;
        S[mt][1] = -INFINITY;
      }
      if (t0 + 16 * mt + g + 8 >= row_end) {
        S[mt][2] = -INFINITY;
        S[mt][3] = -INFINITY;
      }
    }

    // ---- online softmax per head (heads 2t4 and 2t4+1 of this thread) --------
    float mt0 = fmaxf(fmaxf(S[0][0], S[0][2]), fmaxf(S[1][0], S[1][2]));
    float mt1 = fmaxf(fmaxf(S[0][1], S[0][3]), fmaxf(S[1][1], S[1][3]));
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mt0 = fmaxf(mt0, __shfl_xor_sync(kFull, mt0, off));
      mt1 = fmaxf(mt1, __shfl_xor_sync(kFull, mt1, off));
    }
    const bool up0 = mt0 > m0 + kLazy, up1 = mt1 > m1 + kLazy;
    if (__any_sync(kFull, up0 || up1)) {
      const float n0 = up0 ? mt0 : m0, n1 = up1 ? mt1 : m1;
      const float al0 = up0 ? exp2f(m0 - n0) : 1.0f, al1 = up1 ? exp2f(m1 - n1) : 1.0f;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        z0[q] *= al0;
        z1[q] *= al1;
      }
#pragma unroll
      for (int mv = 0; mv < 8; ++mv) {
        o[mv][0] *= al0;
        o[mv][1] *= al1;
        o[mv][2] *= al0;
        o[mv][3] *= al1;
      }
      m0 = n0;
      m1 = n1;
    }
    float P[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      P[mt][0] = exp2f(S[mt][0] - m0);
      P[mt][1] = exp2f(S[mt][1] - m1);
      P[mt][2] = exp2f(S[mt][2] - m0);
      P[mt][3] = exp2f(S[mt][3] - m1);
      l0 += P[mt][0] + P[mt][2];
      l1 += P[mt][1] + P[mt][3];
    }

    // ---- PV: per 16-token step; B operand (P' = p * s_t) per value group ---------
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int r0 = 16 * ks + g, r1 = r0 + 8;  // rows this thread holds in C layout
      const int ra = 16 * ks + 2 * t4;          // value rows of the A operand: ra, ra+1, ra+8, ra+9
      uint32_t bph0[4], bph1[4], bpl0[4], bpl1[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        bph0[q] = bph1[q] = bpl0[q] = bpl1[q] = 0u;
        if (q < vgpr) {  // warp-uniform
          float sv0, sv1, zv0 = 0.0f, zv1 = 0.0f;
          if (C::VSC) {
            sv0 = __half2float(reinterpret_cast<const __half*>(vm)[r0 * vgpr + q]);
            sv1 = __half2float(reinterpret_cast<const __half*>(vm)[r1 * vgpr + q]);
          } else {
            const float2 a0 = __half22float2(reinterpret_cast<const __half2*>(vm)[r0 * vgpr + q]);
            const float2 a1 = __half22float2(reinterpret_cast<const __half2*>(vm)[r1 * vgpr + q]);
            sv0 = a0.x; zv0 = a0.y; sv1 = a1.x; zv1 = a1.y;
          }
          z0[q] += fmaf(P[ks][0], zv0, P[ks][2] * zv1);  // sum_t p z, heads 2t4 / 2t4+1
          z1[q] += fmaf(P[ks][1], zv0, P[ks][3] * zv1);
          __half e_hi[4], e_lo[4];
          split2(P[ks][0] * sv0, e_hi[0], e_lo[0]);
          split2(P[ks][1] * sv0, e_hi[1], e_lo[1]);
          split2(P[ks][2] * sv1, e_hi[2], e_lo[2]);
          split2(P[ks][3] * sv1, e_hi[3], e_lo[3]);
          const uint32_t h01h = h2u(e_hi[0], e_hi[1]), h23h = h2u(e_hi[2], e_hi[3]);
          const uint32_t h01l = h2u(e_lo[0], e_lo[1]), h23l = h2u(e_lo[2], e_lo[3]);
          // transpose C layout -> B layout: b0 = P'[head g][tok 2t4, 2t4+1], b1 = [2t4+8, 2t4+9]
          const int ls1 = 4 * (2 * t4) + (g >> 1), ls2 = 4 * (2 * t4 + 1) + (g >> 1);
          const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
          bph0[q] = __byte_perm(__shfl_sync(kFull, h01h, ls1), __shfl_sync(kFull, h01h, ls2), sel);
          bph1[q] = __byte_perm(__shfl_sync(kFull, h23h, ls1), __shfl_sync(kFull, h23h, ls2), sel);
          bpl0[q] = __byte_perm(__shfl_sync(kFull, h01l, ls1), __shfl_sync(kFull, h01l, ls2), sel);
          bpl1[q] = __byte_perm(__shfl_sync(kFull, h23l, ls1), __shfl_sync(kFull, h23l, ls2), sel);
        }
      }
#pragma unroll
      for (int mv = 0; mv < 8; ++mv) {
        const int q = mv >> mpg_log2, l = mv & (mpg - 1);
        uint32_t b0h = bph0[0], b1h = bph1[0], b0l = bpl0[0], b1l = bpl1[0];
#pragma unroll
        for (int qq = 1; qq < 4; ++qq)
          if (qq == q) {
            b0h = bph0[qq]; b1h = bph1[qq]; b0l = bpl0[qq]; b1l = bpl1[qq];
          }
        uint32_t af[4];
        if (VB == 3) {
          // code pair P = 8 mv + g: word P / 5, codes (2j, 2j+1), j = P mod 5;
          // P >= 60: codes of the 8-code last word
          const int P = 8 * mv + g;
          const int wi = P < 60 ? P / 5 : 12;
          const int sh = P < 60 ? 6 * (P % 5) : 6 * (P - 60);
          const uint32_t wa = vc_s[ra * C::VW + wi] >> sh, wb2 = vc_s[(ra + 1) * C::VW + wi] >> sh;
          const uint32_t wc = vc_s[(ra + 8) * C::VW + wi] >> sh, wd = vc_s[(ra + 9) * C::VW + wi] >> sh;
          const uint32_t xab = __byte_perm(wa, wb2, 0x5410u), xcd = __byte_perm(wc, wd, 0x5410u);
          af[0] = hsub2u((xab & 0x00070007u) | kH1024, kH1024);
          af[1] = hsub2u(((xab >> 3) & 0x00070007u) | kH1024, kH1024);
          af[2] = hsub2u((xcd & 0x00070007u) | kH1024, kH1024);
          af[3] = hsub2u(((xcd >> 3) & 0x00070007u) | kH1024, kH1024);
        } else if (VB == 4) {
          const int u = g >> 2, i = g & 3;
          const int wi = q * (Gv / 8) + u * (Gv / 16) + l;
          const uint32_t wa = vc_s[ra * C::VW + wi], wb2 = vc_s[(ra + 1) * C::VW + wi];
          const uint32_t wc = vc_s[(ra + 8) * C::VW + wi], wd = vc_s[(ra + 9) * C::VW + wi];
          const uint32_t sel2 = (uint32_t)(i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12));
          const uint32_t xab = __byte_perm(wa, wb2, sel2), xcd = __byte_perm(wc, wd, sel2);
          if (C::VCB) {
            af[0] = cbl[(xab & 0xFu) | ((xab >> 12) & 0xF0u)];
            af[1] = cbl[((xab >> 4) & 0xFu) | ((xab >> 16) & 0xF0u)];
            af[2] = cbl[(xcd & 0xFu) | ((xcd >> 12) & 0xF0u)];
            af[3] = cbl[((xcd >> 4) & 0xFu) | ((xcd >> 16) & 0xF0u)];
          } else {
            af[0] = hsub2u((xab & 0x000F000Fu) | kH1024, kH1024);
            af[1] = hsub2u(((xab >> 4) & 0x000F000Fu) | kH1024, kH1024);
            af[2] = hsub2u((xcd & 0x000F000Fu) | kH1024, kH1024);
            af[3] = hsub2u(((xcd >> 4) & 0x000F000Fu) | kH1024, kH1024);
          }
        } else {
          const int u = g >> 1, bb = g & 1;
          const int wi = q * (Gv / 4) + u * (Gv / 16) + l;
          uint32_t wa = vc_s[ra * C::VW + wi], wb2 = vc_s[(ra + 1) * C::VW + wi];
          uint32_t wc = vc_s[(ra + 8) * C::VW + wi], wd = vc_s[(ra + 9) * C::VW + wi];
          if (C::VSYM) {
            wa ^= 0x80808080u;
            wb2 ^= 0x80808080u;
            wc ^= 0x80808080u;
            wd ^= 0x80808080u;
          }
          const uint32_t sel2 = (uint32_t)(bb | ((4 + bb) << 4) | ((bb + 2) << 8) | ((6 + bb) << 12));
          const uint32_t xab = __byte_perm(wa, wb2, sel2), xcd = __byte_perm(wc, wd, sel2);
          const uint32_t bias = C::VSYM ? kH1152 : kH1024;
          af[0] = hsub2u(__byte_perm(xab, 0x64646464u, 0x4140u), bias);
          af[1] = hsub2u(__byte_perm(xab, 0x64646464u, 0x4342u), bias);
          af[2] = hsub2u(__byte_perm(xcd, 0x64646464u, 0x4140u), bias);
          af[3] = hsub2u(__byte_perm(xcd, 0x64646464u, 0x4342u), bias);
        }
        mma16816(o[mv], af, b0h, b1h);
        mma16816(o[mv], af, b0l, b1l);
      }
    }

    __syncwarp();
    if (lane == 0 && ti + kStagesPerWarp < w_count) {
      fence_proxy_async_smem();
      issue(ti + kStagesPerWarp, s);
    }
  }
  if (failed && lane == 0) {
    raise_status(L.status, kStatusTimeout);
    for (int tj = ti; tj < w_count && tj < ti + kStagesPerWarp; ++tj)
      (void)mbar_wait_bounded(&wb[tj % kStagesPerWarp], (uint32_t)(tj / kStagesPerWarp) & 1u);
  }

  // ---- warp totals: l and the zero-point sums are spread over g ----------------
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, off);
    l1 += __shfl_xor_sync(kFull, l1, off);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      z0[q] += __shfl_xor_sync(kFull, z0[q], off);
      z1[q] += __shfl_xor_sync(kFull, z1[q], off);
    }
  }
  __syncthreads();  // stages are free: reuse them for the merge buffers
  float* my = mo + warp * 8 * kHeadDim;  // [8 heads][128]
#pragma unroll
  for (int mv = 0; mv < 8; ++mv) {
    const int q = mv >> mpg_log2, l = mv & (mpg - 1);
    int cg, cg8;
    if (VB == 3) {
      const int P = 8 * mv + g;
      cg = P < 60 ? 10 * (P / 5) + 2 * (P % 5) : 120 + 2 * (P - 60);
      cg8 = cg + 1;
    } else if (VB == 4) {
      const int u = g >> 2, i = g & 3;
      const int wi = q * (Gv / 8) + u * (Gv / 16) + l;
      cg = 8 * wi + 2 * i;
      cg8 = cg + 1;
    } else {
      const int u = g >> 1, bb = g & 1;
      const int wi = q * (Gv / 4) + u * (Gv / 16) + l;
      cg = 4 * wi + bb;
      cg8 = cg + 2;
    }
    float za0 = 0.0f, za1 = 0.0f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
      if (qq == q) {
        za0 = z0[qq];
        za1 = z1[qq];
      }
    my[(2 * t4) * kHeadDim + cg] = o[mv][0] + za0;
    my[(2 * t4 + 1) * kHeadDim + cg] = o[mv][1] + za1;
    my[(2 * t4) * kHeadDim + cg8] = o[mv][2] + za0;
    my[(2 * t4 + 1) * kHeadDim + cg8] = o[mv][3] + za1;
  }
  if (g == 0) {
    ml[(warp * 8 + 2 * t4) * 2] = w_count > 0 ? m0 : -INFINITY;
    ml[(warp * 8 + 2 * t4) * 2 + 1] = l0;
    ml[(warp * 8 + 2 * t4 + 1) * 2] = w_count > 0 ? m1 : -INFINITY;
    ml[(warp * 8 + 2 * t4 + 1) * 2 + 1] = l1;
  }
  __shared__ int any_failed;
  if (tid == 0) any_failed = 0;
  __syncthreads();
  if (failed && lane == 0) atomicOr(&any_failed, 1);
  __syncthreads();

  const int c = tid;
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[(w * 8 + h) * 2]);
    float ov = 0.0f, lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = ml[(w * 8 + h) * 2];
      const float wt = mw == -INFINITY ? 0.0f : exp2f(mw - M);
      ov = fmaf(wt, mo[(w * 8 + h) * kHeadDim + c], ov);
      lsum = fmaf(wt, ml[(w * 8 + h) * 2 + 1], lsum);
    }
    if (any_failed) {
      ov = NAN;
      lsum = NAN;
    }
    const int64_t prow = (int64_t)b * a.num_q_heads + hq0 + h;
    if (a.splits == 1) {
      const float res = finish_row(a.sink_part, prow, c, ov, M, lsum);
      if (a.out_dtype == KVQ_F32)
        reinterpret_cast<float*>(a.out)[prow * kHeadDim + c] = res;
      else
        reinterpret_cast<__half*>(a.out)[prow * kHeadDim + c] = __float2half_rn(res);
    } else {
      const int64_t r = prow * a.splits + split;
      a.part_o[r * kHeadDim + c] = ov;
      if (c == 0) {
        a.part_ml[r * 2] = M;
        a.part_ml[r * 2 + 1] = lsum;
      }
    }
  }
  if (a.splits > 1) merge_splits_if_last<kWarps>(L.counters + n, a, b * a.num_q_heads + hq0, G);
}

template <int KB, int KMODE, int VB, int VMODE, int FG = 0>
cudaError_t launch_t(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<KB, KMODE, VB, VMODE>;
  const size_t sm = C::smem_bytes();
  static SmemAttr attr;
  {
    const cudaError_t e = attr.ensure(decode_gqa_kernel<KB, KMODE, VB, VMODE, FG>, sm);
    if (e != cudaSuccess) return e;
  }
  if (a.occupancy_out)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        a.occupancy_out, decode_gqa_kernel<KB, KMODE, VB, VMODE, FG>, kThreads, sm);
  dim3 grid(a.splits, L.n_streams);
  decode_gqa_kernel<KB, KMODE, VB, VMODE, FG><<<grid, kThreads, sm, st>>>(L, a);
  return cudaGetLastError();
}

}  // namespace gqa
}  // namespace kvq
