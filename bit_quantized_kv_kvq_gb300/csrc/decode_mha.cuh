// Decode attention for one query head per kv-head (MHA) on the CUDA cores.
//
// Per CTA: one (batch, kv-head) stream and one split of its tokens. Each of
// the 4 warps owns a contiguous range of 32-token tiles and its own 2-deep
// ring of 1-D bulk copies (codes + scales of K and V for one tile), so the
// main loop has no block-wide barrier. Lane l handles channel quarter
// j = l & 3 (32 channels) of row r = l >> 2 of each 8-row group: it unpacks
// its codes to floats f = a + b * code (PRMT / shift into the mantissa of a
// fixed exponent), so
//   q.k   = sum_c (q_c s_c / b) f_c + sum_c q_c (z_c - (a/b) s_c)   (per-channel keys)
//   o_c  += (p_t s_t / b) f_tc, with sum_t p_t z_t and the a-offset applied once
// (the scale folding of the TurboQuant KV-cache page, demingchina.com/news/57821,
// §2.3: dequantization inside the attention products). Softmax runs in log2
// units with a lazily moved running max (rescale only when the max grows by
// more than 2^8), the four warps are merged by log-sum-exp at the end.
// Outliers (KVQuant page, cf-1.com/news/2306543, §2.2 item 3) add
// q_c (x - z_c) to a score and p_t (x - z_t) to the output.
#pragma once

#include "common.cuh"
#include "decode_merge.cuh"

namespace kvq {
namespace mha {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kRows = 32;          // rows per tile
constexpr int kStagesPerWarp = 2;
constexpr float kLazy = 8.0f;      // log2 headroom before the running max moves

template <int B>
struct Unpack;  // f = kA + kB * code (unsigned code)

template <>
struct Unpack<4> {
  static constexpr float kA = 0.5f, kB = 1.0f / 256.0f;
  static constexpr int kWordsPerQuarter = 4;  // 32 channels
  __device__ static __forceinline__ void run(const uint32_t (&w)[4], float (&f)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo = w[q] & 0x0F0F0F0Fu;
      const uint32_t hi = (w[q] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[8 * q + 2 * i] = __uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7054u | (i << 8)));
        f[8 * q + 2 * i + 1] = __uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7054u | (i << 8)));
      }
    }
  }
};

template <>
struct Unpack<8> {
  static constexpr float kA = 1.0f, kB = 1.0f / 256.0f;
  static constexpr int kWordsPerQuarter = 8;
  __device__ static __forceinline__ void run(const uint32_t (&w)[8], float (&f)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      f[4 * q + 0] = __uint_as_float(((w[q] << 15) & 0x007F8000u) | 0x3F800000u);
      f[4 * q + 1] = __uint_as_float(((w[q] << 7) & 0x007F8000u) | 0x3F800000u);
      f[4 * q + 2] = __uint_as_float(((w[q] >> 1) & 0x007F8000u) | 0x3F800000u);
      f[4 * q + 3] = __uint_as_float(((w[q] >> 9) & 0x007F8000u) | 0x3F800000u);
    }
  }
};

template <int KB, int KMODE, int VB, int VMODE, bool OUTL>
struct Cfg {
  static constexpr bool KCH = KMODE == KVQ_ASYM_PER_CHANNEL;
  static constexpr bool KSYM = KMODE == KVQ_SYM_PER_TOKEN;
  static constexpr bool VSYM = VMODE == KVQ_SYM_PER_TOKEN;
  static constexpr int KW = Pack<KB>::kWords, VW = Pack<VB>::kWords;
  static constexpr int KQW = Unpack<KB>::kWordsPerQuarter, VQW = Unpack<VB>::kWordsPerQuarter;
  static constexpr int KC_BYTES = kRows * KW * 4;
  static constexpr int VC_BYTES = kRows * VW * 4;
  static constexpr int META = 512;  // per tile, K and V each (groups of >= 32 channels)
  // outliers: columns and values of the tile's K and V rows (<= 8 per row)
  static constexpr int OUT_ONE = kRows * kMaxOutliers * 2;
  static constexpr int OUT_BYTES = OUTL ? 4 * OUT_ONE : 0;
  static constexpr int STAGE = KC_BYTES + VC_BYTES + 2 * META + OUT_BYTES;
  static constexpr size_t smem_bytes() {
    return (size_t)kWarps * kStagesPerWarp * STAGE + kHeadDim * 4 /*q*/ +
           (size_t)kWarps * kHeadDim * 4 * 2 /*o, ocorr*/ + kWarps * 2 * 4 /*m, l*/ +
           kWarps * kStagesPerWarp * 8 /*bars*/ + 16;
  }
};

template <int N>
__device__ __forceinline__ void lds_words(const uint32_t* p, uint32_t (&w)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + i);
    w[i] = v.x;
    w[i + 1] = v.y;
    w[i + 2] = v.z;
    w[i + 3] = v.w;
  }
}

template <int KB, int KMODE, int VB, int VMODE, bool OUTL>
__global__ void __launch_bounds__(kThreads, 4)
    decode_mha_kernel(LayerDev L, DecodeArgs a) {
  using C = Cfg<KB, KMODE, VB, VMODE, OUTL>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane & 3, r8 = lane >> 2;
  const int split = blockIdx.x, n = blockIdx.y;
  const int b = n / L.num_kv_heads;
  const int hq = n - b * L.num_kv_heads;  // one query head per kv-head

  unsigned char* stages = smem;
  float* qf = reinterpret_cast<float*>(smem + (size_t)kWarps * kStagesPerWarp * C::STAGE);
  float* mo = qf + kHeadDim;               // [warps][128]
  float* oc = mo + kWarps * kHeadDim;      // [warps][128] outlier corrections
  float* ml = oc + kWarps * kHeadDim;      // [warps][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ml + kWarps * 2);  // offset is a multiple of 16

  const int len = a.length, kq = a.k_quant_len;
  const int row_begin = split * a.tiles_per_split * kTile;
  const int row_end = min(row_begin + a.tiles_per_split * kTile, len);
  const int ntiles = (row_end - row_begin + kRows - 1) / kRows;
  const int per_warp = (ntiles + kWarps - 1) / kWarps;
  const int w_first = min(warp * per_warp, ntiles);
  const int w_count = min(per_warp, ntiles - w_first);
  const int Gk = L.k.group, Gv = L.v.group;
  const int kgpr = C::KCH ? 1 : kHeadDim / Gk;
  const int vgpr = kHeadDim / Gv;
  const int kout = L.outliers;

  const uint32_t* kcodes = L.k.codes + (int64_t)n * L.k.codes_sstride;
  const uint32_t* vcodes = L.v.codes + (int64_t)n * L.v.codes_sstride;
  const unsigned char* kmeta = L.k.meta + (int64_t)n * L.k.meta_sstride;
  const unsigned char* vmeta = L.v.meta + (int64_t)n * L.v.meta_sstride;
  float* myoc = oc + warp * kHeadDim;

  for (int i = tid; i < kHeadDim; i += kThreads)
    qf[i] = __half2float(a.q[((int64_t)b * a.num_q_heads + hq) * kHeadDim + i]) * a.scale_log2;
  for (int i = tid; i < kWarps * kHeadDim; i += kThreads) oc[i] = 0.0f;
  uint64_t* wb = bars + warp * kStagesPerWarp;
  if (lane == 0) {
    for (int s = 0; s < kStagesPerWarp; ++s) mbar_init(&wb[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  auto stage_ptr = [&](int s) { return stages + (size_t)(warp * kStagesPerWarp + s) * C::STAGE; };
  auto issue = [&](int ti, int s) {
    unsigned char* base = stage_ptr(s);
    const int t0 = row_begin + (w_first + ti) * kRows;
    const bool rt = C::KCH && t0 >= kq;
    const uint32_t kmb = C::KCH ? (uint32_t)(kHeadDim * 4) : (uint32_t)(kRows * kgpr * (C::KSYM ? 2 : 4));
    const uint32_t vmb = (uint32_t)(kRows * vgpr * (C::VSYM ? 2 : 4));
    const uint32_t ob = OUTL ? (uint32_t)(kRows * kout * 2) : 0u;  // one outlier array of the tile
    mbar_arrive_expect_tx(&wb[s], C::VC_BYTES + vmb + 2 * ob + (rt ? 0u : C::KC_BYTES + kmb + 2 * ob));
    if (!rt) {
      bulk_g2s(base, kcodes + (int64_t)t0 * C::KW, C::KC_BYTES, &wb[s]);
      const unsigned char* ks = C::KCH ? kmeta + (int64_t)(t0 / Gk) * kHeadDim * 4
                                       : kmeta + (int64_t)t0 * kgpr * (C::KSYM ? 2 : 4);
      bulk_g2s(base + C::KC_BYTES + C::VC_BYTES, ks, kmb, &wb[s]);
    }
    bulk_g2s(base + C::KC_BYTES, vcodes + (int64_t)t0 * C::VW, C::VC_BYTES, &wb[s]);
    bulk_g2s(base + C::KC_BYTES + C::VC_BYTES + C::META, vmeta + (int64_t)t0 * vgpr * (C::VSYM ? 2 : 4),
             vmb, &wb[s]);
    if (OUTL) {
      // every row holds exactly kout entries, so the tile's entries are contiguous
      unsigned char* ot = base + C::KC_BYTES + C::VC_BYTES + 2 * C::META;
      const int64_t e0 = (int64_t)t0 * kout;
      if (!rt) {
        bulk_g2s(ot, L.k.col + (int64_t)n * L.k.out_sstride + e0, ob, &wb[s]);
        bulk_g2s(ot + C::OUT_ONE, L.k.val + (int64_t)n * L.k.out_sstride + e0, ob, &wb[s]);
      }
      bulk_g2s(ot + 2 * C::OUT_ONE, L.v.col + (int64_t)n * L.v.out_sstride + e0, ob, &wb[s]);
      bulk_g2s(ot + 3 * C::OUT_ONE, L.v.val + (int64_t)n * L.v.out_sstride + e0, ob, &wb[s]);
    }
  };
  if (lane == 0)
    for (int s = 0; s < kStagesPerWarp && s < w_count; ++s) issue(s, s);

  // per-lane constants
  constexpr float KA = Unpack<KB>::kA, KBETA = Unpack<KB>::kB;
  constexpr float VA = Unpack<VB>::kA, VBETA = Unpack<VB>::kB;
  float qq[32];       // per-channel keys: q_c s_c / b (per block); else q_c / b
  float kcorr = 0.0f; // per-channel keys: sum_c q_c (z_c - (a/b) s_c) over the quarter
  float qsum = 0.0f;  // per-token keys: sum_c q_c over the quarter
  int cur_blk = -1;
  if (!C::KCH) {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float qv = qf[32 * j + k];
      qq[k] = qv * (1.0f / KBETA);
      qsum += qv;
    }
  }
  const float k0 = -(KA / KBETA + (C::KSYM ? 128.0f : 0.0f)) * qsum;  // per-token keys
  const int kgrp = C::KCH ? 0 : (32 * j) / Gk;
  const int vgrp = (32 * j) / Gv;

  float m_run = -INFINITY, l_run = 0.0f;
  float acc[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) acc[k] = 0.0f;
  float cb = 0.0f, zacc = 0.0f;

  bool failed = false;
  int ti = 0;
  for (; ti < w_count; ++ti) {
    const int s = ti % kStagesPerWarp;
    const uint32_t par = (uint32_t)(ti / kStagesPerWarp) & 1u;
    const int t0 = row_begin + (w_first + ti) * kRows;
    const bool rt = C::KCH && t0 >= kq;
    unsigned char* base = stage_ptr(s);
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(base);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(base + C::KC_BYTES);
    const unsigned char* km = base + C::KC_BYTES + C::VC_BYTES;
    const unsigned char* vm = km + C::META;
    if (!mbar_wait_bounded(&wb[s], par)) {
      failed = true;
      break;
    }
    __syncwarp();

    // ---- scores of the 32 rows (4 per lane) ------------------------------
    float sc[4];
    if (!rt) {
      if (C::KCH && (t0 / Gk) != cur_blk) {
        cur_blk = t0 / Gk;
        kcorr = 0.0f;
        const __half2* sz = reinterpret_cast<const __half2*>(km) + 32 * j;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 f2 = __half22float2(sz[k]);
          const float qv = qf[32 * j + k];
          qq[k] = qv * f2.x * (1.0f / KBETA);
          kcorr += qv * (f2.y - (KA / KBETA) * f2.x);
        }
      }
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int row = it * 8 + r8;
        uint32_t w[C::KQW];
        lds_words<C::KQW>(kc + row * C::KW + j * C::KQW, w);
        if (C::KSYM) {
#pragma unroll
          for (int q = 0; q < C::KQW; ++q) w[q] ^= 0x80808080u;
        }
        float f[32];
        Unpack<KB>::run(w, f);
        uint64_t dA = 0, dB = 0;  // (0.0f, 0.0f) pairs
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          dA = f2_fma(f2_pack(qq[k], qq[k + 1]), f2_pack(f[k], f[k + 1]), dA);
          dB = f2_fma(f2_pack(qq[k + 2], qq[k + 3]), f2_pack(f[k + 2], f[k + 3]), dB);
        }
        float a0, a1;
        f2_unpack(f2_add(dA, dB), a0, a1);
        float d = a0 + a1;
        if (C::KCH) {
          d += kcorr;
        } else if (C::KSYM) {
          const float st = __half2float(reinterpret_cast<const __half*>(km)[row * kgpr + kgrp]);
          d = (d + k0) * st;
        } else {
          const float2 sz = __half22float2(reinterpret_cast<const __half2*>(km)[row * kgpr + kgrp]);
          d = fmaf(d + k0, sz.x, qsum * sz.y);
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        sc[it] = (t0 + row < row_end) ? d : -INFINITY;
      }
    } else {
      const __half* res =
          L.k.resid + (int64_t)n * L.k.resid_sstride + (int64_t)(t0 - kq) * kHeadDim;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int row = it * 8 + r8;
        float d = 0.0f;
        if (t0 + row < row_end) {
          const uint4* p4 = reinterpret_cast<const uint4*>(res + (size_t)row * kHeadDim + 32 * j);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const uint4 u = p4[v4];
            const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 x = __half22float2(h[e]);
              d = fmaf(qf[32 * j + 8 * v4 + 2 * e], x.x, d);
              d = fmaf(qf[32 * j + 8 * v4 + 2 * e + 1], x.y, d);
            }
          }
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        sc[it] = (t0 + row < row_end) ? d : -INFINITY;
      }
    }

    // ---- key outliers: e_t += q_c (x - dequant(code 0)) -----------------------
    const uint16_t* ocol = reinterpret_cast<const uint16_t*>(base + C::KC_BYTES + C::VC_BYTES + 2 * C::META);
    const __half* oval = reinterpret_cast<const __half*>(ocol + C::OUT_ONE / 2);
    if (OUTL && !rt) {
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int lr = it * 8 + r8;
        float add = 0.0f;
        const int ke = (t0 + lr < row_end) ? kout : 0;  // rows past the end: no entries read
        for (int e = j; e < ke; e += 4) {
          const int c = ocol[lr * kout + e] & (kHeadDim - 1);
          const float x = __half2float(oval[lr * kout + e]);
          float z0 = 0.0f;
          if (C::KCH) z0 = __high2float(reinterpret_cast<const __half2*>(km)[c]);
          else if (!C::KSYM) z0 = __high2float(reinterpret_cast<const __half2*>(km)[lr * kgpr + c / Gk]);
          add = fmaf(qf[c], x - z0, add);
        }
        add += __shfl_xor_sync(0xffffffffu, add, 1);
        add += __shfl_xor_sync(0xffffffffu, add, 2);
        if (t0 + lr < row_end) sc[it] += add;
      }
    }

    // ---- online softmax (warp-local) ---------------------------------------
    float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
    if (mt > m_run + kLazy) {  // warp-uniform
      const float mnew = mt;
      const float alpha = exp2f(m_run - mnew);
      l_run *= alpha;
      cb *= alpha;
      zacc *= alpha;
      const uint64_t AL = f2_pack(alpha, alpha);
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const uint64_t A = f2_mul(AL, f2_pack(acc[k], acc[k + 1]));
        f2_unpack(A, acc[k], acc[k + 1]);
      }
      if (OUTL) {
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) myoc[lane + 32 * k] *= alpha;
        __syncwarp();
      }
      m_run = mnew;
    }
    float p[4];
    float ps = 0.0f;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      p[it] = exp2f(sc[it] - m_run);
      ps += p[it];
    }
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    l_run += ps;

    // ---- PV with the value scales folded into p ------------------------------
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int row = it * 8 + r8;
      uint32_t w[C::VQW];
      lds_words<C::VQW>(vc + row * C::VW + j * C::VQW, w);
      if (C::VSYM) {
#pragma unroll
        for (int q = 0; q < C::VQW; ++q) w[q] ^= 0x80808080u;
      }
      float st, zt = 0.0f;
      if (C::VSYM) {
        st = __half2float(reinterpret_cast<const __half*>(vm)[row * vgpr + vgrp]);
      } else {
        const float2 sz = __half22float2(reinterpret_cast<const __half2*>(vm)[row * vgpr + vgrp]);
        st = sz.x;
        zt = sz.y;
      }
      const float pb = p[it] * st * (1.0f / VBETA);
      cb += pb;
      if (!C::VSYM) zacc = fmaf(p[it], zt, zacc);
      float f[32];
      Unpack<VB>::run(w, f);
      const uint64_t PB = f2_pack(pb, pb);
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const uint64_t A = f2_fma(PB, f2_pack(f[k], f[k + 1]), f2_pack(acc[k], acc[k + 1]));
        f2_unpack(A, acc[k], acc[k + 1]);
      }
    }

    // ---- value outliers: o_c += p_t (x - dequant(code 0)) ----------------------
    if (OUTL) {
      const uint16_t* vcol = ocol + C::OUT_ONE;
      const __half* vval = reinterpret_cast<const __half*>(ocol + 3 * (C::OUT_ONE / 2));
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int lr = it * 8 + r8;
        if (t0 + lr < row_end) {
          for (int e = j; e < kout; e += 4) {
            const int c = vcol[lr * kout + e] & (kHeadDim - 1);
            const float x = __half2float(vval[lr * kout + e]);
            float z0 = 0.0f;
            if (!C::VSYM) z0 = __high2float(reinterpret_cast<const __half2*>(vm)[lr * vgpr + c / Gv]);
            atomicAdd(&myoc[c], p[it] * (x - z0));
          }
        }
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

  // ---- reduce the warp's rows: lanes with the same quarter j ------------------
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
    cb += __shfl_xor_sync(0xffffffffu, cb, off);
    zacc += __shfl_xor_sync(0xffffffffu, zacc, off);
  }
  // acc_c = sum_t pb_t (a + b n_tc) with pb = p s / b, so
  // sum_t p_t s_t n_tc = acc_c - a * cb; symmetric codes were offset by +128.
  const float off_c = VA * cb + (C::VSYM ? 128.0f * VBETA * cb : 0.0f);
  if (r8 == 0) {
#pragma unroll
    for (int k = 0; k < 32; ++k) mo[warp * kHeadDim + 32 * j + k] = (acc[k] - off_c) + zacc;
  }
  if (lane == 0) {
    ml[warp * 2] = w_count > 0 ? m_run : -INFINITY;
    ml[warp * 2 + 1] = l_run;
  }
  __shared__ int any_failed;
  if (tid == 0) any_failed = 0;
  __syncthreads();
  if (failed && lane == 0) atomicOr(&any_failed, 1);
  __syncthreads();

  // ---- merge the warps (log-sum-exp) and write the split's result -----------
  const int c = tid;  // kThreads == kHeadDim
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[2 * w]);
  float o = 0.0f, lsum = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float m_w = ml[2 * w];
    const float wt = m_w == -INFINITY ? 0.0f : exp2f(m_w - M);
    o = fmaf(wt, mo[w * kHeadDim + c] + oc[w * kHeadDim + c], o);
    lsum = fmaf(wt, ml[2 * w + 1], lsum);
  }
  const int64_t prow = (int64_t)b * a.num_q_heads + hq;
  if (any_failed) {
    o = NAN;
    lsum = NAN;
  }
  if (a.splits == 1) {
    const float res = finish_row(a.sink_part, prow, c, o, M, lsum);
    if (a.out_dtype == KVQ_F32)
      reinterpret_cast<float*>(a.out)[prow * kHeadDim + c] = res;
    else
      reinterpret_cast<__half*>(a.out)[prow * kHeadDim + c] = __float2half_rn(res);
  } else {
    const int64_t r = prow * a.splits + split;
    a.part_o[r * kHeadDim + c] = o;
    if (c == 0) {
      a.part_ml[r * 2] = M;
      a.part_ml[r * 2 + 1] = lsum;
    }
  }
  if (a.splits > 1) merge_splits_if_last<kWarps>(L.counters + n, a, (int64_t)b * a.num_q_heads + hq, 1);
}

template <int KB, int KMODE, int VB, int VMODE, bool OUTL>
cudaError_t launch_t(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<KB, KMODE, VB, VMODE, OUTL>;
  const size_t sm = C::smem_bytes();
  static SmemAttr attr;
  {
    const cudaError_t e = attr.ensure(decode_mha_kernel<KB, KMODE, VB, VMODE, OUTL>, sm);
    if (e != cudaSuccess) return e;
  }
  if (a.occupancy_out)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        a.occupancy_out, decode_mha_kernel<KB, KMODE, VB, VMODE, OUTL>, kThreads, sm);
  dim3 grid(a.splits, L.n_streams);
  decode_mha_kernel<KB, KMODE, VB, VMODE, OUTL><<<grid, kThreads, sm, st>>>(L, a);
  return cudaGetLastError();
}

}  // namespace mha
}  // namespace kvq
