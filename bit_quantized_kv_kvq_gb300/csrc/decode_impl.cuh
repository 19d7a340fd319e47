// Split-K decode attention over the packed cache, dequantizing in registers.
//
// Per CTA: one (batch, kv-head) stream, one split of its tokens, all query
// heads that share the kv-head (GQA). Packed K/V tiles of 64 tokens, their
// scales/zero points, are staged into shared memory by 1-D bulk copies
// (cp.async.bulk) on a 4-deep mbarrier ring; every wait is bounded.
//
// Per tile: QK^T on the codes with the scales folded into the query
// (per-channel keys: q'_c = q_c s_c and bias sum_c q_c z_c per block;
// per-token keys: score = s_t <q, codes> + z_t sum q), outlier corrections
// e_t += q_c (x_out - z) (KVQuant page, cf-1.com/news/2306543, §2.2 item 3:
// the dense and the sparse parts are combined), online softmax in log2
// units, then PV with the value scales folded into the probabilities
// (p'_t = p_t s_t, plus sum_t p_t z_t) and value outlier corrections.
// The cache is never expanded to fp16 in memory (TurboQuant KV-cache page,
// demingchina.com/news/57821, §2.3).
//
// Each CTA writes (m, l, o) partials; a combine kernel merges the splits by
// log-sum-exp.
#pragma once

#include "common.cuh"

namespace kvq {

constexpr int kDecThreads = 128;
constexpr int kStages = 4;
constexpr int kMetaMax = 2048;  // bytes of K or V metadata per stage, at most

template <int KB, int KMODE, int VB, int VMODE, int G>
struct DecodeCfg {
  using PK = Pack<KB>;
  using PV = Pack<VB>;
  static constexpr int WK = PK::kWords, WV = PV::kWords;
  static constexpr int CK = PK::kCpw, CV = PV::kCpw;
  static constexpr bool KCH = KMODE == KVQ_ASYM_PER_CHANNEL;
  static constexpr bool KCB = KMODE == KVQ_CODEBOOK_PER_TOKEN;  // codes index the codebook
  static constexpr bool VCB = VMODE == KVQ_CODEBOOK_PER_TOKEN;
  // scale-only groups (zero point 0): symmetric integer codes and codebook codes
  static constexpr bool KSYM = KMODE == KVQ_SYM_PER_TOKEN || KCB;
  static constexpr bool VSYM = VMODE == KVQ_SYM_PER_TOKEN || VCB;
  static constexpr int KMB = KSYM ? 2 : 4;
  static constexpr int VMB = VSYM ? 2 : 4;
  static constexpr int LPRK = WK > 16 ? 32 : 16;  // lanes per key row
  static constexpr int RPIK = 32 / LPRK;          // key rows per warp iteration
  static constexpr int LPRV = WV > 16 ? 32 : 16;  // threads per value row
  static constexpr int RGV = kDecThreads / LPRV;  // value row groups
  static constexpr int KC_BYTES = kTile * WK * 4;
  static constexpr int VC_BYTES = kTile * WV * 4;
  static constexpr int STAGE = KC_BYTES + VC_BYTES + 2 * kMetaMax;
  static constexpr size_t smem_bytes() {
    return (size_t)kStages * STAGE + (size_t)(3 * G * kHeadDim + 2 * G * kTile) * 4 +
           kStages * 8;
  }
};

// Exact float of the code in position k of word w (magic-number conversion:
// the code is placed in the mantissa of 2^23 and 2^23 is subtracted).
template <int B, bool SYM>
__device__ __forceinline__ float code_f(uint32_t w, int k) {
  if (SYM) {
    uint32_t u = ((w >> (8 * k)) & 0xFFu) ^ 0x80u;  // two's complement -> offset binary
    return __uint_as_float(0x4B000000u | u) - 8388736.0f;
  }
  uint32_t c = (w >> (B * k)) & ((1u << B) - 1u);
  return __uint_as_float(0x4B000000u | c) - 8388608.0f;
}

template <int LANES>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int off = 1; off < LANES; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <int KB, int KMODE, int VB, int VMODE, int G>
__global__ void __launch_bounds__(kDecThreads)
    decode_split_kernel(LayerDev L, DecodeArgs a) {
  using C = DecodeCfg<KB, KMODE, VB, VMODE, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, n = blockIdx.y;
  const int b = n / L.num_kv_heads;
  const int kvh = n - b * L.num_kv_heads;
  const int hq0 = kvh * G;

  float* qf = reinterpret_cast<float*>(smem + (size_t)kStages * C::STAGE);  // [G][128]
  float* sc = qf + G * kHeadDim;                                            // [G][64]
  float* pb = sc + G * kTile;                                               // [G][64]
  float* oc = pb + G * kTile;                                               // [G][128]
  float* ob = oc + G * kHeadDim;                                            // [G][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ob + G * kHeadDim);
  __shared__ float cbt[16];  // codebook levels (codebook codes only)
  if ((C::KCB || C::VCB) && tid < 16) cbt[tid] = __half2float(__ushort_as_half(L.codebook[tid]));

  const int len = a.varlen ? a.lens[b] : a.length, kq = a.k_quant_len;  // this batch row's tokens
  const int ntiles = (len + kTile - 1) / kTile;
  const int t_begin = split * a.tiles_per_split;
  const int t_end = min(t_begin + a.tiles_per_split, ntiles);
  const int nt = max(t_end - t_begin, 0);  // empty past a short batch row
  const int Gk = L.k.group, Gv = L.v.group;
  const int vgpr = kHeadDim / Gv;
  const int kgpr = C::KCH ? 1 : kHeadDim / Gk;
  const int kout = L.outliers;

  const uint32_t* kcodes = L.k.codes + (int64_t)n * L.k.codes_sstride;
  const uint32_t* vcodes = L.v.codes + (int64_t)n * L.v.codes_sstride;
  const unsigned char* kmeta = L.k.meta + (int64_t)n * L.k.meta_sstride;
  const unsigned char* vmeta = L.v.meta + (int64_t)n * L.v.meta_sstride;

  for (int i = tid; i < G * kHeadDim; i += kDecThreads) {
    const int h = i >> 7, c = i & 127;
    qf[i] = __half2float(a.q[((int64_t)b * a.num_q_heads + hq0 + h) * kHeadDim + c]) *
            a.scale_log2;
    oc[i] = 0.0f;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  auto stage_ptr = [&](int s) { return smem + (size_t)s * C::STAGE; };
  auto issue = [&](int tile, int s) {
    unsigned char* base = stage_ptr(s);
    const int t0 = tile * kTile;
    const bool rt = C::KCH && t0 >= kq;
    const uint32_t vmb = (uint32_t)(kTile * vgpr * C::VMB);
    const uint32_t kmb = C::KCH ? (uint32_t)(kHeadDim * 4) : (uint32_t)(kTile * kgpr * C::KMB);
    uint32_t bytes = C::VC_BYTES + vmb + (rt ? 0u : (uint32_t)C::KC_BYTES + kmb);
    mbar_arrive_expect_tx(&bars[s], bytes);
    if (!rt) {
      bulk_g2s(base, kcodes + (int64_t)t0 * C::WK, C::KC_BYTES, &bars[s]);
      const unsigned char* ksrc =
          C::KCH ? kmeta + (int64_t)(t0 / Gk) * kHeadDim * 4 : kmeta + (int64_t)t0 * kgpr * C::KMB;
      bulk_g2s(base + C::KC_BYTES + C::VC_BYTES + kMetaMax, ksrc, kmb, &bars[s]);
    }
    bulk_g2s(base + C::KC_BYTES, vcodes + (int64_t)t0 * C::WV, C::VC_BYTES, &bars[s]);
    bulk_g2s(base + C::KC_BYTES + C::VC_BYTES, vmeta + (int64_t)t0 * vgpr * C::VMB, vmb, &bars[s]);
  };

  if (tid == 0)
    for (int j = 0; j < kStages && j < nt; ++j) issue(t_begin + j, j);

  // key mapping: lane -> word jw of row (warp*16 + it*RPIK + rsub)
  const int jw = lane % C::LPRK;
  const int rsub = lane / C::LPRK;
  const bool wk_on = jw < C::WK;
  const int c0k = jw * C::CK;
  // value mapping: thread -> word jv of rows rgv, rgv + RGV, ...
  const int jv = tid % C::LPRV;
  const int rgv = tid / C::LPRV;
  const bool wv_on = jv < C::WV;
  const int c0v = jv * C::CV;
  const int vgrp = wv_on ? c0v / Gv : 0;

  float m_run[G], l_run[G], acc[G][C::CV], zacc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.0f;
    zacc[h] = 0.0f;
#pragma unroll
    for (int k = 0; k < C::CV; ++k) acc[h][k] = 0.0f;
  }

  bool failed = false;
  int j = 0;
  for (; j < nt; ++j) {
    const int s = j % kStages;
    const uint32_t par = (uint32_t)(j / kStages) & 1u;
    const int t0 = (t_begin + j) * kTile;
    const int nv = min(kTile, len - t0);
    const bool rt = C::KCH && t0 >= kq;
    unsigned char* base = stage_ptr(s);
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(base);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(base + C::KC_BYTES);
    const unsigned char* vm = base + C::KC_BYTES + C::VC_BYTES;
    const unsigned char* km = vm + kMetaMax;

    const bool ok = mbar_wait_bounded(&bars[s], par);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }

    // ---- (a) scores, log2 units -------------------------------------------
    if (!rt) {
      float qk[G][C::CK], bias[G], qsum[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        bias[h] = 0.0f;
        qsum[h] = 0.0f;
#pragma unroll
        for (int k = 0; k < C::CK; ++k) {
          const int c = c0k + k;
          const bool on = wk_on && c < kHeadDim;
          const float qv = on ? qf[h * kHeadDim + c] : 0.0f;
          if (C::KCH) {
            const __half2 sz = reinterpret_cast<const __half2*>(km)[on ? c : 0];
            qk[h][k] = qv * __low2float(sz);
            bias[h] += qv * __high2float(sz);
          } else {
            qk[h][k] = qv;
            qsum[h] += qv;
          }
        }
        if (C::KCH) bias[h] = group_sum<C::LPRK>(bias[h]);
      }
      const int kgrp = wk_on ? c0k / Gk : 0;
#pragma unroll 1
      for (int it = 0; it < 16 / C::RPIK; ++it) {
        const int row = warp * 16 + it * C::RPIK + rsub;
        const uint32_t w = wk_on ? kc[row * C::WK + jw] : 0u;
        float dot[G];
#pragma unroll
        for (int h = 0; h < G; ++h) dot[h] = 0.0f;
#pragma unroll
        for (int k = 0; k < C::CK; ++k) {
          const float f = C::KCB ? cbt[(w >> (4 * k)) & 15u] : code_f<KB, C::KSYM>(w, k);
#pragma unroll
          for (int h = 0; h < G; ++h) dot[h] += qk[h][k] * f;
        }
        if (!C::KCH) {
          if (C::KSYM) {
            const float st = __half2float(reinterpret_cast<const __half*>(km)[row * kgpr + kgrp]);
#pragma unroll
            for (int h = 0; h < G; ++h) dot[h] *= st;
          } else {
            const __half2 sz = reinterpret_cast<const __half2*>(km)[row * kgpr + kgrp];
            const float st = __low2float(sz), zt = __high2float(sz);
#pragma unroll
            for (int h = 0; h < G; ++h) dot[h] = dot[h] * st + qsum[h] * zt;
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float tot = group_sum<C::LPRK>(dot[h]);
          if (jw == 0) sc[h * kTile + row] = row < nv ? tot + bias[h] : -INFINITY;
        }
      }
    } else {
      const __half* res =
          L.k.resid + (int64_t)n * L.k.resid_sstride + (int64_t)(t0 - kq) * kHeadDim;
#pragma unroll 1
      for (int it = 0; it < 16; ++it) {
        const int row = warp * 16 + it;
        float dot[G];
#pragma unroll
        for (int h = 0; h < G; ++h) dot[h] = 0.0f;
        if (row < nv) {
          const uint2 raw = *reinterpret_cast<const uint2*>(res + (size_t)row * kHeadDim + 4 * lane);
          const __half2 x01 = *reinterpret_cast<const __half2*>(&raw.x);
          const __half2 x23 = *reinterpret_cast<const __half2*>(&raw.y);
          const float x[4] = {__low2float(x01), __high2float(x01), __low2float(x23),
                              __high2float(x23)};
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) dot[h] += qf[h * kHeadDim + 4 * lane + i] * x[i];
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float tot = group_sum<32>(dot[h]);
          if (lane == 0) sc[h * kTile + row] = row < nv ? tot : -INFINITY;
        }
      }
    }
    __syncthreads();

    // ---- (b) key outliers: e_t += q_c (x_out - dequant(code 0)) ------------
    if (kout > 0 && !rt) {
      if (tid < nv) {
        const int t = t0 + tid;
        const int32_t* rp = L.k.rowptr + (int64_t)n * L.k.rowptr_sstride;
        const int beg = rp[t], end = rp[t + 1];
        for (int e = beg; e < end; ++e) {
          const int64_t ei = (int64_t)n * L.k.out_sstride + e;
          const int c = L.k.col[ei];
          const float x = __half2float(L.k.val[ei]);
          float z0 = 0.0f;
          if (C::KCH) z0 = __high2float(reinterpret_cast<const __half2*>(km)[c]);
          else if (!C::KSYM) z0 = __high2float(reinterpret_cast<const __half2*>(km)[tid * kgpr + c / Gk]);
          const float d = x - z0;
#pragma unroll
          for (int h = 0; h < G; ++h) sc[h * kTile + tid] += qf[h * kHeadDim + c] * d;
        }
      }
      __syncthreads();
    }

    // ---- (c) online softmax ---------------------------------------------------
    float alpha[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float v0 = sc[h * kTile + lane], v1 = sc[h * kTile + lane + 32];
      float tmax = fmaxf(v0, v1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float mnew = fmaxf(m_run[h], tmax);
      alpha[h] = exp2f(m_run[h] - mnew);
      const float p0 = exp2f(v0 - mnew), p1 = exp2f(v1 - mnew);
      const float psum = group_sum<32>(p0 + p1);
      l_run[h] = l_run[h] * alpha[h] + psum;
      m_run[h] = mnew;
      if (warp == (h & 3)) {
        pb[h * kTile + lane] = p0;
        pb[h * kTile + lane + 32] = p1;
      }
      if (kout > 0) oc[h * kHeadDim + tid] *= alpha[h];
    }
    __syncthreads();

    // ---- (d) PV with folded value scales ------------------------------------
#pragma unroll
    for (int h = 0; h < G; ++h) {
      zacc[h] *= alpha[h];
#pragma unroll
      for (int k = 0; k < C::CV; ++k) acc[h][k] *= alpha[h];
    }
#pragma unroll 1
    for (int row = rgv; row < nv; row += C::RGV) {
      const uint32_t w = wv_on ? vc[row * C::WV + jv] : 0u;
      float st, zt = 0.0f;
      if (C::VSYM) {
        st = __half2float(reinterpret_cast<const __half*>(vm)[row * vgpr + vgrp]);
      } else {
        const __half2 sz = reinterpret_cast<const __half2*>(vm)[row * vgpr + vgrp];
        st = __low2float(sz);
        zt = __high2float(sz);
      }
      float f[C::CV];
#pragma unroll
      for (int k = 0; k < C::CV; ++k) f[k] = C::VCB ? cbt[(w >> (4 * k)) & 15u] : code_f<VB, C::VSYM>(w, k);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pv = pb[h * kTile + row];
        const float ps = pv * st;
        if (!C::VSYM) zacc[h] += pv * zt;
#pragma unroll
        for (int k = 0; k < C::CV; ++k) acc[h][k] += ps * f[k];
      }
    }
    if (kout > 0 && tid < nv) {
      const int t = t0 + tid;
      const int32_t* rp = L.v.rowptr + (int64_t)n * L.v.rowptr_sstride;
      const int beg = rp[t], end = rp[t + 1];
      for (int e = beg; e < end; ++e) {
        const int64_t ei = (int64_t)n * L.v.out_sstride + e;
        const int c = L.v.col[ei];
        const float x = __half2float(L.v.val[ei]);
        float z0 = 0.0f;
        if (!C::VSYM) z0 = __high2float(reinterpret_cast<const __half2*>(vm)[tid * vgpr + c / Gv]);
        const float d = x - z0;
#pragma unroll
        for (int h = 0; h < G; ++h) atomicAdd(&oc[h * kHeadDim + c], pb[h * kTile + tid] * d);
      }
    }
    __syncthreads();
    if (tid == 0 && j + kStages < nt) {
      fence_proxy_async_smem();
      issue(t_begin + j + kStages, s);
    }
  }

  const int64_t prow0 = (int64_t)b * a.num_q_heads + hq0;
  if (failed) {
    // give the copies still in flight a bounded chance to land, then report
    if (tid == 0) {
      raise_status(L.status, kStatusTimeout);
      for (int jj = j; jj < nt && jj < j + kStages; ++jj)
        (void)mbar_wait_bounded(&bars[jj % kStages], (uint32_t)(jj / kStages) & 1u);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int64_t r = (prow0 + h) * a.splits + split;
      a.part_o[r * kHeadDim + tid] = NAN;
      if (tid == 0) {
        a.part_ml[r * 2] = 0.0f;
        a.part_ml[r * 2 + 1] = NAN;
      }
    }
    __syncthreads();
    return;
  }

  // ---- reduce the value accumulators over row groups and write partials -----
  for (int i = tid; i < G * kHeadDim; i += kDecThreads) ob[i] = 0.0f;
  __syncthreads();
  if (wv_on) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int k = 0; k < C::CV; ++k) {
        const int c = c0v + k;
        if (c < kHeadDim) atomicAdd(&ob[h * kHeadDim + c], acc[h][k] + zacc[h]);
      }
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int64_t r = (prow0 + h) * a.splits + split;
    a.part_o[r * kHeadDim + tid] = ob[h * kHeadDim + tid] + oc[h * kHeadDim + tid];
    if (tid == h) {
      a.part_ml[r * 2] = m_run[h];
      a.part_ml[r * 2 + 1] = l_run[h];
    }
  }
}

template <int KB, int KMODE, int VB, int VMODE, int G>
cudaError_t launch_decode_t(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  using C = DecodeCfg<KB, KMODE, VB, VMODE, G>;
  const size_t sm = C::smem_bytes();
  static SmemAttr attr;
  {
    const cudaError_t e = attr.ensure(decode_split_kernel<KB, KMODE, VB, VMODE, G>, sm);
    if (e != cudaSuccess) return e;
  }
  if (a.occupancy_out)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        a.occupancy_out, decode_split_kernel<KB, KMODE, VB, VMODE, G>, kDecThreads, sm);
  dim3 grid(a.splits, L.n_streams);
  decode_split_kernel<KB, KMODE, VB, VMODE, G><<<grid, kDecThreads, sm, st>>>(L, a);
  return cudaGetLastError();
}

// Dispatch over the supported (key codec, value codec) pairs for one G.
template <int G>
cudaError_t launch_decode_g(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  const int km = L.k.mode, kb = L.k.bits, vm = L.v.mode, vb = L.v.bits;
  if (km == KVQ_SYM_PER_TOKEN && vm == KVQ_SYM_PER_TOKEN)
    return launch_decode_t<8, KVQ_SYM_PER_TOKEN, 8, KVQ_SYM_PER_TOKEN, G>(L, a, st);
  if (km == KVQ_CODEBOOK_PER_TOKEN && vm == KVQ_CODEBOOK_PER_TOKEN)
    return launch_decode_t<4, KVQ_CODEBOOK_PER_TOKEN, 4, KVQ_CODEBOOK_PER_TOKEN, G>(L, a, st);
  if (vm != KVQ_ASYM_PER_TOKEN || km == KVQ_SYM_PER_TOKEN) return cudaErrorNotSupported;
#define KVQ_V(KB_, KM_)                                                                    \
  switch (vb) {                                                                            \
    case 3: return launch_decode_t<KB_, KM_, 3, KVQ_ASYM_PER_TOKEN, G>(L, a, st);          \
    case 4: return launch_decode_t<KB_, KM_, 4, KVQ_ASYM_PER_TOKEN, G>(L, a, st);          \
    default: return launch_decode_t<KB_, KM_, 8, KVQ_ASYM_PER_TOKEN, G>(L, a, st);         \
  }
  if (km == KVQ_ASYM_PER_CHANNEL) {
    switch (kb) {
      case 3: KVQ_V(3, KVQ_ASYM_PER_CHANNEL)
      case 4: KVQ_V(4, KVQ_ASYM_PER_CHANNEL)
      default: KVQ_V(8, KVQ_ASYM_PER_CHANNEL)
    }
  }
  switch (kb) {
    case 3: KVQ_V(3, KVQ_ASYM_PER_TOKEN)
    case 4: KVQ_V(4, KVQ_ASYM_PER_TOKEN)
    default: KVQ_V(8, KVQ_ASYM_PER_TOKEN)
  }
#undef KVQ_V
}

cudaError_t launch_decode_g1(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_g2(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_g4(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_g8(const LayerDev& L, const DecodeArgs& a, cudaStream_t st);

}  // namespace kvq
