// Prefill attention over the quantized cache: the queries of the last C
// cached positions of a layer (the chunk just quantized into the cache)
// attend, causally, the cache as the decode sees it -- fp16 sink tokens,
// dequantized codes with their outliers, fp16 residual keys (NIAH q8_0
// page, cf-1.com/news/5482713, §4.2: the prefill's time to first token; the
// KVQuant page, cf-1.com/news/2306543, §3.4: attention runs on the
// dequantized cache). Query i sits at position length - C + i and attends
// tokens 0 .. length - C + i.
//
// This is a dense contraction (C x G query rows against every visible token)
// and runs on the tensor cores as flash attention: per CTA 128 (position,
// head) rows of one (batch, kv-head) stream, 16 per warp, over key/value
// tiles of 64 tokens. The CTA dequantizes each tile once into shared memory
// as fp16 pairs x = hi + lo (about 22 bits, x formed in fp32 from the codes,
// scales and zero points), so one kernel serves every codec. Then
//   S = Q (Khi + Klo)^T                 two m16n8k16 products per fragment
//   O += (Phi + Plo)(Vhi + Vlo), less Plo Vlo     three products
// with fp32 accumulation and an exact online softmax in log2 units.
// Dequantization is pipelined: the tile buffers are double, and while the
// warps compute on one tile each thread holds the next tile's packed codes
// and scales in registers (loaded before the products), converting them
// into the other buffer afterwards. Tiles that hold fp16 rows (sinks,
// residual keys) or outliers take a direct path.
#include <cstdint>

#include "common.cuh"
#include "kvq_internal.h"
#include "mma_frag.cuh"

namespace kvq {
namespace pa {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kRowsCta = 16 * kWarps;  // (position, head) rows per CTA
constexpr int kTT = 64;                // tokens per tile
constexpr int kLd = kHeadDim + 8;      // shared row stride in halves (272 B: ldmatrix rows on distinct banks)
constexpr size_t kSmemBytes = (size_t)(kRowsCta + 8 * kTT) * kLd * 2;  // queries + two tile buffers

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// The code words holding channels c0 .. c0 + 7 (c0 a multiple of 8) of a
// packed row of `bits`-bit codes, and the eight codes taken out of them.
__device__ __forceinline__ void load_words(const uint32_t* row, int bits, int c0, uint32_t (&w)[2]) {
  if (bits == 4) {
    w[0] = __ldg(row + (c0 >> 3));
    w[1] = 0u;
  } else if (bits == 8) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + (c0 >> 2)));
    w[0] = u.x;
    w[1] = u.y;
  } else {  // ten per word: channels c0 .. c0 + 7 lie in words c0 / 10 and (c0 + 7) / 10
    const int w0 = c0 / 10;
    w[0] = __ldg(row + w0);
    w[1] = (c0 + 7) / 10 > w0 ? __ldg(row + w0 + 1) : 0u;
  }
}

__device__ __forceinline__ void extract8(const uint32_t (&w)[2], int bits, int c0, uint32_t (&c)[8]) {
  if (bits == 4) {
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = (w[0] >> (4 * j)) & 15u;
  } else if (bits == 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = ((j < 4 ? w[0] : w[1]) >> (8 * (j & 3))) & 255u;
  } else {
    const int w0 = c0 / 10;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int cj = c0 + j, wj = cj / 10;
      c[j] = ((wj > w0 ? w[1] : w[0]) >> (3 * (cj - 10 * wj))) & 7u;
    }
  }
}

// x = code * s + z per channel (per-channel keys: mch holds the eight
// channels' (s, z)), per token group (asymmetric: mtok = (s, z)), signed
// code * s (symmetric) or level[code] * s (codebook), in fp32.
__device__ __forceinline__ void decode8(int mode, const uint32_t (&c)[8], uint32_t mtok, const uint32_t (&mch)[8],
                                        const float* cbt, float (&x)[8]) {
  if (mode == KVQ_ASYM_PER_CHANNEL) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&mch[j]));
      x[j] = fmaf((float)c[j], f.x, f.y);
    }
  } else if (mode == KVQ_ASYM_PER_TOKEN) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&mtok));
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = fmaf((float)c[j], f.x, f.y);
  } else {
    const float sc = __half2float(__ushort_as_half((unsigned short)(mtok & 0xFFFFu)));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float v = mode == KVQ_CODEBOOK_PER_TOKEN ? cbt[c[j] & 15u] : (float)(int)(int8_t)(uint8_t)c[j];
      x[j] = v * sc;
    }
  }
}

// Scale word of coded row r for channels c0 .. (per-token groups; the
// scale alone in the low half for scale-only groups).
__device__ __forceinline__ uint32_t token_meta(const TensorDev& T, const unsigned char* meta, int r, int c0) {
  const int gi = r * (kHeadDim / T.group) + c0 / T.group;  // c0 .. c0 + 7 share a group (G >= 16)
  return T.meta_bytes == 4 ? __ldg(reinterpret_cast<const uint32_t*>(meta) + gi)
                           : (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(meta) + gi);
}

__device__ __forceinline__ void channel_meta(const unsigned char* meta, int blk, int c0, uint32_t (&m)[8]) {
  const uint4* p = reinterpret_cast<const uint4*>(meta + ((int64_t)blk * kHeadDim + c0) * 4);
  const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
  m[0] = u0.x; m[1] = u0.y; m[2] = u0.z; m[3] = u0.w;
  m[4] = u1.x; m[5] = u1.y; m[6] = u1.z; m[7] = u1.w;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Asks L2 for the packed rows, scales and outliers of cached tokens
// t0 .. t0 + 63 of stream n (thread `tid` of the CTA takes a few lines).
__device__ __forceinline__ void prefetch_tile(const LayerDev& L, int n, int t0, int length, int sink_len, int tid) {
  const int r0 = max(t0 - sink_len, 0), r1 = min(t0 + kTT, length) - sink_len;  // coded rows [r0, r1)
  if (r1 <= r0) return;
  const TensorDev* Ts[2] = {&L.k, &L.v};
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const TensorDev& T = *Ts[which];
    const unsigned char* codes = reinterpret_cast<const unsigned char*>(T.codes + (int64_t)n * T.codes_sstride);
    const int64_t cb0 = (int64_t)r0 * T.words * 4, cb1 = (int64_t)r1 * T.words * 4;
    for (int64_t o = cb0 + 128 * (int64_t)(tid & 127); o < cb1; o += 128 * 128)
      if ((tid >> 7) == which) prefetch_l2(codes + o);
    if (tid == 128 * which + 127) {
      const unsigned char* meta = T.meta + (int64_t)n * T.meta_sstride;
      if (T.mode == KVQ_ASYM_PER_CHANNEL)
        prefetch_l2(meta + (int64_t)(r0 / T.group) * kHeadDim * 4);
      else
        prefetch_l2(meta + (int64_t)r0 * (kHeadDim / T.group) * T.meta_bytes);
    }
  }
}

// Eight channels c0 .. c0 + 7 of cached token `tok` of stream n, in fp32.
template <bool IS_K>
__device__ __forceinline__ void dequant8(const LayerDev& L, int n, int tok, int c0, int length, int sink_len, int kq,
                                         const float* cbt, float (&x)[8]) {
  const bool is_k = IS_K;
  const TensorDev& T = IS_K ? L.k : L.v;
  const __half* src = nullptr;  // fp16 row (sinks, residual keys)
  if (tok >= length) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    return;
  }
  if (tok < sink_len) {
    src = (is_k ? L.sink_k : L.sink_v) + ((int64_t)n * L.sink_tokens + tok) * kHeadDim + c0;
  } else if (is_k && T.mode == KVQ_ASYM_PER_CHANNEL && tok - sink_len >= kq) {
    src = T.resid + (int64_t)n * T.resid_sstride + (int64_t)(tok - sink_len - kq) * kHeadDim + c0;
  }
  if (src) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(h[j]);
      x[2 * j] = f.x;
      x[2 * j + 1] = f.y;
    }
    return;
  }
  const int r = tok - sink_len;  // coded row
  const unsigned char* meta = T.meta + (int64_t)n * T.meta_sstride;
  uint32_t w[2], c[8], mch[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u}, mtok = 0u;
  load_words(T.codes + (int64_t)n * T.codes_sstride + (int64_t)r * T.words, T.bits, c0, w);
  if (T.mode == KVQ_ASYM_PER_CHANNEL)
    channel_meta(meta, r / T.group, c0, mch);
  else
    mtok = token_meta(T, meta, r, c0);
  extract8(w, T.bits, c0, c);
  decode8(T.mode, c, mtok, mch, cbt, x);
  if (L.outliers > 0) {  // every coded row holds exactly `outliers` entries
    const int64_t e0 = (int64_t)n * T.out_sstride + (int64_t)r * L.outliers;
    for (int e = 0; e < L.outliers; ++e) {
      const int cc = (int)(__ldg(T.col + e0 + e) & (kHeadDim - 1)) - c0;
      if (cc >= 0 && cc < 8) {
        const float v = __half2float(__ldg(T.val + e0 + e));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j == cc) x[j] = v;
      }
    }
  }
}

__device__ __forceinline__ uint4 split8(const float (&x)[8], uint4& lo) {
  uint4 hi;
  hi.x = tc::split_pair(x[0], x[1], lo.x);
  hi.y = tc::split_pair(x[2], x[3], lo.y);
  hi.z = tc::split_pair(x[4], x[5], lo.z);
  hi.w = tc::split_pair(x[6], x[7], lo.w);
  return hi;
}

// A tile whose 64 tokens are all coded rows held as codes, with at most
// kMaxFastOutliers outliers per row (OUTL) or none, in one key block: its
// packed data can be loaded ahead.
constexpr int kMaxFastOutliers = 2;

template <bool OUTL>
__device__ __forceinline__ bool fast_tile(const LayerDev& L, int t0, int length, int sink_len, int kq) {
  if ((OUTL ? L.outliers > kMaxFastOutliers : L.outliers > 0) || t0 < sink_len || t0 + kTT > length) return false;
  if (L.k.mode == KVQ_ASYM_PER_CHANNEL) {
    const int r0 = t0 - sink_len, r1 = r0 + kTT - 1;
    if (r1 >= kq || r0 / L.k.group != r1 / L.k.group) return false;
  }
  return true;
}

// The thread's packed data of a fast tile: four (token, 8-channel) units of
// K and of V (tokens (tid >> 4) + 16 k, channels 8 (tid & 15) ..).
template <bool OUTL>
struct Raw {
  uint32_t kw[4][2], vw[4][2];  // code words
  uint32_t km[4], vm[4];        // per-token scale words
  uint32_t kch[8];              // per-channel key (s, z) of the eight channels (one block)
  // outliers of each unit's row: columns and fp16 values, two per word
  uint32_t kc[OUTL ? 4 : 1], kv[OUTL ? 4 : 1], vc[OUTL ? 4 : 1], vv[OUTL ? 4 : 1];
};

// Outlier slots of a unit (channels c0 .. c0 + 7) from its row's packed
// columns and values (at most two per row).
__device__ __forceinline__ void apply_outliers(float (&x)[8], uint32_t cols, uint32_t vals, int kout, int c0) {
#pragma unroll
  for (int e = 0; e < kMaxFastOutliers; ++e) {
    if (e >= kout) break;
    const int cc = (int)((cols >> (16 * e)) & (kHeadDim - 1)) - c0;
    const float v = __half2float(__ushort_as_half((unsigned short)(vals >> (16 * e))));
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j == cc) x[j] = v;
  }
}

// Packed outlier columns and values (two per word) of coded row r.
__device__ __forceinline__ void row_outliers(const TensorDev& T, int n, int r, int kout, uint32_t& cols,
                                             uint32_t& vals) {
  const int64_t e0 = (int64_t)n * T.out_sstride + (int64_t)r * kout;
  if (kout == 2) {  // e0 is even: four-byte aligned pairs
    cols = __ldg(reinterpret_cast<const uint32_t*>(T.col + e0));
    vals = __ldg(reinterpret_cast<const uint32_t*>(T.val + e0));
  } else {
    cols = __ldg(T.col + e0);
    vals = __half_as_ushort(__ldg(T.val + e0));
  }
}

template <bool OUTL>
__global__ void __launch_bounds__(kThreads, 1) prefill_attn_kernel(const LayerDev L, const PrefillAttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __half* qs = reinterpret_cast<__half*>(smem);   // [128][kLd]
  __half* tiles = qs + kRowsCta * kLd;             // [2 buffers][khi, klo, vhi, vlo][64][kLd]
  __shared__ float cbt[16];
  auto tb = [&](int buf, int which) { return tiles + (size_t)(4 * buf + which) * kTT * kLd; };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int n = blockIdx.y;
  const int b = n / L.num_kv_heads, kvh = n - b * L.num_kv_heads;
  const int G = a.G;
  const int rows_total = a.chunk * G;
  const int R0 = blockIdx.x * kRowsCta;
  // this batch row's tokens (variable lengths: its own, with its own key blocks; no sinks)
  const int length = a.varlen ? a.lens[b] : a.length;
  const int kq = a.varlen ? length / L.k.group * L.k.group : a.kq;
  const int first_pos = length - a.chunk;  // position of query 0
  const int ut = tid >> 4, uc = 8 * (tid & 15);  // the thread's units: tokens ut + 16 k, channels uc ..

  for (int idx = tid; idx < kRowsCta * 16; idx += kThreads) {
    const int r = idx >> 4, part = idx & 15;
    const int R = R0 + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (R < rows_total) {
      const int i = R / G, h = R - i * G;
      v = __ldg(reinterpret_cast<const uint4*>(
          a.q + (((int64_t)b * a.chunk + i) * a.num_q_heads + kvh * G + h) * kHeadDim + 8 * part));
    }
    *reinterpret_cast<uint4*>(qs + r * kLd + 8 * part) = v;
  }
  if (tid < 16) cbt[tid] = __half2float(__ushort_as_half(L.codebook[tid]));

  // positions of the thread's rows g and g + 8 (rows past the chunk attend
  // the whole cache and are not stored)
  const int Rw = R0 + 16 * warp;
  auto pos_of = [&](int R) { return R < rows_total ? first_pos + R / G : length - 1; };
  const int pos0 = pos_of(Rw + g), pos1 = pos_of(Rw + g + 8);
  const int warp_pos_max = Rw < rows_total ? pos_of(min(Rw + 15, rows_total - 1)) : -1;  // -1: no rows
  const int last_R = min(R0 + kRowsCta, rows_total) - 1;
  const int n_tiles = (first_pos + last_R / G) / kTT + 1;

  // direct dequantization of the tile at t0 into buffer buf
  auto dequant_tile = [&](int t0, int buf) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = ut + 16 * k;
      float x[8];
      dequant8<true>(L, n, t0 + t, uc, length, a.sink_len, kq, cbt, x);
      uint4 lo;
      const uint4 hi = split8(x, lo);
      *reinterpret_cast<uint4*>(tb(buf, 0) + t * kLd + uc) = hi;
      *reinterpret_cast<uint4*>(tb(buf, 1) + t * kLd + uc) = lo;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = ut + 16 * k;
      float x[8];
      dequant8<false>(L, n, t0 + t, uc, length, a.sink_len, kq, cbt, x);
      uint4 lo;
      const uint4 hi = split8(x, lo);
      *reinterpret_cast<uint4*>(tb(buf, 2) + t * kLd + uc) = hi;
      *reinterpret_cast<uint4*>(tb(buf, 3) + t * kLd + uc) = lo;
    }
  };
  const uint32_t* kcodes = L.k.codes + (int64_t)n * L.k.codes_sstride;
  const uint32_t* vcodes = L.v.codes + (int64_t)n * L.v.codes_sstride;
  const unsigned char* kmeta = L.k.meta + (int64_t)n * L.k.meta_sstride;
  const unsigned char* vmeta = L.v.meta + (int64_t)n * L.v.meta_sstride;
  auto load_raw = [&](int t0, Raw<OUTL>& w) {
    const int r0 = t0 - a.sink_len;
    if (L.k.mode == KVQ_ASYM_PER_CHANNEL) channel_meta(kmeta, r0 / L.k.group, uc, w.kch);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = r0 + ut + 16 * k;
      load_words(kcodes + (int64_t)r * L.k.words, L.k.bits, uc, w.kw[k]);
      load_words(vcodes + (int64_t)r * L.v.words, L.v.bits, uc, w.vw[k]);
      w.km[k] = L.k.mode == KVQ_ASYM_PER_CHANNEL ? 0u : token_meta(L.k, kmeta, r, uc);
      w.vm[k] = token_meta(L.v, vmeta, r, uc);
      if (OUTL) {
        row_outliers(L.k, n, r, L.outliers, w.kc[k], w.kv[k]);
        row_outliers(L.v, n, r, L.outliers, w.vc[k], w.vv[k]);
      }
    }
  };
  auto convert_raw = [&](const Raw<OUTL>& w, int buf) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = ut + 16 * k;
      uint32_t c[8];
      float x[8];
      uint4 lo, hi;
      extract8(w.kw[k], L.k.bits, uc, c);
      decode8(L.k.mode, c, w.km[k], w.kch, cbt, x);
      if (OUTL) apply_outliers(x, w.kc[k], w.kv[k], L.outliers, uc);
      hi = split8(x, lo);
      *reinterpret_cast<uint4*>(tb(buf, 0) + t * kLd + uc) = hi;
      *reinterpret_cast<uint4*>(tb(buf, 1) + t * kLd + uc) = lo;
      extract8(w.vw[k], L.v.bits, uc, c);
      decode8(L.v.mode, c, w.vm[k], w.kch, cbt, x);  // per-token values: the channel words are unused
      if (OUTL) apply_outliers(x, w.vc[k], w.vv[k], L.outliers, uc);
      hi = split8(x, lo);
      *reinterpret_cast<uint4*>(tb(buf, 2) + t * kLd + uc) = hi;
      *reinterpret_cast<uint4*>(tb(buf, 3) + t * kLd + uc) = lo;
    }
  };

  __syncthreads();  // cbt
  dequant_tile(0, 0);

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  const uint32_t qbase = smem_u32(qs + (16 * warp + (lane & 15)) * kLd + 8 * (lane >> 4));

  Raw<OUTL> raw;
  for (int tile = 0; tile < n_tiles; ++tile) {
    const int t0 = tile * kTT, buf = tile & 1;
    // buffer buf holds this tile; every warp is done with the other one
    __syncthreads();
    const int tn = t0 + kTT;
    const bool more = tile + 1 < n_tiles;
    const bool nfast = more && fast_tile<OUTL>(L, tn, length, a.sink_len, kq);
    if (nfast)
      load_raw(tn, raw);  // in flight during the products
    else if (more)
      prefetch_tile(L, n, tn, length, a.sink_len, tid);

    if (t0 <= warp_pos_max) {  // some token of the tile is visible to the warp's rows
      const __half* khi = tb(buf, 0);
      const __half* klo = tb(buf, 1);
      const __half* vhi = tb(buf, 2);
      const __half* vlo = tb(buf, 3);
      // ---- S = Q K^T (n-tile nt: tokens 8 nt .. 8 nt + 7) ----
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] = 0.0f;
      {
        const int trow = (lane & 7) + ((lane >> 4) << 3), tcol = ((lane >> 3) & 1) * 8;
        const uint32_t bh = smem_u32(khi + trow * kLd + tcol), bl = smem_u32(klo + trow * kLd + tcol);
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
          uint32_t qa[4];
          ldsm_x4(qbase + 32u * kc, qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            const uint32_t off = (uint32_t)(16 * np * kLd + 16 * kc) * 2u;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(bh + off, b0, b1, b2, b3);
            tc::mma(s[2 * np], qa[0], qa[1], qa[2], qa[3], b0, b1);
            tc::mma(s[2 * np + 1], qa[0], qa[1], qa[2], qa[3], b2, b3);
            ldsm_x4(bl + off, b0, b1, b2, b3);
            tc::mma(s[2 * np], qa[0], qa[1], qa[2], qa[3], b0, b1);
            tc::mma(s[2 * np + 1], qa[0], qa[1], qa[2], qa[3], b2, b3);
          }
        }
      }

      // ---- scale, causal mask, online softmax (rows g: e = 0, 1; g + 8: e = 2, 3) ----
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = t0 + 8 * nt + 2 * t4 + (e & 1);
          const float v = (tok <= (e < 2 ? pos0 : pos1)) ? s[nt][e] * a.scale_log2 : -INFINITY;
          s[nt][e] = v;
          if (e < 2)
            mx0 = fmaxf(mx0, v);
          else
            mx1 = fmaxf(mx1, v);
        }
      mx0 = fmaxf(mx0, __shfl_xor_sync(tc::kFull, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(tc::kFull, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(tc::kFull, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(tc::kFull, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: token 0 is in every row's first tile
      const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= al0;
        o[j][1] *= al0;
        o[j][2] *= al1;
        o[j][3] *= al1;
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - mn0);
        s[nt][1] = exp2f(s[nt][1] - mn0);
        s[nt][2] = exp2f(s[nt][2] - mn1);
        s[nt][3] = exp2f(s[nt][3] - mn1);
        l0 += s[nt][0] + s[nt][1];
        l1 += s[nt][2] + s[nt][3];
      }

      // ---- O += P V (k-chunk kk: tokens 16 kk .. 16 kk + 15) ----
      {
        const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = (lane >> 4) * 8;
        const uint32_t vh = smem_u32(vhi + vrow * kLd + vcol), vl = smem_u32(vlo + vrow * kLd + vcol);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t ph[4], pl[4];
          ph[0] = tc::split_pair(s[2 * kk][0], s[2 * kk][1], pl[0]);
          ph[1] = tc::split_pair(s[2 * kk][2], s[2 * kk][3], pl[1]);
          ph[2] = tc::split_pair(s[2 * kk + 1][0], s[2 * kk + 1][1], pl[2]);
          ph[3] = tc::split_pair(s[2 * kk + 1][2], s[2 * kk + 1][3], pl[3]);
#pragma unroll
          for (int nc = 0; nc < 8; ++nc) {
            const uint32_t off = (uint32_t)(16 * kk * kLd + 16 * nc) * 2u;
            uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
            ldsm_x4_t(vh + off, b0, b1, b2, b3);
            ldsm_x4_t(vl + off, c0, c1, c2, c3);
            tc::mma(o[2 * nc], ph[0], ph[1], ph[2], ph[3], b0, b1);
            tc::mma(o[2 * nc + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
            tc::mma(o[2 * nc], ph[0], ph[1], ph[2], ph[3], c0, c1);
            tc::mma(o[2 * nc + 1], ph[0], ph[1], ph[2], ph[3], c2, c3);
            tc::mma(o[2 * nc], pl[0], pl[1], pl[2], pl[3], b0, b1);
            tc::mma(o[2 * nc + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
          }
        }
      }
    }

    // the next tile into the other buffer
    if (nfast)
      convert_raw(raw, buf ^ 1);
    else if (more)
      dequant_tile(tn, buf ^ 1);
  }

  // ---- normalise and store rows g and g + 8 ----
  l0 += __shfl_xor_sync(tc::kFull, l0, 1);
  l0 += __shfl_xor_sync(tc::kFull, l0, 2);
  l1 += __shfl_xor_sync(tc::kFull, l1, 1);
  l1 += __shfl_xor_sync(tc::kFull, l1, 2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int R = Rw + g + 8 * half;
    if (R >= rows_total) continue;
    const int i = R / G, h = R - i * G;
    const float il = 1.0f / (half ? l1 : l0);
    const int64_t base = (((int64_t)b * a.chunk + i) * a.num_q_heads + kvh * G + h) * kHeadDim + 2 * t4;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float v0 = o[j][2 * half] * il, v1 = o[j][2 * half + 1] * il;
      if (a.out_dtype == KVQ_F32) {
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + base + 8 * j) = make_float2(v0, v1);
      } else {
        *reinterpret_cast<__half2*>(reinterpret_cast<__half*>(a.out) + base + 8 * j) = __floats2half2_rn(v0, v1);
      }
    }
  }
}

}  // namespace
}  // namespace pa

namespace {
template <bool OUTL>
cudaError_t launch_pa(const LayerDev& L, const PrefillAttnArgs& a, cudaStream_t st) {
  static SmemAttr attr;
  {
    const cudaError_t e = attr.ensure(pa::prefill_attn_kernel<OUTL>, pa::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  const int rows = a.chunk * a.G;
  const dim3 grid((rows + pa::kRowsCta - 1) / pa::kRowsCta, L.n_streams);
  pa::prefill_attn_kernel<OUTL><<<grid, pa::kThreads, pa::kSmemBytes, st>>>(L, a);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefill_attention(const LayerDev& L, const PrefillAttnArgs& a, cudaStream_t st) {
  // rows with a few outliers keep the pipelined path in their own instance
  return L.outliers > 0 && L.outliers <= pa::kMaxFastOutliers ? launch_pa<true>(L, a, st) : launch_pa<false>(L, a, st);
}

}  // namespace kvq
