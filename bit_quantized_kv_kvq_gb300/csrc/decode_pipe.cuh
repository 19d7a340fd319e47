// Decode attention with the scores computed transposed, for per-channel keys
// and per-token values of 3/3, 4/4, 4/8, 8/4 or 8/8 bits, 1, 2, 4 or 8 query
// heads per kv-head, with or without fp16 outliers.
//
// Both products of a tile are fp16 tensor-core contractions (mma.sync
// m16n8k16, fp32 accumulation) whose M rows are the query heads of the
// kv-head, each as an fp16 pair hi + lo (head h: rows h and h + 8):
//   S^T[row][t] = sum_slot Q''[row][slot] K[slot][t]     (N = 8 tokens)
//   O[row][c]   = sum_t    P'[row][t]     V[t][c]        (N = 8 channels)
// so the probabilities leave QK^T in exactly the register layout of the A
// operand of PV (no transposition). Codes enter the mma unconverted, as
// subnormal fp16 halves (a code n masked into the low mantissa bits is
// n * 2^-24, or 2^k n * 2^-24 when it sits k bits up); the 2^-24 and 2^k
// factors are folded into Q'' (keys) or undone on the output (values).
//
// Dequantization is folded into the products (TurboQuant KV-cache page,
// demingchina.com/news/57821, §2.3): per key block, Q''[c] = q_c s_c and the
// bias sum_c q_c z_c; per token, P'[t] = p_t s_t and sum_t p_t z_t. Outliers
// (KVQuant page, cf-1.com/news/2306543, §2.2 item 3) add q_c (x - z_c) to a
// score and p_t (x - z_t) to the output.
//
// Work split (stream-K): the key blocks ("chunks") of all (batch, kv-head)
// streams are laid end to end and cut into one contiguous range per CTA,
// one CTA per SM. A chunk's packed tiles ("units" of 32 tokens) are
// staged in a ring of shared-memory stages by TMA copies (tensor-map copies
// with a bank swizzle for 4/8-bit code rows, 1-D bulk copies otherwise); the
// eight warps take whole chunks in turn and keep their own online softmax
// state, and a warp that finishes a unit refills its stage with the unit one
// ring length ahead (so there is no producer warp, and a warp may hold up to
// 255 registers: two warps per SM sub-partition). When a warp leaves a stream it
// merges its state into a per-stream accumulator of the CTA; the last warp
// writes the CTA's partial (or the output, when no other CTA holds part of
// the stream), and the last CTA of a stream merges the partials. Every wait
// is bounded: a wait that gives up raises the status word, stops the CTA and
// drains its copies in flight.
#pragma once

#include <cuda.h>

#include "decode_merge.cuh"
#include "mma_frag.cuh"
#include "tensor_map.cuh"

namespace kvq {
namespace pipe {

constexpr int kCons = 8;                    // warps
constexpr int kThreads = 32 * kCons;
constexpr int kHMax = 8;                    // query heads per kv-head
constexpr int kFragRow = 9;                 // uint4 per lane row of the fragment exchange (8 + pad)
constexpr int kPartRow = 132;               // floats per partial row: o[128], m, l, pad
constexpr float kLazy = 8.0f;               // the running max moves only when exceeded by this
constexpr unsigned kFull = 0xffffffffu;

struct __align__(64) Maps {
  CUtensorMap k;  // key codes, uint8 [stream][row][bytes] (4/8-bit codes)
  CUtensorMap v;  // value codes
};

struct Args {
  const __half* q;      // [B][Hq][D]
  const float* sink_part;  // attention over the fp16 sink tokens per row, or NULL
  void* out;            // [B][Hq][D]
  float* part;          // [streams][jmax][H][kPartRow]
  uint32_t* counters;   // [streams], zero between calls
  int out_dtype;
  int num_q_heads;
  int H;                // query heads per kv-head
  float scale_log2;     // softmax scale * log2(e)
  int length;           // tokens cached
  int kq;               // key rows held as codes (a multiple of T)
  int T;                // key block (tokens) = one chunk
  int UT;               // tokens per unit (64: two subtiles of 32)
  int U;                // units per chunk
  int cps;              // chunks per stream
  long long n_chunks;   // chunks of all streams
  int vex;              // virtual chunks after each stream's blocks (the cost of a stream switch)
  long long n_virtual;  // n_streams * (cps + vex): the space the CTAs split evenly
  int P;                // CTAs
  int jmax;             // partial rows per stream
  int kout;             // outliers per row
  // one ring stage
  int ns, stage_bytes, off_vc, off_km, off_vm, off_out;
  int kc_bytes, vc_bytes, vm_bytes;
  // shared-memory regions
  int ring_bytes, warp_bytes, slot_bytes;
  int w_qn, w_frag, w_eq, w_kz, w_ocr;  // offsets inside a consumer warp's scratch
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  return __byte_perm(a, b, sel);
}

__device__ __forceinline__ uint32_t u4(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Value n-tile j (8 channels, column n = lane group g) -> channel, bits the
// code sits up in its half, value group. Channels >= 128 are padding (3-bit
// rows: 13 words over 8 lane groups).
template <int VB, int VG>
__host__ __device__ __forceinline__ void vchan(int j, int n, int& ch, int& sh, int& q) {
  if (VB == 4) {
    const int wi = j >> 3, nib = j & 7;
    ch = 64 * wi + 8 * n + nib;
    sh = (nib & 1) ? 4 : 0;
    q = VG == 64 ? wi : 0;
  } else if (VB == 8) {
    const int wi = j >> 2, byte = j & 3;
    const int word = wi < 2 ? 2 * n + wi : 16 + 2 * n + (wi - 2);
    ch = 4 * word + byte;
    sh = 0;
    q = VG == 64 ? (wi >= 2 ? 1 : 0) : 0;
  } else {
    const int wi = j / 10, code = j % 10;
    const int word = wi == 0 ? n : n + 8;
    ch = word > 12 ? 255 : 10 * word + code;
    sh = code == 1 || code == 4 ? 3 : code == 2 ? 6 : code == 5 ? 7 : code == 6 || code == 8 ? 2
       : code == 7 || code == 9 ? 5 : 0;
    q = 0;
  }
}

template <int KB, int VB, int VG, bool OUTL>
__global__ void __launch_bounds__(kThreads, 1)
    decode_pipe_kernel(const __grid_constant__ Maps maps, const LayerDev L, const Args a) {
  constexpr int KW = Pack<KB>::kWords;
  constexpr int VW = Pack<VB>::kWords;
  constexpr int KROW = 4 * KW, VROW = 4 * VW;
  constexpr int VGPR = kHeadDim / VG;
  constexpr int NTV = VB == 3 ? 20 : 16;  // PV n-tiles
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // swizzled copies need 1024-byte aligned stages: align the base by hand
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int H = a.H;
  // Even split of the virtual chunk space (each stream's blocks followed by
  // vex empty places), mapped back to real chunks: a CTA whose range crosses
  // a stream boundary takes fewer blocks, paying for the switch.
  auto real_of = [&](long long v) {
    const long long n = v / (a.cps + a.vex), r = v - n * (a.cps + a.vex);
    return n * a.cps + (r < a.cps ? r : a.cps);
  };
  const long long cA = real_of((long long)blockIdx.x * a.n_virtual / a.P);
  const long long cB = real_of((long long)(blockIdx.x + 1) * a.n_virtual / a.P);

  unsigned char* ring = smem;
  unsigned char* wbase = smem + a.ring_bytes;
  unsigned char* slots = wbase + (size_t)kCons * a.warp_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(slots + 2 * a.slot_bytes);
  int* last = reinterpret_cast<int*>(full + a.ns);  // last unit issued into each stage
  int* ctl = last + a.ns;  // owner[2], done[2], lock[2], abort, merges, merge streams[2]
  volatile int* vctl = ctl;
  const int n_units = (int)(cB - cA) * a.U;

  if (tid == 0) {
    for (int s = 0; s < a.ns; ++s) {
      mbar_init(&full[s], 1);
      last[s] = -1;
    }
    ctl[0] = 0;
    ctl[1] = 1;
    ctl[2] = ctl[3] = ctl[4] = ctl[5] = ctl[6] = ctl[7] = 0;
    mbar_fence_init();
  }
  for (int i = tid; i < 2 * a.slot_bytes / 4; i += kThreads) {
    const int within = i % (a.slot_bytes / 4);
    reinterpret_cast<float*>(slots)[i] = (within >= H * kHeadDim && within < H * kHeadDim + kHMax)
                                             ? -INFINITY : 0.0f;
  }
  __syncthreads();

  auto aborted = [&]() { return vctl[6] != 0; };
  auto abort_now = [&]() {
    raise_status(L.status, kStatusTimeout);
    atomicExch(&ctl[6], 1);
  };

  // Stages unit u of this CTA (unit k of key block blk of stream n) in stage
  // s = u mod ns: key codes, the key block's scales (first unit of a block),
  // key outliers, value codes, value scales, value outliers. A unit past the
  // end of its stream completes its stage's phase with a plain arrival.
  auto issue = [&](int u, int s, int n, int blk, int k) {
    const int t0 = blk * a.T + k * a.UT;
    *reinterpret_cast<volatile int*>(&last[s]) = u;
    if (t0 >= a.length) {
      mbar_arrive(&full[s]);
      return;
    }
    unsigned char* st = ring + (size_t)s * a.stage_bytes;
    const bool rt = t0 >= a.kq;
    const uint32_t ob = OUTL ? (uint32_t)(a.UT * a.kout * 2) : 0u;
    uint32_t bytes = a.vc_bytes + a.vm_bytes + 2 * ob;
    if (!rt) bytes += a.kc_bytes + (k == 0 ? kHeadDim * 4u : 0u) + 2 * ob;
    mbar_arrive_expect_tx(&full[s], bytes);
    if (!rt) {
      if (KB == 3)
        bulk_g2s(st, L.k.codes + (int64_t)n * L.k.codes_sstride + (int64_t)t0 * KW, a.kc_bytes, &full[s]);
      else
        tma_rows(st, &maps.k, t0, n, &full[s]);
      if (k == 0)
        bulk_g2s(st + a.off_km, L.k.meta + (int64_t)n * L.k.meta_sstride + (int64_t)blk * kHeadDim * 4,
                 kHeadDim * 4, &full[s]);
      if (OUTL) {
        const int64_t e0 = (int64_t)n * L.k.out_sstride + (int64_t)t0 * a.kout;
        bulk_g2s(st + a.off_out, L.k.col + e0, ob, &full[s]);
        bulk_g2s(st + a.off_out + ob, L.k.val + e0, ob, &full[s]);
      }
    }
    if (VB == 3)
      bulk_g2s(st + a.off_vc, L.v.codes + (int64_t)n * L.v.codes_sstride + (int64_t)t0 * VW, a.vc_bytes, &full[s]);
    else
      tma_rows(st + a.off_vc, &maps.v, t0, n, &full[s]);
    bulk_g2s(st + a.off_vm, L.v.meta + (int64_t)n * L.v.meta_sstride + (int64_t)t0 * VGPR * 4, a.vm_bytes,
             &full[s]);
    if (OUTL) {
      const int64_t e0 = (int64_t)n * L.v.out_sstride + (int64_t)t0 * a.kout;
      bulk_g2s(st + a.off_out + 2 * ob, L.v.col + e0, ob, &full[s]);
      bulk_g2s(st + a.off_out + 3 * ob, L.v.val + e0, ob, &full[s]);
    }
  };
  // first fill of the ring: warp w stages units w, w + 8, ... (< ns)
  if (lane == 0 && cA < cB) {
    if (warp == 0) {
      if (KB != 3) prefetch_map(&maps.k);
      if (VB != 3) prefetch_map(&maps.v);
      // the query rows of this CTA's streams into L2 while the ring fills
      const int Hkv = L.num_kv_heads;
      for (int n = (int)(cA / a.cps); n <= (int)((cB - 1) / a.cps); ++n) {
        const int b = n / Hkv, kvh = n - b * Hkv;
        const __half* qr = a.q + ((int64_t)b * a.num_q_heads + (int64_t)kvh * H) * kHeadDim;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(qr), "r"((uint32_t)(H * kHeadDim * 2))
                     : "memory");
      }
    }
    for (int u = warp; u < a.ns && u < n_units; u += kCons) {
      const long long ci = cA + u / a.U;
      const int n = (int)(ci / a.cps);
      issue(u, u, n, (int)(ci - (long long)n * a.cps), u % a.U);
    }
  }
  __syncthreads();

  if (cA < cB) {
    // ------------------------------------------------------------------ warps
    unsigned char* wsp = wbase + (size_t)warp * a.warp_bytes;
    float* qn = reinterpret_cast<float*>(wsp + a.w_qn);        // [H][128] q * scale_log2 * 2^-e_q
    uint4* frag = reinterpret_cast<uint4*>(wsp + a.w_frag);     // [32][kFragRow] fragment exchange
    int* eqs = reinterpret_cast<int*>(wsp + a.w_eq);            // [8] e_q per head
    float* kz = reinterpret_cast<float*>(wsp + a.w_kz);         // [128] key zero points (outliers)
    float* ocr = reinterpret_cast<float*>(wsp + a.w_ocr);       // [H][128] value-outlier sums
    const int Hkv = L.num_kv_heads;

    // ---- state of the warp for the current stream ---------------------------------
    uint32_t aq[8][4];      // Q'' fragments of the current chunk
    float kf = 0.0f, kb = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;
    float zacc[VGPR];
    int ev[VGPR];
    float vsf[VGPR];
    float O[NTV][4];
    int eq_g = 0;

    auto reset_state = [&]() {
      m_run = -INFINITY;
      l_run = 0.0f;
#pragma unroll
      for (int q = 0; q < VGPR; ++q) {
        zacc[q] = 0.0f;
        ev[q] = -30;
        vsf[q] = tc::exp2i(36);
      }
#pragma unroll
      for (int j = 0; j < NTV; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[j][e] = 0.0f;
      if (OUTL) {
        for (int i = lane; i < H * kHeadDim; i += 32) ocr[i] = 0.0f;
        __syncwarp();
      }
    };

    // query rows of stream n, scaled into [1, 2) magnitudes per head
    auto load_q = [&](int n) {
      const int b = n / Hkv, kvh = n - b * Hkv;
      __syncwarp();
      uint2 rq[kHMax];  // every head's row in flight at once
#pragma unroll
      for (int h = 0; h < kHMax; ++h)
        if (h < H)
          rq[h] = __ldg(reinterpret_cast<const uint2*>(a.q + ((int64_t)b * a.num_q_heads + kvh * H + h) * kHeadDim +
                                                        4 * lane));
#pragma unroll
      for (int h = 0; h < kHMax; ++h) {
        if (h >= H) break;
        const uint2 raw = rq[h];
        const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        float v[4] = {x01.x * a.scale_log2, x01.y * a.scale_log2, x23.x * a.scale_log2,
                      x23.y * a.scale_log2};
        uint32_t mb = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) mb = max(mb, __float_as_uint(fabsf(v[i])));
        mb = __reduce_max_sync(kFull, mb);
        const int e = mb ? (int)(mb >> 23) - 127 : 0;
        const float f = tc::exp2i(-e);
        *reinterpret_cast<float4*>(qn + h * kHeadDim + 4 * lane) =
            make_float4(v[0] * f, v[1] * f, v[2] * f, v[3] * f);
        if (lane == 0) eqs[h] = e;
      }
      __syncwarp();
      eq_g = g < H ? eqs[g] : 0;
    };

    // Q'' fragments, key bias and score factor of a chunk. Lane l = kc + 8 t4
    // computes the four k-slots (kc, t4) of every head and hands them to the
    // fragment owners (head h, t4) through shared memory.
    auto rebuild = [&](bool rt, const unsigned char* km_s) {
      __syncwarp();
      const int kcl = lane & 7, t4l = lane >> 3;
      float s2[4], z2[4];
      int ch[4];
      int es = 0;
      if (!rt) {
        const __half2* km = reinterpret_cast<const __half2*>(km_s);
        uint32_t sb = 0;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          int sh;
          tc::key_slot<KB>(t4l, kcl, s, ch[s], sh);
          const float2 sz = __half22float2(km[ch[s]]);
          s2[s] = sz.x * tc::exp2i(-sh);
          z2[s] = sz.y;
          sb = max(sb, __float_as_uint(sz.x));
          if (OUTL) kz[ch[s]] = sz.y;
        }
        sb = __reduce_max_sync(kFull, sb);
        es = sb ? max((int)(sb >> 23) - 127, -30) : -30;
        const float sf = tc::exp2i(13 - es);
#pragma unroll
        for (int s = 0; s < 4; ++s) s2[s] *= sf;
      } else {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          ch[s] = 32 * t4l + 4 * kcl + s;
          s2[s] = 8192.0f;
          z2[s] = 0.0f;
        }
      }
      // every query value first: the fragment stores below would otherwise
      // order each head's loads after the previous head's stores
      float qv[kHMax][4];
#pragma unroll
      for (int h = 0; h < kHMax; ++h)
#pragma unroll
        for (int s = 0; s < 4; ++s) qv[h][s] = h < H ? qn[h * kHeadDim + ch[s]] : 0.0f;
      float bias[kHMax];
#pragma unroll
      for (int h = 0; h < kHMax; ++h) {
        bias[h] = 0.0f;
        if (h < H) {
          float v[4];
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            v[s] = qv[h][s] * s2[s];
            bias[h] = fmaf(qv[h][s], z2[s], bias[h]);
          }
          uint32_t lo01, lo23;
          const uint32_t hi01 = tc::split_pair(v[0], v[1], lo01);
          const uint32_t hi23 = tc::split_pair(v[2], v[3], lo23);
          frag[(4 * h + t4l) * kFragRow + kcl] = make_uint4(hi01, lo01, hi23, lo23);
        }
      }
      // bias of every head: reduce-scatter over lane bits 4, 3, 2, then sum
      // over bits 1, 0; lane l ends with head l >> 2
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool up = (lane & 16) != 0;
        const float send = up ? bias[i] : bias[i + 4];
        const float keep = up ? bias[i + 4] : bias[i];
        bias[i] = keep + __shfl_xor_sync(kFull, send, 16);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bool up = (lane & 8) != 0;
        const float send = up ? bias[i] : bias[i + 2];
        const float keep = up ? bias[i + 2] : bias[i];
        bias[i] = keep + __shfl_xor_sync(kFull, send, 8);
      }
      {
        const bool up = (lane & 4) != 0;
        const float send = up ? bias[0] : bias[1];
        const float keep = up ? bias[1] : bias[0];
        bias[0] = keep + __shfl_xor_sync(kFull, send, 4);
      }
      bias[0] += __shfl_xor_sync(kFull, bias[0], 1);
      bias[0] += __shfl_xor_sync(kFull, bias[0], 2);
      __syncwarp();
      // rows of heads >= H stay zero (their rows of the products are unused)
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        const uint4 f = g < H ? frag[(4 * g + t4) * kFragRow + kc] : make_uint4(0u, 0u, 0u, 0u);
        aq[kc][0] = f.x;
        aq[kc][1] = f.y;
        aq[kc][2] = f.z;
        aq[kc][3] = f.w;
      }
      kf = rt ? tc::exp2i(eq_g - 13) : tc::exp2i(eq_g + es + 11);
      kb = rt ? 0.0f : bias[0] * tc::exp2i(eq_g);
      if (OUTL) __syncwarp();
    };

    // One subtile of 32 tokens: rows r0 .. r0+31 of the unit in stage st;
    // nv valid tokens; rt: keys from the fp16 residual (krow: first row).
    auto subtile = [&](const unsigned char* st, int r0, int nv, bool rt, const __half* kres) {
      float c[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[nt][e] = 0.0f;

      // ---- S^T = Q'' K^T: n-tile nt holds tokens 8 nt .. 8 nt + 7 (column g) ----
      if (!rt) {
        if (KB == 4) {
          uint4 kw[4];
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
            kw[nt] = *reinterpret_cast<const uint4*>(st + swz<64>((uint32_t)(r0 + 8 * nt + g) * 64u + 16u * t4));
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int nt = 0; nt < 4; ++nt) {
                const uint32_t x = u4(kw[nt], j) >> (8 * h);
                tc::mma(c[nt], aq[2 * j + h][0], aq[2 * j + h][1], aq[2 * j + h][2], aq[2 * j + h][3],
                        x & 0x000F000Fu, x & 0x00F000F0u);
              }
        } else if (KB == 8) {
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            uint4 kw[4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
              kw[nt] = *reinterpret_cast<const uint4*>(
                  st + swz<128>((uint32_t)(r0 + 8 * nt + g) * 128u + 16u * (2 * t4 + hq)));
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int nt = 0; nt < 4; ++nt) {
                const uint32_t w = u4(kw[nt], j);
                const int kc = 4 * hq + j;
                tc::mma(c[nt], aq[kc][0], aq[kc][1], aq[kc][2], aq[kc][3], w & 0x00FF00FFu,
                        (w >> 8) & 0x00FF00FFu);
              }
          }
        } else {
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t P[2][16];
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2) {
              const int nt = 2 * np + i2;
              const uint32_t* rw = reinterpret_cast<const uint32_t*>(st) + (r0 + 8 * nt + g) * 13;
              const uint32_t X[3] = {rw[t4], rw[t4 + 4], rw[t4 + 8]};
              const uint32_t D = rw[12];
#pragma unroll
              for (int i = 0; i < 3; ++i) {
                P[i2][4 * i + 0] = X[i] & 0x001C0007u;
                P[i2][4 * i + 1] = X[i] & 0x00E00038u;
                P[i2][4 * i + 2] = (X[i] >> 6) & 0x001C0007u;
                P[i2][4 * i + 3] = (X[i] >> 9) & 0x001C0007u;
              }
              const uint32_t ab = prmt(X[0] >> 12, X[1] >> 12, 0x5410u);
              const uint32_t cd = prmt(X[2] >> 12, D >> (6 * t4), 0x5410u);
              P[i2][12] = ab & 0x00070007u;
              P[i2][13] = ab & 0x00380038u;
              P[i2][14] = cd & 0x00070007u;
              P[i2][15] = cd & 0x00380038u;
            }
            // even and odd k-chunks in separate accumulators: four independent mma chains
            float c2[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
            for (int kc = 0; kc < 8; ++kc)
#pragma unroll
              for (int i2 = 0; i2 < 2; ++i2)
                tc::mma((kc & 1) ? c2[i2] : c[2 * np + i2], aq[kc][0], aq[kc][1], aq[kc][2], aq[kc][3],
                        P[i2][2 * kc], P[i2][2 * kc + 1]);
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
              for (int e = 0; e < 4; ++e) c[2 * np + i2][e] += c2[i2][e];
          }
        }
      } else {
        // fp16 residual keys: lane t4 reads channels 32 t4 .. 32 t4 + 31 of its token
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t kr[2][16];
#pragma unroll
          for (int i2 = 0; i2 < 2; ++i2) {
            const uint4* p = reinterpret_cast<const uint4*>(kres + (size_t)(r0 + 8 * (2 * np + i2) + g) * kHeadDim +
                                                            32 * t4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 v = __ldg(p + i);
              kr[i2][4 * i] = v.x;
              kr[i2][4 * i + 1] = v.y;
              kr[i2][4 * i + 2] = v.z;
              kr[i2][4 * i + 3] = v.w;
            }
          }
          float c2[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
          for (int kc = 0; kc < 8; ++kc)
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2)
              tc::mma((kc & 1) ? c2[i2] : c[2 * np + i2], aq[kc][0], aq[kc][1], aq[kc][2], aq[kc][3],
                      kr[i2][2 * kc], kr[i2][2 * kc + 1]);
#pragma unroll
          for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
            for (int e = 0; e < 4; ++e) c[2 * np + i2][e] += c2[i2][e];
        }
      }

      // ---- scores of head g for tokens 8 nt + 2 t4 + e (log2 units) --------------
      float sc[4][2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = fmaf(c[nt][0] + c[nt][2], kf, kb);
        sc[nt][1] = fmaf(c[nt][1] + c[nt][3], kf, kb);
      }
      const unsigned char* ot = st + a.off_out;
      const uint32_t ob = OUTL ? (uint32_t)(a.UT * a.kout * 2) : 0u;
      if (OUTL && !rt) {
        // key outliers: the lane of token `lane` sums q_c (x - z_c) for every head
        const uint16_t* kcol = reinterpret_cast<const uint16_t*>(ot);
        const __half* kval = reinterpret_cast<const __half*>(ot + ob);
        float corr[kHMax];
#pragma unroll
        for (int h = 0; h < kHMax; ++h) corr[h] = 0.0f;
        for (int e = 0; e < a.kout; ++e) {
          const int i = (r0 + lane) * a.kout + e;
          const int cc = kcol[i] & (kHeadDim - 1);
          const float d = __half2float(kval[i]) - kz[cc];
#pragma unroll
          for (int h = 0; h < kHMax; ++h)
            if (h < H) corr[h] = fmaf(qn[h * kHeadDim + cc], d, corr[h]);
        }
        if (H == 1) {
          const float f = tc::exp2i(eq_g);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) sc[nt][e] = fmaf(__shfl_sync(kFull, corr[0], 8 * nt + 2 * t4 + e), f, sc[nt][e]);
        } else {
          float* pst = reinterpret_cast<float*>(frag);  // [32 tokens][8 heads]
#pragma unroll
          for (int h = 0; h < kHMax; ++h) pst[lane * kHMax + h] = corr[h];
          __syncwarp();
          const float f = tc::exp2i(eq_g);
          if (g < H)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) sc[nt][e] = fmaf(pst[(8 * nt + 2 * t4 + e) * kHMax + g], f, sc[nt][e]);
          __syncwarp();
        }
      }
      if (nv < 32) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (8 * nt + 2 * t4 + e >= nv) sc[nt][e] = -INFINITY;
      }

      // ---- online softmax (lazy running max) ----------------------------------------
      float mx = fmaxf(fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1])),
                       fmaxf(fmaxf(sc[2][0], sc[2][1]), fmaxf(sc[3][0], sc[3][1])));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      const bool up = mx > m_run + kLazy;
      if (__any_sync(kFull, up)) {
        const float mnew = up ? mx : m_run;
        const float al = ex2(m_run - mnew);
        l_run *= al;
#pragma unroll
        for (int q = 0; q < VGPR; ++q) zacc[q] *= al;
#pragma unroll
        for (int j = 0; j < NTV; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) O[j][e] *= al;
        if (OUTL) {
          __syncwarp();
          for (int h = 0; h < H; ++h) {
            const float alh = __shfl_sync(kFull, al, 4 * h);
#pragma unroll
            for (int i = 0; i < 4; ++i) ocr[h * kHeadDim + lane + 32 * i] *= alh;
          }
          __syncwarp();
        }
        m_run = mnew;
      }
      float p[4][2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          p[nt][e] = ex2(sc[nt][e] - m_run);
          l_run += p[nt][e];
        }

      // ---- value scales of the lane's tokens; value-scale exponents -----------------
      const unsigned char* vm_s = st + a.off_vm;
      uint32_t mw[4][2][VGPR];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int row = r0 + 8 * nt + 2 * t4;
        if (VGPR == 1) {
          const uint2 u = *reinterpret_cast<const uint2*>(vm_s + (size_t)row * 4);
          mw[nt][0][0] = u.x;
          mw[nt][1][0] = u.y;
        } else {
          const uint4 u = *reinterpret_cast<const uint4*>(vm_s + (size_t)row * 8);
          mw[nt][0][0] = u.x;
          mw[nt][0][VGPR - 1] = u.y;
          mw[nt][1][0] = u.z;
          mw[nt][1][VGPR - 1] = u.w;
        }
      }
      if (nv < 32) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (8 * nt + 2 * t4 + e >= nv)
#pragma unroll
              for (int q = 0; q < VGPR; ++q) mw[nt][e][q] = 0u;
      }
#pragma unroll
      for (int q = 0; q < VGPR; ++q) {
        uint32_t sm = 0;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) sm = max(sm, max(mw[nt][0][q] & 0xFFFFu, mw[nt][1][q] & 0xFFFFu));
        sm = max(sm, __shfl_xor_sync(kFull, sm, 1));
        sm = max(sm, __shfl_xor_sync(kFull, sm, 2));
        const float sf = __half2float(__ushort_as_half((unsigned short)sm));
        const int e = sm ? (int)(__float_as_uint(sf) >> 23) - 127 : -127;
        if (e > ev[q]) {  // warp-uniform: every lane saw the same tokens' scales
          const float f = tc::exp2i(max(ev[q] - e, -126));
#pragma unroll
          for (int j = 0; j < NTV; ++j) {
            int cch, csh, cq;
            vchan<VB, VG>(j, 0, cch, csh, cq);
            if (cq == q)
#pragma unroll
              for (int k = 0; k < 4; ++k) O[j][k] *= f;
          }
          ev[q] = e;
          vsf[q] = tc::exp2i(6 - e);
        }
      }

      // ---- P' = p s 2^(6 - ev) as hi/lo A fragments; zero-point sums ----------------
      uint32_t ap[VGPR][2][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int q = 0; q < VGPR; ++q) {
          const float2 sz0 = __half22float2(*reinterpret_cast<const __half2*>(&mw[nt][0][q]));
          const float2 sz1 = __half22float2(*reinterpret_cast<const __half2*>(&mw[nt][1][q]));
          zacc[q] = fmaf(p[nt][0], sz0.y, fmaf(p[nt][1], sz1.y, zacc[q]));
          uint32_t lo;
          const uint32_t hi = tc::split_pair(p[nt][0] * (sz0.x * vsf[q]), p[nt][1] * (sz1.x * vsf[q]), lo);
          ap[q][nt >> 1][2 * (nt & 1)] = hi;
          ap[q][nt >> 1][2 * (nt & 1) + 1] = lo;
        }

      // ---- value outliers: the lane of token `lane` adds p (x - z) per head ----------
      if (OUTL) {
        float pl[kHMax];
        if (H == 1) {
          const int src = (lane & 7) >> 1;
          float v = 0.0f;
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float t = __shfl_sync(kFull, p[nt][e], src);
              if (nt == (lane >> 3) && e == (lane & 1)) v = t;
            }
          pl[0] = v;
        } else {
          float* pst = reinterpret_cast<float*>(frag);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) pst[(8 * nt + 2 * t4 + e) * kHMax + g] = p[nt][e];
          __syncwarp();
#pragma unroll
          for (int h = 0; h < kHMax; ++h) pl[h] = pst[lane * kHMax + h];
          __syncwarp();
        }
        if (lane < nv) {
          const uint16_t* vcol = reinterpret_cast<const uint16_t*>(ot + 2 * ob);
          const __half* vval = reinterpret_cast<const __half*>(ot + 3 * ob);
          const __half2* vmr = reinterpret_cast<const __half2*>(vm_s) + (size_t)(r0 + lane) * VGPR;
          for (int e = 0; e < a.kout; ++e) {
            const int i = (r0 + lane) * a.kout + e;
            const int cc = vcol[i] & (kHeadDim - 1);
            const float d = __half2float(vval[i]) - __high2float(vmr[VGPR == 1 ? 0 : cc / VG]);
#pragma unroll
            for (int h = 0; h < kHMax; ++h)
              if (h < H) atomicAdd(&ocr[h * kHeadDim + cc], pl[h] * d);
          }
        }
      }

      // ---- O += P' V: k-chunk kk holds tokens 16 kk + {2t4, 2t4+1, 2t4+8, 2t4+9} -----
      const unsigned char* vc_s = st + a.off_vc;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int ra = r0 + 16 * kk + 2 * t4, rb = ra + 8;
        if (VB == 4) {
          uint32_t w[4][2];  // rows ra, ra+1, rb, rb+1; words g, 8+g
          const int rows[4] = {ra, ra + 1, rb, rb + 1};
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int wi = 0; wi < 2; ++wi)
              w[r][wi] = *reinterpret_cast<const uint32_t*>(
                  vc_s + swz<64>((uint32_t)rows[r] * 64u + 4u * (8 * wi + g)));
#pragma unroll
          for (int wi = 0; wi < 2; ++wi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t sel = hh ? 0x7632u : 0x5410u;
              const uint32_t xa = prmt(w[0][wi], w[1][wi], sel), xb = prmt(w[2][wi], w[3][wi], sel);
              const uint32_t ya = xa >> 8, yb = xb >> 8;
              const int q = VG == 64 ? wi : 0;
              const int j0 = 8 * wi + 4 * hh;
              tc::mma(O[j0 + 0], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], xa & 0x000F000Fu,
                      xb & 0x000F000Fu);
              tc::mma(O[j0 + 1], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], xa & 0x00F000F0u,
                      xb & 0x00F000F0u);
              tc::mma(O[j0 + 2], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], ya & 0x000F000Fu,
                      yb & 0x000F000Fu);
              tc::mma(O[j0 + 3], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], ya & 0x00F000F0u,
                      yb & 0x00F000F0u);
            }
        } else if (VB == 8) {
          uint32_t w[4][4];  // rows; words 2g, 2g+1, 16+2g, 17+2g
          const int rows[4] = {ra, ra + 1, rb, rb + 1};
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const uint2 u = *reinterpret_cast<const uint2*>(
                  vc_s + swz<128>((uint32_t)rows[r] * 128u + 64u * hf + 8u * g));
              w[r][2 * hf] = u.x;
              w[r][2 * hf + 1] = u.y;
            }
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const uint32_t xa = prmt(w[0][wi], w[1][wi], 0x6420u), xb = prmt(w[2][wi], w[3][wi], 0x6420u);
            const uint32_t ya = prmt(w[0][wi], w[1][wi], 0x7531u), yb = prmt(w[2][wi], w[3][wi], 0x7531u);
            const int q = VG == 64 ? (wi >> 1) : 0;
            const int j0 = 4 * wi;
            tc::mma(O[j0 + 0], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], xa & 0x00FF00FFu,
                    xb & 0x00FF00FFu);
            tc::mma(O[j0 + 2], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], (xa >> 8) & 0x00FF00FFu,
                    (xb >> 8) & 0x00FF00FFu);
            tc::mma(O[j0 + 1], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], ya & 0x00FF00FFu,
                    yb & 0x00FF00FFu);
            tc::mma(O[j0 + 3], ap[q][kk][0], ap[q][kk][1], ap[q][kk][2], ap[q][kk][3], (ya >> 8) & 0x00FF00FFu,
                    (yb >> 8) & 0x00FF00FFu);
          }
        } else {
          const uint32_t* vr = reinterpret_cast<const uint32_t*>(vc_s);
          const int wd[2] = {g, min(g + 8, 12)};
#pragma unroll
          for (int wi = 0; wi < 2; ++wi) {
            const uint32_t a0 = vr[ra * 13 + wd[wi]], a1 = vr[(ra + 1) * 13 + wd[wi]];
            const uint32_t b0 = vr[rb * 13 + wd[wi]], b1 = vr[(rb + 1) * 13 + wd[wi]];
            const uint32_t xa = prmt(a0, a1, 0x5410u), xb = prmt(b0, b1, 0x5410u);
            const uint32_t za = prmt(a0, a1, 0x6521u), zb = prmt(b0, b1, 0x6521u);
            const uint32_t ya = prmt(a0, a1, 0x7632u), yb = prmt(b0, b1, 0x7632u);
            const uint32_t xa9 = xa >> 9, xb9 = xb >> 9, ya6 = ya >> 6, yb6 = yb >> 6;
            const int j0 = 10 * wi;
            const uint32_t(&A)[4] = ap[0][kk];
            tc::mma(O[j0 + 0], A[0], A[1], A[2], A[3], xa & 0x00070007u, xb & 0x00070007u);
            tc::mma(O[j0 + 1], A[0], A[1], A[2], A[3], xa & 0x00380038u, xb & 0x00380038u);
            tc::mma(O[j0 + 2], A[0], A[1], A[2], A[3], xa & 0x01C001C0u, xb & 0x01C001C0u);
            tc::mma(O[j0 + 3], A[0], A[1], A[2], A[3], xa9 & 0x00070007u, xb9 & 0x00070007u);
            tc::mma(O[j0 + 4], A[0], A[1], A[2], A[3], xa9 & 0x00380038u, xb9 & 0x00380038u);
            tc::mma(O[j0 + 5], A[0], A[1], A[2], A[3], za & 0x03800380u, zb & 0x03800380u);
            tc::mma(O[j0 + 6], A[0], A[1], A[2], A[3], ya & 0x001C001Cu, yb & 0x001C001Cu);
            tc::mma(O[j0 + 7], A[0], A[1], A[2], A[3], ya & 0x00E000E0u, yb & 0x00E000E0u);
            tc::mma(O[j0 + 8], A[0], A[1], A[2], A[3], ya6 & 0x001C001Cu, yb6 & 0x001C001Cu);
            tc::mma(O[j0 + 9], A[0], A[1], A[2], A[3], ya6 & 0x00E000E0u, yb6 & 0x00E000E0u);
          }
        }
      }
    };

    // CTA that holds global chunk x (through its place in the virtual space)
    auto owner_of = [&](long long x) {
      const long long n = x / a.cps, vx = n * (a.cps + a.vex) + (x - n * a.cps);
      return (int)(((vx + 1) * a.P - 1) / a.n_virtual);
    };

    // Finalizes stream n from accumulator slot `so`: output, or this CTA's
    // partial and, from the last CTA of the stream, the merge of all partials.
    auto finalize = [&](const float* so, int n) {
      const float* sm = so + H * kHeadDim;
      const float* sl = sm + kHMax;
      const int b = n / Hkv, kvh = n - b * Hkv;
      const int cf = owner_of((long long)n * a.cps), cl = owner_of((long long)(n + 1) * a.cps - 1);
      const int K = cl - cf + 1, jj = (int)blockIdx.x - cf;
      auto write_out = [&](int h, float4 o) {
        const int64_t base = ((int64_t)b * a.num_q_heads + kvh * H + h) * kHeadDim + 4 * lane;
        if (a.out_dtype == KVQ_F32) {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + base) = o;
        } else {
          __half2 h01 = __floats2half2_rn(o.x, o.y), h23 = __floats2half2_rn(o.z, o.w);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&h01);
          u.y = *reinterpret_cast<uint32_t*>(&h23);
          *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.out) + base) = u;
        }
      };
      if (K == 1) {
        for (int h = 0; h < H; ++h) {
          const float4 o = *reinterpret_cast<const float4*>(so + h * kHeadDim + 4 * lane);
          write_out(h, finish_row4(a.sink_part, (int64_t)b * a.num_q_heads + kvh * H + h, 4 * lane, o, sm[h], sl[h]));
        }
        return;
      }
      for (int h = 0; h < H; ++h) {
        float* pr = a.part + (((int64_t)n * a.jmax + jj) * H + h) * kPartRow;
        *reinterpret_cast<float4*>(pr + 4 * lane) = *reinterpret_cast<const float4*>(so + h * kHeadDim + 4 * lane);
        if (lane == 0) {
          pr[kHeadDim] = sm[h];
          pr[kHeadDim + 1] = sl[h];
        }
      }
      __threadfence();
      __syncwarp();
      uint32_t t = 0;
      if (lane == 0) t = atomicAdd(&a.counters[n], 1u);
      t = __shfl_sync(kFull, t, 0);
      if ((int)t != K - 1) return;
      // this CTA holds the last partial of stream n: merge them after the
      // main loop, when every warp of the CTA can take part
      if (lane == 0) {
        const int slot_i = atomicAdd(&ctl[7], 1);
        if (slot_i < 2) ctl[8 + slot_i] = n;
        a.counters[n] = 0u;
      }
    };

    // Leaves segment sig (stream n): merges the warp's state into the CTA's
    // accumulator; the last warp to leave finalizes the stream.
    auto finish_segment = [&](int sig, int n, bool have) -> bool {
      __syncwarp();
      const int slot = sig & 1;
      float* so = reinterpret_cast<float*>(slots + (size_t)slot * a.slot_bytes);
      float* sm = so + H * kHeadDim;
      float* sl = sm + kHMax;
      bool ok = true;
      if (lane == 0) {
        int it = 0;
        while (vctl[slot] != sig) {
          if (aborted() || ++it > (kWaitLimit << 6)) {
            ok = false;
            break;
          }
        }
      }
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (!aborted()) abort_now();
        return false;
      }
      if (have) {
        float lt = l_run;
        lt += __shfl_xor_sync(kFull, lt, 1);
        lt += __shfl_xor_sync(kFull, lt, 2);
        float zt[VGPR];
#pragma unroll
        for (int q = 0; q < VGPR; ++q) {
          zt[q] = zacc[q];
          zt[q] += __shfl_xor_sync(kFull, zt[q], 1);
          zt[q] += __shfl_xor_sync(kFull, zt[q], 2);
        }
        if (lane == 0) {
          int it = 0;
          while (atomicCAS(&ctl[4 + slot], 0, 1) != 0) {
            if (++it > (kWaitLimit << 6)) {
              ok = false;
              break;
            }
          }
        }
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          abort_now();
          return false;
        }
        __threadfence_block();
        // every lane reads the accumulator's running max and sum of its head
        // before any lane writes them back
        const float mA = sm[g], lA = sl[g];
        __syncwarp();
        if (g < H) {
          const float M = fmaxf(mA, m_run);
          const float al = ex2(mA - M), be = ex2(m_run - M);
          // the accumulator's values first, so its loads are not ordered
          // after the stores of earlier channels
          float sv[NTV][2];
#pragma unroll
          for (int j = 0; j < NTV; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              int ch, sh, q;
              vchan<VB, VG>(j, 2 * t4 + e, ch, sh, q);
              sv[j][e] = ch < kHeadDim ? so[g * kHeadDim + ch] : 0.0f;
            }
#pragma unroll
          for (int j = 0; j < NTV; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              int ch, sh, q;
              vchan<VB, VG>(j, 2 * t4 + e, ch, sh, q);
              if (ch < kHeadDim) {
                float zq = zt[0];
                int eq = ev[0];
#pragma unroll
                for (int qq = 1; qq < VGPR; ++qq)
                  if (qq == q) {
                    zq = zt[qq];
                    eq = ev[qq];
                  }
                // undo 2^-24 of the codes, 2^sh of the code position and 2^(6 - ev)
                float o = fmaf(O[j][e] + O[j][e + 2], tc::exp2i(18 + eq - sh), zq);
                if (OUTL) o += ocr[g * kHeadDim + ch];
                so[g * kHeadDim + ch] = fmaf(al, sv[j][e], be * o);
              }
            }
          if (t4 == 0) {
            sm[g] = M;
            sl[g] = fmaf(al, lA, be * lt);
          }
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) atomicExch(&ctl[4 + slot], 0);
      }
      int d = 0;
      if (lane == 0) {
        __threadfence_block();
        d = atomicAdd(&ctl[2 + slot], 1);
      }
      d = __shfl_sync(kFull, d, 0);
      if (d == kCons - 1) {
        __threadfence_block();
        finalize(so, n);
        __syncwarp();
        for (int i = lane; i < H * kHeadDim; i += 32) so[i] = 0.0f;
        if (lane < kHMax) {
          sm[lane] = -INFINITY;
          sl[lane] = 0.0f;
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          ctl[2 + slot] = 0;
          __threadfence_block();
          atomicExch(&ctl[slot], sig + 2);
        }
      }
      return true;
    };

    const int n0 = (int)(cA / a.cps), n1 = (int)((cB - 1) / a.cps);
    const int ahead = a.ns / a.U;  // key blocks between a unit and its stage's next unit (ns is a multiple of U)
    for (int n = n0; n <= n1; ++n) {
      if (aborted()) break;
      const long long s0 = max(cA, (long long)n * a.cps), s1 = min(cB, (long long)(n + 1) * a.cps);
      const int sig = n - n0;
      const int l0 = (int)((s0 - cA) % kCons);
      const long long first = s0 + ((warp - l0) % kCons + kCons) % kCons;
      const bool have = first < s1;
      if (have) {
        load_q(n);
        reset_state();
      }
      bool ok = true;
      for (long long ci = first; ci < s1 && ok; ci += kCons) {
        if (aborted()) {
          ok = false;
          break;
        }
        const int blk = (int)(ci - (long long)n * a.cps);
        const int ub = (int)(ci - cA) * a.U;
        int s = ub % a.ns;
        uint32_t ph = (uint32_t)(ub / a.ns) & 1u;
        const int t0c = blk * a.T;
        const bool rt = t0c >= a.kq;
        // stream and block of the units one ring length ahead (staged on release)
        int nn = n, nb = blk + ahead;
        while (nb >= a.cps) {
          nb -= a.cps;
          ++nn;
        }
        for (int k = 0; k < a.U; ++k) {
          const int u = ub + k;
          // Stages are shared by all warps, so a warp running ahead can reach
          // unit u while the stage still holds (or is still receiving) unit
          // u - ns; a parity wait alone cannot tell those phases apart. Wait
          // until unit u has been issued into the stage, then for its copies.
          bool got = true;
          for (int it = 0; *reinterpret_cast<volatile int*>(&last[s]) != u; ++it) {
            if (it > kWaitLimit || aborted()) {
              got = false;
              break;
            }
            __nanosleep(32);
          }
          if (!got || !mbar_wait_bounded(&full[s], ph)) {
            if (!aborted()) abort_now();
            ok = false;
          }
          if (!__all_sync(kFull, ok)) ok = false;
          if (!ok) break;
          const unsigned char* st = ring + (size_t)s * a.stage_bytes;
          const int t0 = t0c + k * a.UT;
          if (k == 0) rebuild(rt, st + a.off_km);
          const __half* kres = rt ? L.k.resid + (int64_t)n * L.k.resid_sstride + (int64_t)(t0 - a.kq) * kHeadDim
                                  : nullptr;
#pragma unroll 1
          for (int r0 = 0; r0 < a.UT && t0 + r0 < a.length; r0 += 32)
            subtile(st, r0, min(32, a.length - t0 - r0), rt, kres);
          __syncwarp();
          if (lane == 0 && u + a.ns < n_units) {
            fence_proxy_async_smem();
            issue(u + a.ns, s, nn, nb, k);
          }
          if (++s == a.ns) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) break;
      if (!finish_segment(sig, n, have)) break;
    }
  }
  __syncthreads();
  // Merges of the streams whose last partial this CTA wrote (at most two: only
  // a CTA's first and last streams can be shared with other CTAs). Warp w
  // merges heads w, w + 8, ...; loads are batched 8 partials at a time so the
  // warp waits for a few memory round trips.
  const int n_merge = aborted() ? 0 : min(ctl[7], 2);
  for (int mi = 0; mi < n_merge; ++mi) {
    __threadfence();
    const int n = ctl[8 + mi];
    const int Hkv = L.num_kv_heads;
    const int b = n / Hkv, kvh = n - b * Hkv;
    const long long va = (long long)n * (a.cps + a.vex), vb = va + a.cps - 1;  // the stream's first, last block
    const int cf = (int)(((va + 1) * a.P - 1) / a.n_virtual);
    const int cl = (int)(((vb + 1) * a.P - 1) / a.n_virtual);
    const int K = cl - cf + 1;
    const float* prn = a.part + (int64_t)n * a.jmax * H * kPartRow;
    for (int h = warp; h < H; h += kCons) {
      float M = -INFINITY;
      for (int j = lane; j < K; j += 32) M = fmaxf(M, __ldcg(prn + ((int64_t)j * H + h) * kPartRow + kHeadDim));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
      float Ls = 0.0f;
      float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int j0 = 0; j0 < K; j0 += 8) {
        float4 v[8];
        float mm[8], ll[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const bool in = j0 + jj < K;
          const float* pr = prn + ((int64_t)(j0 + jj) * H + h) * kPartRow;
          v[jj] = in ? __ldcg(reinterpret_cast<const float4*>(pr) + lane) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          mm[jj] = in ? __ldcg(pr + kHeadDim) : -INFINITY;
          ll[jj] = in ? __ldcg(pr + kHeadDim + 1) : 0.0f;
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float w = ex2(mm[jj] - M);
          Ls = fmaf(w, ll[jj], Ls);
          o.x = fmaf(w, v[jj].x, o.x);
          o.y = fmaf(w, v[jj].y, o.y);
          o.z = fmaf(w, v[jj].z, o.z);
          o.w = fmaf(w, v[jj].w, o.w);
        }
      }
      const int64_t row = (int64_t)b * a.num_q_heads + kvh * H + h;
      const int64_t base = row * kHeadDim + 4 * lane;
      const float4 r = finish_row4(a.sink_part, row, 4 * lane, o, M, Ls);
      if (a.out_dtype == KVQ_F32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + base) = r;
      } else {
        __half2 h01 = __floats2half2_rn(r.x, r.y), h23 = __floats2half2_rn(r.z, r.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&h01);
        u.y = *reinterpret_cast<uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.out) + base) = u;
      }
    }
  }
  if (tid == 0 && aborted()) {
    // copies still in flight: the last issue into every stage
    for (int s = 0; s < a.ns; ++s)
      if (last[s] >= 0) (void)mbar_wait_bounded(&full[s], (uint32_t)(last[s] / a.ns) & 1u);
  }
}

}  // namespace pipe
}  // namespace kvq
