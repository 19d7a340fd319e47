// Decode attention on the tensor cores for 1, 2, 4 or 8 query heads per
// kv-head: per-channel keys and per-token values of 3, 4 or 8 bits, with
// optional fp16 outliers.
//
// Per CTA: one (batch, kv-head) stream and one split of its tokens; each of
// the four warps owns a contiguous range of 32-token tiles and its own ring
// of 1-D bulk copies (codes, scales and outliers of K and V for one tile).
// Both products of a tile are small dense contractions (mma.sync m16n8k16,
// fp16 inputs, fp32 accumulation):
//   S[t][col]   = sum_slot K[t][slot] Q''[slot][col]      (M = 16 tokens)
//   O^T[c][col] = sum_t V^T[c][t] P'[t][col]               (M = 16 channels)
// The columns hold, for each query head, its fp32 operand as an fp16 pair
// hi + lo (head h: columns 2h and 2h + 1), so one mma carries about 22 bits
// and the two result columns are added in fp32.
//
// Codes enter the mma unconverted: a code n masked into the low bits of an
// fp16 half is the subnormal n * 2^-24 (exact, and the tensor cores multiply
// subnormals exactly), or 2^k n * 2^-24 when it sits k bits up; the 2^-24
// and 2^k factors are folded into the other operand (keys: per k-slot into
// Q'') or undone on the output row (values). So a register of two codes
// costs one AND (plus a byte permute where two tokens' codes meet).
//
// Dequantization is folded into the products (TurboQuant KV-cache page,
// demingchina.com/news/57821, §2.3): Q''[c] = q_c s_c per key block with the
// bias sum_c q_c z_c added in fp32; P'[t] = p_t s_t per value group with
// sum_t p_t z_t added once. Softmax runs in log2 units with a lazily moved
// running max; the four warps are merged by log-sum-exp at the end.
// Outliers (KVQuant page, cf-1.com/news/2306543, §2.2 item 3) add
// q_c (x - z_c) to a score and p_t (x - z_t) to the output.
#pragma once

#include "decode_merge.cuh"
#include "mma_frag.cuh"

namespace kvq {
namespace tc {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kRows = 32;  // tokens per warp tile (two m16 tiles)
constexpr float kLazy = 8.0f;

// ---------------------------------------------------------------------------
// Values: m-tile mv, output row half r (0: m-row g, 1: m-row g+8) -> channel,
// shift and value group.
//  4-bit (group VG): a thread's bytes are VG/16 consecutive bytes of each
//         group at q*VG/2 + g*VG/16 (its eight bytes in all); m-tile mv uses
//         its byte mv: low nibble -> m-row g, high nibble -> m-row g+8
//         (4 bits up).
//  8-bit: VG/8 consecutive bytes per group at q*VG + g*VG/8 (sixteen in
//         all); m-tile mv uses its bytes 2mv (m-row g) and 2mv+1 (g+8).
//  3-bit (VG = 128): words g and g+8 of the row; m-tile mv = code mv of
//         word g (m-row g) and of word g+8 (m-row g+8, none past word 12).
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int val3_shift_of_code(int i) {
  return i == 0 ? 0 : i == 1 ? 3 : i == 2 ? 6 : i == 3 ? 1 : i == 4 ? 4 : i == 5 ? 7
       : i == 6 ? 2 : i == 7 ? 5 : i == 8 ? 0 : 3;
}

template <int VB, int VG>
__device__ __forceinline__ void val_row(int mv, int g, int r, int& ch, int& shift, int& q) {
  if (VB == 4) {
    constexpr int bpt = VG / 16;
    q = mv / bpt;
    const int beta = q * (VG / 2) + g * bpt + (mv % bpt);
    ch = 2 * beta + r;
    shift = r ? 4 : 0;
  } else if (VB == 8) {
    constexpr int mpt = VG / 16;
    q = mv / mpt;
    ch = q * VG + g * (VG / 8) + 2 * (mv % mpt) + r;
    shift = 0;
  } else {
    q = 0;
    ch = 10 * (g + 8 * r) + mv;
    shift = val3_shift_of_code(mv);
  }
}

template <int KB, int VB, int VG, int NT, bool OUTL>
struct Cfg {
  static constexpr int KW = Pack<KB>::kWords, VW = Pack<VB>::kWords;
  static constexpr int KC = kRows * KW * 4;
  static constexpr int VC = kRows * VW * 4;
  static constexpr int KMETA = kHeadDim * 4;
  static constexpr int VGPR = kHeadDim / VG;
  static constexpr int VMETA = kRows * VGPR * 4 < 128 ? 128 : kRows * VGPR * 4;
  static constexpr int STAGE0 = KC + VC + KMETA + VMETA;  // + outliers: 4 arrays of kRows * k entries
  static constexpr int kStages = 2;
  static constexpr int MTV = VB == 3 ? 10 : 8;  // value m-tiles
  static constexpr int H = 4 * NT;              // head slots
  static constexpr int FRAG = 32 * NT * 16 * 4;  // key B fragments of the warp
  static constexpr int KBIAS = 2 * 8 * 4;        // bias and score factor per head
  static constexpr int OUTS = OUTL ? (2 * kRows * H + H * kHeadDim) * 4 : 0;
  static constexpr int WSCR = FRAG + KBIAS + OUTS;
  // With one query head (a run-time case of NT = 1) only head 0's output
  // corrections and query rows are kept: about 13 KB less per CTA, which
  // lets four outlier CTAs share an SM instead of three.
  static constexpr int OUTS1 = OUTL ? kHeadDim * 4 : 0;
  static constexpr int WSCR1 = FRAG + KBIAS + OUTS1;
  static constexpr size_t kMergeBytes = (size_t)kWarps * H * kHeadDim * 4;
  __host__ __device__ static constexpr int stage(int kout) { return STAGE0 + (OUTL ? 8 * kRows * kout : 0); }
  __host__ __device__ static constexpr size_t big(int kout) {
    return (size_t)kWarps * kStages * stage(kout) > kMergeBytes ? (size_t)kWarps * kStages * stage(kout)
                                                                 : kMergeBytes;
  }
  __host__ __device__ static constexpr size_t smem_bytes(int kout, bool one = false) {
    return big(kout) + (size_t)kWarps * (one ? WSCR1 : WSCR) + 2 * (one ? 1 : H) * kHeadDim * 4 /*qf, qm*/ +
           kWarps * H * 2 * 4 /*m, l*/ + kWarps * kStages * 8 + 16;
  }
};

// GF: 0, or the query heads per kv-head fixed at compile time (1, or every
// head slot: 4 NT), which removes the per-head guards and the run-time
// choice of the one-head path.
template <int KB, int VB, int VG, int NT, bool OUTL, int GF>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 4 : 3)
    decode_tc_kernel(LayerDev L, DecodeArgs a) {
  using C = Cfg<KB, VB, VG, NT, OUTL>;
  constexpr int S = C::kStages;
  constexpr int VGPR = C::VGPR;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int split = blockIdx.x, n = blockIdx.y;
  const int b = n / L.num_kv_heads;
  const int kvh = n - b * L.num_kv_heads;
  const int G = GF ? GF : a.gqa;  // query heads of this kv-head (<= 4 NT)
  const int hq0 = kvh * G;

  constexpr int H = C::H;
  const int kout = OUTL ? L.outliers : 0;
  const int STG = C::stage(kout);
  const size_t big = C::big(kout);
  unsigned char* stages = smem;
  float* mo = reinterpret_cast<float*>(smem);  // merge area, after the main loop: [warps][H][128]
  const bool one_head = NT == 1 && G == 1;  // warp-uniform
  const int HQ = one_head ? 1 : H;           // query rows and output-correction rows kept
  const size_t wsz = one_head ? C::WSCR1 : C::WSCR;
  unsigned char* wscr = smem + big + (size_t)warp * wsz;
  uint32_t* frag = reinterpret_cast<uint32_t*>(wscr);           // [32][NT][8][2]
  float* kbias = reinterpret_cast<float*>(wscr + C::FRAG);       // [8] bias, [8] score factor
  float* ocs = reinterpret_cast<float*>(wscr + C::FRAG + C::KBIAS);  // [32 rows][H] score corrections
  float* pst = ocs + kRows * H;                                   // [32 rows][H] probabilities
  float* ocr = one_head ? ocs : pst + kRows * H;                  // [HQ][128] output corrections
  float* qf = reinterpret_cast<float*>(smem + big + (size_t)kWarps * wsz);  // [HQ][128]
  float* qm = qf + HQ * kHeadDim;                                 // [HQ][128] qf * 2^-shift
  float* ml = qm + HQ * kHeadDim;                                 // [warps][H][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ml + kWarps * H * 2);

  // variable lengths: this batch row's tokens and its quantized key blocks
  const int len = a.varlen ? a.lens[b] : a.length;
  const int kq = a.varlen ? len / L.k.group * L.k.group : a.k_quant_len;
  const int row_begin = split * a.tiles_per_split * kTile;
  const int row_end = max(row_begin, min(row_begin + a.tiles_per_split * kTile, len));  // empty past a short row
  const int ntiles = (row_end - row_begin + kRows - 1) / kRows;
  const int per_warp = (ntiles + kWarps - 1) / kWarps;
  const int w_first = min(warp * per_warp, ntiles);
  const int w_count = min(per_warp, ntiles - w_first);
  const int Gk = L.k.group;

  const uint32_t* kcodes = L.k.codes + (int64_t)n * L.k.codes_sstride;
  const uint32_t* vcodes = L.v.codes + (int64_t)n * L.v.codes_sstride;
  const unsigned char* kmeta = L.k.meta + (int64_t)n * L.k.meta_sstride;
  const unsigned char* vmeta = L.v.meta + (int64_t)n * L.v.meta_sstride;

  uint64_t* wb = bars + warp * S;
  auto stage_ptr = [&](int s) { return stages + (size_t)(warp * S + s) * STG; };
  // Staging of tile ti into stage s (one lane issues every copy).
  auto issue = [&](int ti, int s) {
    unsigned char* base = stage_ptr(s);
    const int t0 = row_begin + (w_first + ti) * kRows;
    const bool rt = t0 >= kq;
    const uint32_t vmb = (uint32_t)(kRows * VGPR * 4);
    const uint32_t ob = OUTL ? (uint32_t)(kRows * kout * 2) : 0u;
    mbar_arrive_expect_tx(&wb[s], C::VC + vmb + 2 * ob + (rt ? 0u : C::KC + C::KMETA + 2 * ob));
    if (!rt) {
      bulk_g2s(base, kcodes + (int64_t)t0 * C::KW, C::KC, &wb[s]);
      bulk_g2s(base + C::KC + C::VC, kmeta + (int64_t)(t0 / Gk) * kHeadDim * 4, C::KMETA, &wb[s]);
    }
    bulk_g2s(base + C::KC, vcodes + (int64_t)t0 * C::VW, C::VC, &wb[s]);
    bulk_g2s(base + C::KC + C::VC + C::KMETA, vmeta + (int64_t)t0 * VGPR * 4, vmb, &wb[s]);
    if (OUTL) {
      // every row holds exactly kout entries: the tile's entries are contiguous
      unsigned char* ot = base + C::STAGE0;
      const int64_t e0 = (int64_t)t0 * kout;
      if (!rt) {
        bulk_g2s(ot, L.k.col + (int64_t)n * L.k.out_sstride + e0, ob, &wb[s]);
        bulk_g2s(ot + ob, L.k.val + (int64_t)n * L.k.out_sstride + e0, ob, &wb[s]);
      }
      bulk_g2s(ot + 2 * ob, L.v.col + (int64_t)n * L.v.out_sstride + e0, ob, &wb[s]);
      bulk_g2s(ot + 3 * ob, L.v.val + (int64_t)n * L.v.out_sstride + e0, ob, &wb[s]);
    }
  };
  // lane 0 of each warp: its barriers and its first copies, before the
  // query load, so that the two latencies overlap
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&wb[s], 1);
    mbar_fence_init();
    for (int s = 0; s < S && s < w_count; ++s) issue(s, s);
  }

  for (int i = tid; i < HQ * kHeadDim; i += kThreads) {
    const int h = i >> 7, c = i & 127;
    const float v = h < G ? __half2float(a.q[((int64_t)b * a.num_q_heads + hq0 + h) * kHeadDim + c]) *
                                a.scale_log2
                          : 0.0f;
    qf[i] = v;
    qm[i] = v * __uint_as_float((uint32_t)(127 - key_shift<KB>(c)) << 23);
  }
  for (int i = lane; i < 32 * NT * 16; i += 32) frag[i] = 0u;
  if (OUTL)
    for (int i = lane; i < HQ * kHeadDim; i += 32) ocr[i] = 0.0f;
  __syncthreads();

  // ---- state ------------------------------------------------------------------
  uint32_t bq[NT][8][2];
  float kb[NT], kf[NT];  // bias and score factor of the thread's head in the current key block
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    kb[nt] = 0.0f;
    kf[nt] = 0.0f;
  }
  // value side: P' = p s_t 2^(6 - ev[q]) with ev[q] the largest scale exponent
  // of group q seen by the warp (so |P'| < 2^15 while p <= 2^8)
  int ev[VGPR];
#pragma unroll
  for (int q = 0; q < VGPR; ++q) ev[q] = -127;
  int cur_blk = -1;
  float m_run[NT], l_run[NT], zacc[NT][VGPR];
  float o[C::MTV][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.0f;
#pragma unroll
    for (int q = 0; q < VGPR; ++q) zacc[nt][q] = 0.0f;
#pragma unroll
    for (int mv = 0; mv < C::MTV; ++mv)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mv][nt][e] = 0.0f;
  }

  // key slots this lane fills when the Q'' fragments are rebuilt: thread
  // t4 = lane & 3 of chunk kc = lane >> 2, slots s0..s3
  int cs[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int sh;
    key_slot<KB>(lane & 3, lane >> 2, k, cs[k], sh);
  }

  // Per tile: front (wait for the copies, key operand rebuild, scores,
  // outliers, tile max), middle (running max, probabilities, value outliers,
  // value-scale exponents, P' per token with one head), back (PV, then the
  // stage is refilled). Issuing QK^T of tile i+1 before PV of tile i was
  // measured slower (register pressure), so the phases run in order.
  bool failed = false;
  int fail_tile = 0;
  float sc[NT][2][2], mx_n[NT], p[NT][2][2];
  float vsf[VGPR];  // 2^(6 - ev[q])
  uint32_t pw[VGPR];
  // One query head: value-outlier corrections p_t (x - z_t) of the lane's
  // tokens are summed in registers for the first four channels the lane
  // meets (outliers gather in a few channels, which then stay in registers
  // for the whole split) and added into ocr at the end; other channels go
  // to ocr by shared-memory atomics. Evicting entries would send the
  // frequent channels back through the atomics, which conflict.
  int occ[4];
  float oca[4];
  int ovic = 0;  // entries in use
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    occ[k] = -1;
    oca[k] = 0.0f;
  }

  auto front = [&](int tj) -> bool {
    {
      if (!mbar_wait_bounded(&wb[tj % S], (uint32_t)(tj / S) & 1u)) return false;
      __syncwarp();
      const int t0 = row_begin + (w_first + tj) * kRows;
      const bool rt = t0 >= kq;
      unsigned char* base = stage_ptr(tj % S);
      const uint32_t* kc_s = reinterpret_cast<const uint32_t*>(base);
      const uint32_t* vc_s = reinterpret_cast<const uint32_t*>(base + C::KC);
      const __half2* km = reinterpret_cast<const __half2*>(base + C::KC + C::VC);
      const __half2* vm = reinterpret_cast<const __half2*>(base + C::KC + C::VC + C::KMETA);
      const unsigned char* ot = base + C::KC + C::VC + C::KMETA + C::VMETA;
      (void)rt; (void)kc_s; (void)vc_s; (void)km; (void)vm; (void)ot;
      // ---- key block change: rebuild the Q'' fragments and the bias -------------
      if (!rt && (t0 / Gk) != cur_blk) {
        cur_blk = t0 / Gk;
        const int kt4 = lane & 3, kkc = lane >> 2;
        float sv[4], zv[4];
  #pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 sz = __half22float2(km[cs[k]]);
          sv[k] = sz.x;
          zv[k] = sz.y;
        }
        float zp[H];
  #pragma unroll
        for (int h = 0; h < H; ++h) {
          zp[h] = 0.0f;
          if (h < G) {
            float v[4], mx = 0.0f;
  #pragma unroll
            for (int k = 0; k < 4; ++k) {
              v[k] = qm[h * kHeadDim + cs[k]] * sv[k];
              mx = fmaxf(mx, fabsf(v[k]));
              zp[h] = fmaf(qf[h * kHeadDim + cs[k]], zv[k], zp[h]);
            }
            // scale the head's operand so that its largest |Q''| lies in [2^14, 2^15)
            const uint32_t mb = __reduce_max_sync(kFull, __float_as_uint(mx));
            const int e = mb ? (int)(mb >> 23) - 127 : 0;
            const float up = exp2i(14 - e);
            const int lh = 8 * (h & 3) + kt4;  // lane of column 2(h&3) (hi); lh + 4 holds lo
  #pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t lo;
              const uint32_t hi = split_pair(v[2 * j] * up, v[2 * j + 1] * up, lo);
              frag[((lh * NT + (h >> 2)) * 8 + kkc) * 2 + j] = hi;
              frag[(((lh + 4) * NT + (h >> 2)) * 8 + kkc) * 2 + j] = lo;
            }
            if (lane == 0) kbias[8 + h] = exp2i(24 - (14 - e));  // undoes 2^-24 and the head scale
          }
        }
        // bias sum_c q_c z_c of every head: butterfly reduce-scatter (lane keeps
        // head (lane >> 2) & (H - 1)), then the sum over the remaining lanes
        {
          float kept[H];
  #pragma unroll
          for (int h = 0; h < H; ++h) kept[h] = zp[h];
  #pragma unroll
          for (int half = H / 2, off = 8 * (H / 4); half >= 1; half >>= 1, off >>= 1) {
            const bool upper = (lane & off) != 0;
  #pragma unroll
            for (int i = 0; i < half; ++i) {
              const float send = upper ? kept[i] : kept[i + half];
              const float keep = upper ? kept[i + half] : kept[i];
              kept[i] = keep + __shfl_xor_sync(kFull, send, off);
            }
          }
          float tot = kept[0];
          if (H == 4) tot += __shfl_xor_sync(kFull, tot, 16);
          tot += __shfl_xor_sync(kFull, tot, 2);
          tot += __shfl_xor_sync(kFull, tot, 1);
          if ((lane & 3) == 0 && (lane >> 2) < H) kbias[(lane >> 2) & (H - 1)] = tot;
        }
        __syncwarp();
  #pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
  #pragma unroll
          for (int kc = 0; kc < 8; kc += 2) {
            const uint4 v = *reinterpret_cast<const uint4*>(&frag[((lane * NT + nt) * 8 + kc) * 2]);
            bq[nt][kc][0] = v.x;
            bq[nt][kc][1] = v.y;
            bq[nt][kc + 1][0] = v.z;
            bq[nt][kc + 1][1] = v.w;
          }
          kb[nt] = (4 * nt + t4 < G) ? kbias[4 * nt + t4] : 0.0f;
          kf[nt] = (4 * nt + t4 < G) ? kbias[8 + 4 * nt + t4] : 0.0f;
        }
        __syncwarp();
      }

      // ---- scores: sc[nt][mt][r], rows 16 mt + g + 8 r, head 4 nt + t4 -----------
      if (!rt) {
  #pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int r0 = 16 * mt + g, r1 = r0 + 8;
          // one accumulator chain per head tile, two (even / odd chunks) when
          // there is a single head tile
          constexpr int CH = NT == 1 ? 2 : 1;
          float acc[NT][CH][4];
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
            for (int e = 0; e < 4 * CH; ++e) acc[nt][e >> 2][e & 3] = 0.0f;
          if (KB == 4) {
            const uint4 A0 = reinterpret_cast<const uint4*>(kc_s + r0 * 16)[t4];
            const uint4 A1 = reinterpret_cast<const uint4*>(kc_s + r1 * 16)[t4];
            const uint32_t w0[4] = {A0.x, A0.y, A0.z, A0.w}, w1[4] = {A1.x, A1.y, A1.z, A1.w};
  #pragma unroll
            for (int j = 0; j < 4; ++j) {
  #pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t x0 = w0[j] >> (8 * h), x1 = w1[j] >> (8 * h);
  #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma(acc[nt][h % CH], x0 & 0x000F000Fu, x1 & 0x000F000Fu, x0 & 0x00F000F0u, x1 & 0x00F000F0u,
                      bq[nt][2 * j + h][0], bq[nt][2 * j + h][1]);
              }
            }
          } else if (KB == 8) {
  #pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
              const uint4 A0 = reinterpret_cast<const uint4*>(kc_s + r0 * 32)[2 * t4 + hq];
              const uint4 A1 = reinterpret_cast<const uint4*>(kc_s + r1 * 32)[2 * t4 + hq];
              const uint32_t w0[4] = {A0.x, A0.y, A0.z, A0.w}, w1[4] = {A1.x, A1.y, A1.z, A1.w};
  #pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int kc = 4 * hq + j;
  #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma(acc[nt][j % CH], w0[j] & 0x00FF00FFu, w1[j] & 0x00FF00FFu, (w0[j] >> 8) & 0x00FF00FFu,
                      (w1[j] >> 8) & 0x00FF00FFu, bq[nt][kc][0], bq[nt][kc][1]);
              }
            }
          } else {
            uint32_t P0[16], P1[16];
  #pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const uint32_t* rw = kc_s + (rr ? r1 : r0) * 13;
              uint32_t* P = rr ? P1 : P0;
              const uint32_t X[3] = {rw[t4], rw[t4 + 4], rw[t4 + 8]};
  #pragma unroll
              for (int i = 0; i < 3; ++i) {
                P[4 * i + 0] = X[i] & 0x001C0007u;
                P[4 * i + 1] = X[i] & 0x00E00038u;
                P[4 * i + 2] = (X[i] >> 6) & 0x001C0007u;
                P[4 * i + 3] = (X[i] >> 9) & 0x001C0007u;
              }
              const uint32_t ab = __byte_perm(X[0] >> 12, X[1] >> 12, 0x5410u);
              const uint32_t cd = __byte_perm(X[2] >> 12, rw[12] >> (6 * t4), 0x5410u);
              P[12] = ab & 0x00070007u;
              P[13] = ab & 0x00380038u;
              P[14] = cd & 0x00070007u;
              P[15] = cd & 0x00380038u;
            }
  #pragma unroll
            for (int kc = 0; kc < 8; ++kc)
  #pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma(acc[nt][kc % CH], P0[2 * kc], P1[2 * kc], P0[2 * kc + 1], P1[2 * kc + 1], bq[nt][kc][0],
                    bq[nt][kc][1]);
          }
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float c0 = acc[nt][0][0] + acc[nt][0][1], c1 = acc[nt][0][2] + acc[nt][0][3];
            if (CH == 2) {
              c0 += acc[nt][CH - 1][0] + acc[nt][CH - 1][1];
              c1 += acc[nt][CH - 1][2] + acc[nt][CH - 1][3];
            }
            sc[nt][mt][0] = fmaf(c0, kf[nt], kb[nt]);
            sc[nt][mt][1] = fmaf(c1, kf[nt], kb[nt]);
          }
        }
      } else {
        // fp16 residual keys (the last partial key block) on the CUDA cores
        const __half* res = L.k.resid + (int64_t)n * L.k.resid_sstride + (int64_t)(t0 - kq) * kHeadDim;
  #pragma unroll
        for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
          for (int mt = 0; mt < 2; ++mt)
  #pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int row = 16 * mt + g + 8 * r, h = 4 * nt + t4;
              float d = 0.0f;
              if (t0 + row < row_end && h < G) {
                const __half2* kr = reinterpret_cast<const __half2*>(res + (size_t)row * kHeadDim);
                const float* qh = qf + h * kHeadDim;
                for (int c2 = 0; c2 < kHeadDim / 2; ++c2) {
                  const float2 x = __half22float2(kr[c2]);
                  d = fmaf(qh[2 * c2], x.x, fmaf(qh[2 * c2 + 1], x.y, d));
                }
              }
              sc[nt][mt][r] = d;
            }
      }

      // ---- key outliers: score += q_c (x - z_c), one row per lane ---------------
      if (OUTL && one_head) {
        if (!rt) {
          // one head: the lane's row correction reaches the score owners by
          // shuffles
          const __half* kval = reinterpret_cast<const __half*>(ot + 2 * kRows * kout);
          const int ke = (t0 + lane < row_end) ? kout : 0;
          const uint16_t* kcol = reinterpret_cast<const uint16_t*>(ot);
          float corr = 0.0f;
#pragma unroll 2
          for (int e = 0; e < ke; ++e) {
            const int c = kcol[lane * kout + e] & (kHeadDim - 1);
            const float d = __half2float(kval[lane * kout + e]) - __high2float(km[c]);
            corr = fmaf(qf[c], d, corr);
          }
  #pragma unroll
          for (int mt = 0; mt < 2; ++mt)
  #pragma unroll
            for (int r = 0; r < 2; ++r) sc[0][mt][r] += __shfl_sync(kFull, corr, 16 * mt + g + 8 * r);
        }
      } else if (OUTL) {
        if (!rt) {
          const __half* kval = reinterpret_cast<const __half*>(ot + 2 * kRows * kout);
          const int ke = (t0 + lane < row_end) ? kout : 0;
          const uint16_t* kcol = reinterpret_cast<const uint16_t*>(ot);
          float corr[H];
  #pragma unroll
          for (int h = 0; h < H; ++h) corr[h] = 0.0f;
          for (int e = 0; e < ke; ++e) {
            const int c = kcol[lane * kout + e] & (kHeadDim - 1);
            const float d = __half2float(kval[lane * kout + e]) - __high2float(km[c]);
  #pragma unroll
            for (int h = 0; h < H; ++h) corr[h] = fmaf(qf[h * kHeadDim + c], d, corr[h]);
          }
  #pragma unroll
          for (int h = 0; h < H; ++h) ocs[lane * H + h] = corr[h];
          __syncwarp();
  #pragma unroll
          for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
            for (int mt = 0; mt < 2; ++mt)
  #pragma unroll
              for (int r = 0; r < 2; ++r) sc[nt][mt][r] += ocs[(16 * mt + g + 8 * r) * H + 4 * nt + t4];
          __syncwarp();
        }
      }

      // ---- online softmax (per thread: head 4 nt + t4) --------------------------
  #pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const bool hv = 4 * nt + t4 < G;
  #pragma unroll
        for (int mt = 0; mt < 2; ++mt)
  #pragma unroll
          for (int r = 0; r < 2; ++r)
            if (!hv || t0 + 16 * mt + g + 8 * r >= row_end) sc[nt][mt][r] = -INFINITY;
        float& mt_ = mx_n[nt];
        mt_ = fmaxf(fmaxf(sc[nt][0][0], sc[nt][0][1]), fmaxf(sc[nt][1][0], sc[nt][1][1]));
        mt_ = fmaxf(mt_, __shfl_xor_sync(kFull, mt_, 4));
        mt_ = fmaxf(mt_, __shfl_xor_sync(kFull, mt_, 8));
        mt_ = fmaxf(mt_, __shfl_xor_sync(kFull, mt_, 16));
      }
    }
    return true;
  };

  auto middle = [&](int tj) {
      const int t0 = row_begin + (w_first + tj) * kRows;
      const bool rt = t0 >= kq;
      unsigned char* base = stage_ptr(tj % S);
      const uint32_t* kc_s = reinterpret_cast<const uint32_t*>(base);
      const uint32_t* vc_s = reinterpret_cast<const uint32_t*>(base + C::KC);
      const __half2* km = reinterpret_cast<const __half2*>(base + C::KC + C::VC);
      const __half2* vm = reinterpret_cast<const __half2*>(base + C::KC + C::VC + C::KMETA);
      const unsigned char* ot = base + C::KC + C::VC + C::KMETA + C::VMETA;
      (void)rt; (void)kc_s; (void)vc_s; (void)km; (void)vm; (void)ot;
      // ---- online softmax, second half: move the running max, probabilities ----
  #pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float mt_ = mx_n[nt];
        const bool up = mt_ > m_run[nt] + kLazy;
        if (__any_sync(kFull, up)) {
          const float mnew = up ? mt_ : m_run[nt];
          const float al = up ? exp2f(m_run[nt] - mnew) : 1.0f;
          l_run[nt] *= al;
          // with one query head the zero-point sums are kept per token lane,
          // so every lane takes head 0's factor (lane 0 holds it)
          const float alz = one_head ? __shfl_sync(kFull, al, 0) : al;
  #pragma unroll
          for (int q = 0; q < VGPR; ++q) zacc[nt][q] *= alz;
  #pragma unroll
          for (int mv = 0; mv < C::MTV; ++mv)
  #pragma unroll
            for (int e = 0; e < 4; ++e) o[mv][nt][e] *= al;
          if (OUTL) {
            // output corrections of head h follow that head's factor
            __syncwarp();
  #pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              const float alh = __shfl_sync(kFull, al, hh);
              const int h = 4 * nt + hh;
              if (h < HQ)
  #pragma unroll
                for (int k = 0; k < 4; ++k) ocr[h * kHeadDim + lane + 32 * k] *= alh;
            }
            if (one_head) {
              const float al0 = __shfl_sync(kFull, al, 0);
#pragma unroll
              for (int k = 0; k < 4; ++k) oca[k] *= al0;
            }
            __syncwarp();
          }
          m_run[nt] = mnew;
        }
  #pragma unroll
        for (int mt = 0; mt < 2; ++mt)
  #pragma unroll
          for (int r = 0; r < 2; ++r) {
            p[nt][mt][r] = sc[nt][mt][r] == -INFINITY ? 0.0f : exp2f(sc[nt][mt][r] - m_run[nt]);
            l_run[nt] += p[nt][mt][r];
          }
      }

      // ---- value outliers: o_c += p_t (x - z_t), one row per lane ----------------
      if (OUTL && one_head) {
        const int src = 4 * (lane & 7);  // head 0 lives in lanes with t4 = 0
        const float p00 = __shfl_sync(kFull, p[0][0][0], src), p01 = __shfl_sync(kFull, p[0][0][1], src);
        const float p10 = __shfl_sync(kFull, p[0][1][0], src), p11 = __shfl_sync(kFull, p[0][1][1], src);
        const float pl = (lane & 16) ? ((lane & 8) ? p11 : p10) : ((lane & 8) ? p01 : p00);
        if (t0 + lane < row_end) {
          const uint16_t* vcol = reinterpret_cast<const uint16_t*>(ot + 4 * kRows * kout);
          const __half* vval = reinterpret_cast<const __half*>(ot + 6 * kRows * kout);
          // zero points of the token's value groups (at most two: VG >= 64)
          float zq[VGPR];
#pragma unroll
          for (int q = 0; q < VGPR; ++q) zq[q] = __high2float(vm[lane * VGPR + q]);
          auto upd = [&](int c, float v) {
            bool hit = false;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (occ[k] == c) {
                oca[k] += v;
                hit = true;
              }
            if (!hit) {
              if (ovic < 4) {  // a free entry: the channel keeps it
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  if (k == ovic) {
                    occ[k] = c;
                    oca[k] = v;
                  }
                ++ovic;
              } else {
                atomicAdd(&ocr[c], v);
              }
            }
          };
          // two entries per step: their loads overlap
          for (int e = 0; e < kout; e += 2) {
            const bool two = e + 1 < kout;
            const int i0 = lane * kout + e, i1 = two ? i0 + 1 : i0;
            const int c0 = vcol[i0] & (kHeadDim - 1), c1 = vcol[i1] & (kHeadDim - 1);
            const float x0 = __half2float(vval[i0]), x1 = __half2float(vval[i1]);
            const float z0 = VGPR == 1 ? zq[0] : (c0 < VG ? zq[0] : zq[VGPR - 1]);
            const float z1 = VGPR == 1 ? zq[0] : (c1 < VG ? zq[0] : zq[VGPR - 1]);
            upd(c0, pl * (x0 - z0));
            if (two) upd(c1, pl * (x1 - z1));
          }
        }
      } else if (OUTL) {
  #pragma unroll
        for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
          for (int mt = 0; mt < 2; ++mt)
  #pragma unroll
            for (int r = 0; r < 2; ++r) pst[(16 * mt + g + 8 * r) * H + 4 * nt + t4] = p[nt][mt][r];
        __syncwarp();
        if (t0 + lane < row_end) {
          const uint16_t* vcol = reinterpret_cast<const uint16_t*>(ot + 4 * kRows * kout);
          const __half* vval = reinterpret_cast<const __half*>(ot + 6 * kRows * kout);
          for (int e = 0; e < kout; ++e) {
            const int c = vcol[lane * kout + e] & (kHeadDim - 1);
            const float d = __half2float(vval[lane * kout + e]) - __high2float(vm[lane * VGPR + c / VG]);
            for (int h = 0; h < G; ++h) atomicAdd(&ocr[h * kHeadDim + c], pst[lane * H + h] * d);
          }
        }
        __syncwarp();
      }

      // ---- value scale exponents of the tile (per group; lane = row), rescale
      //      the group's accumulators when one grows -------------------------------
  #pragma unroll
      for (int q = 0; q < VGPR; ++q) {
        const float sl = (t0 + lane < row_end) ? __low2float(vm[lane * VGPR + q]) : 0.0f;
        const uint32_t mb = __reduce_max_sync(kFull, __float_as_uint(sl));
        const int e = mb ? (int)(mb >> 23) - 127 : -127;
        if (e > ev[q]) {  // warp-uniform
          const float f = exp2i(max(ev[q] - e, -126));
  #pragma unroll
          for (int mv = 0; mv < C::MTV; ++mv) {
            int ch, sh, qq;
            val_row<VB, VG>(mv, 0, 0, ch, sh, qq);
            if (qq == q)
  #pragma unroll
              for (int nt = 0; nt < NT; ++nt)
  #pragma unroll
                for (int k = 0; k < 4; ++k) o[mv][nt][k] *= f;
          }
          ev[q] = e;
        }
        vsf[q] = exp2i(6 - ev[q]);
      }

      // ---- one query head: P' per token, one token per lane --------------------
      // pw[q] = (lo, hi) fp16 pair of p_t s_t 2^(6 - ev[q]) for token t = lane
      if (one_head) {
        const int src = 4 * (lane & 7);  // head 0 lives in lanes with t4 = 0
        const float p00 = __shfl_sync(kFull, p[0][0][0], src), p01 = __shfl_sync(kFull, p[0][0][1], src);
        const float p10 = __shfl_sync(kFull, p[0][1][0], src), p11 = __shfl_sync(kFull, p[0][1][1], src);
        const float pl = (lane & 16) ? ((lane & 8) ? p11 : p10) : ((lane & 8) ? p01 : p00);
        const bool valid = t0 + lane < row_end;
  #pragma unroll
        for (int q = 0; q < VGPR; ++q) {
          const float2 sz = __half22float2(vm[lane * VGPR + q]);
          zacc[0][q] = valid ? fmaf(pl, sz.y, zacc[0][q]) : zacc[0][q];
          const float e = valid ? pl * (sz.x * vsf[q]) : 0.0f;
          const float h = __half2float(__float2half_rn(e));
          pw[q] = f2h2(__fsub_rn(e, h), e);
        }
      }

  };

  auto back = [&](int tj) {
      const int t0 = row_begin + (w_first + tj) * kRows;
      const bool rt = t0 >= kq;
      unsigned char* base = stage_ptr(tj % S);
      const uint32_t* kc_s = reinterpret_cast<const uint32_t*>(base);
      const uint32_t* vc_s = reinterpret_cast<const uint32_t*>(base + C::KC);
      const __half2* km = reinterpret_cast<const __half2*>(base + C::KC + C::VC);
      const __half2* vm = reinterpret_cast<const __half2*>(base + C::KC + C::VC + C::KMETA);
      const unsigned char* ot = base + C::KC + C::VC + C::KMETA + C::VMETA;
      (void)rt; (void)kc_s; (void)vc_s; (void)km; (void)vm; (void)ot;
      // ---- PV per 16-token step --------------------------------------------------
  #pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        // B operands P' = p s_t per value group (hi/lo columns)
        uint32_t bp[VGPR][NT][2];
        const int rA = 16 * ks + g, rB = rA + 8;  // rows this thread owns in the C layout
        const bool vA = t0 + rA < row_end, vB = t0 + rB < row_end;
        const int L1 = 4 * (2 * t4) + (g >> 1), L2 = 4 * (2 * t4 + 1) + (g >> 1);
        if (one_head) {
          const uint32_t sel = (g & 1) ? 0x5410u : 0x7632u;
          const int tk = 16 * ks + 2 * t4;
  #pragma unroll
          for (int q = 0; q < VGPR; ++q) {
            const uint32_t X1 = __shfl_sync(kFull, pw[q], tk), X2 = __shfl_sync(kFull, pw[q], tk + 1);
            const uint32_t X3 = __shfl_sync(kFull, pw[q], tk + 8), X4 = __shfl_sync(kFull, pw[q], tk + 9);
            bp[q][0][0] = __byte_perm(X1, X2, sel);
            bp[q][0][1] = __byte_perm(X3, X4, sel);
          }
        } else {
  #pragma unroll
          for (int q = 0; q < VGPR; ++q) {
            const float2 szA = __half22float2(vm[rA * VGPR + q]);
            const float2 szB = __half22float2(vm[rB * VGPR + q]);
            const float sA = vA ? szA.x * vsf[q] : 0.0f, sB = vB ? szB.x * vsf[q] : 0.0f;
            const float zA = vA ? szA.y : 0.0f, zB = vB ? szB.y : 0.0f;
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              zacc[nt][q] = fmaf(p[nt][ks][0], zA, fmaf(p[nt][ks][1], zB, zacc[nt][q]));
              uint32_t lo;
              const uint32_t hi = split_pair(p[nt][ks][0] * sA, p[nt][ks][1] * sB, lo);
              const uint32_t H1 = __shfl_sync(kFull, hi, L1), H2 = __shfl_sync(kFull, hi, L2);
              const uint32_t O1 = __shfl_sync(kFull, lo, L1), O2 = __shfl_sync(kFull, lo, L2);
              const uint32_t X1 = (g & 1) ? O1 : H1, X2 = (g & 1) ? O2 : H2;
              bp[q][nt][0] = __byte_perm(X1, X2, 0x5410u);
              bp[q][nt][1] = __byte_perm(X1, X2, 0x7632u);
            }
          }
        }
        // A operands: value codes of rows ra, ra+1 (k-slots 2t4, 2t4+1) and
        // ra+8, ra+9 (2t4+8, 2t4+9)
        const int ra = 16 * ks + 2 * t4;
        const int rows[4] = {ra, ra + 1, ra + 8, ra + 9};
        if (VB == 4) {
          uint32_t vw[4][2];
  #pragma unroll
          for (int k = 0; k < 4; ++k) {
            const unsigned char* rp = reinterpret_cast<const unsigned char*>(vc_s + rows[k] * 16);
            if (VG == 128) {
              const uint2 u = *reinterpret_cast<const uint2*>(rp + 8 * g);
              vw[k][0] = u.x;
              vw[k][1] = u.y;
            } else {  // VG == 64
              vw[k][0] = *reinterpret_cast<const uint32_t*>(rp + 4 * g);
              vw[k][1] = *reinterpret_cast<const uint32_t*>(rp + 32 + 4 * g);
            }
          }
  #pragma unroll
          for (int mv = 0; mv < 8; ++mv) {
            const uint32_t i = mv & 3;
            const uint32_t sel = i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12);
            const uint32_t x01 = __byte_perm(vw[0][mv >> 2], vw[1][mv >> 2], sel);
            const uint32_t x23 = __byte_perm(vw[2][mv >> 2], vw[3][mv >> 2], sel);
            const int q = mv / (VG / 16);
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma(o[mv][nt], x01 & 0x000F000Fu, x01 & 0x00F000F0u, x23 & 0x000F000Fu, x23 & 0x00F000F0u,
                  bp[q][nt][0], bp[q][nt][1]);
          }
        } else if (VB == 8) {
          uint32_t vw[4][4];
  #pragma unroll
          for (int k = 0; k < 4; ++k) {
            const unsigned char* rp = reinterpret_cast<const unsigned char*>(vc_s + rows[k] * 32);
            if (VG == 128) {
              const uint4 u = *reinterpret_cast<const uint4*>(rp + 16 * g);
              vw[k][0] = u.x; vw[k][1] = u.y; vw[k][2] = u.z; vw[k][3] = u.w;
            } else {  // VG == 64
              const uint2 u0 = *reinterpret_cast<const uint2*>(rp + 8 * g);
              const uint2 u1 = *reinterpret_cast<const uint2*>(rp + 64 + 8 * g);
              vw[k][0] = u0.x; vw[k][1] = u0.y; vw[k][2] = u1.x; vw[k][3] = u1.y;
            }
          }
  #pragma unroll
          for (int mv = 0; mv < 8; ++mv) {
            const uint32_t i = mv & 1;
            const uint32_t sel = (2 * i) | ((2 * i + 1) << 4) | ((4 + 2 * i) << 8) | ((5 + 2 * i) << 12);
            const uint32_t x01 = __byte_perm(vw[0][mv >> 1], vw[1][mv >> 1], sel);
            const uint32_t x23 = __byte_perm(vw[2][mv >> 1], vw[3][mv >> 1], sel);
            const int q = mv / (VG / 16);
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma(o[mv][nt], x01 & 0x00FF00FFu, (x01 >> 8) & 0x00FF00FFu, x23 & 0x00FF00FFu,
                  (x23 >> 8) & 0x00FF00FFu, bp[q][nt][0], bp[q][nt][1]);
          }
        } else {
          uint32_t vw[4][2];
  #pragma unroll
          for (int k = 0; k < 4; ++k) {
            vw[k][0] = vc_s[rows[k] * 13 + g];
            vw[k][1] = (g + 8 <= 12) ? vc_s[rows[k] * 13 + g + 8] : 0u;
          }
          constexpr uint32_t kSel[4] = {0x5410u, 0x6521u, 0x7632u, 0x7733u};
          constexpr int kSelOf[10] = {0, 0, 0, 1, 1, 1, 2, 2, 3, 3};
          constexpr uint32_t kMask[10] = {0x00070007u, 0x00380038u, 0x01C001C0u, 0x000E000Eu,
                                          0x00700070u, 0x03800380u, 0x001C001Cu, 0x00E000E0u,
                                          0x00070007u, 0x00380038u};
          uint32_t x[4][2][2];  // selector, word (g / g+8), row pair
  #pragma unroll
          for (int sI = 0; sI < 4; ++sI)
  #pragma unroll
            for (int wi = 0; wi < 2; ++wi) {
              x[sI][wi][0] = __byte_perm(vw[0][wi], vw[1][wi], kSel[sI]);
              x[sI][wi][1] = __byte_perm(vw[2][wi], vw[3][wi], kSel[sI]);
            }
  #pragma unroll
          for (int mv = 0; mv < 10; ++mv) {
            const int sI = kSelOf[mv];
            const uint32_t m = kMask[mv];
  #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma(o[mv][nt], x[sI][0][0] & m, x[sI][1][0] & m, x[sI][0][1] & m, x[sI][1][1] & m,
                  bp[0][nt][0], bp[0][nt][1]);
          }
        }
      }

      __syncwarp();
      if (lane == 0 && tj + S < w_count) {
        fence_proxy_async_smem();
        issue(tj + S, tj % S);
      }
  };

  for (int ti = 0; ti < w_count; ++ti) {
    if (!front(ti)) {
      failed = true;
      fail_tile = ti;
      break;
    }
    middle(ti);
    back(ti);
  }
  if (OUTL && one_head) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (occ[k] >= 0) atomicAdd(&ocr[occ[k]], oca[k]);
  }
  if (failed && lane == 0) {
    raise_status(L.status, kStatusTimeout);
    // copies still in flight: tiles fail_tile .. fail_tile + S - 1
    const int end = fail_tile + S;
    for (int tj = fail_tile; tj < w_count && tj < end; ++tj)
      (void)mbar_wait_bounded(&wb[tj % S], (uint32_t)(tj / S) & 1u);
  }

  // ---- warp totals over the row owners (lanes with the same t4; with one
  //      query head the zero-point sums were kept per token lane) --------------
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_run[nt] += __shfl_xor_sync(kFull, l_run[nt], off);
#pragma unroll
      for (int q = 0; q < VGPR; ++q) zacc[nt][q] += __shfl_xor_sync(kFull, zacc[nt][q], off);
    }
    if (NT == 1 && G == 1)
#pragma unroll
      for (int off = 1; off < 4; off <<= 1)
#pragma unroll
        for (int q = 0; q < VGPR; ++q) zacc[nt][q] += __shfl_xor_sync(kFull, zacc[nt][q], off);
  }
  __syncthreads();  // stages are free: reuse them for the merge buffers
  float* my = mo + warp * H * kHeadDim;  // [H heads][128]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 4 * nt + t4;
    if (h < G) {
#pragma unroll
      for (int mv = 0; mv < C::MTV; ++mv)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          int ch, sh, q;
          val_row<VB, VG>(mv, g, r, ch, sh, q);
          if (ch < kHeadDim) {
            float zq = zacc[nt][0];
            int eq = ev[0];
#pragma unroll
            for (int qq = 1; qq < VGPR; ++qq)
              if (qq == q) {
                zq = zacc[nt][qq];
                eq = ev[qq];
              }
            // undo 2^-24 of the codes, 2^sh of the code position and 2^(6 - ev)
            const float f = exp2i(18 - sh + eq);
            float v = fmaf(o[mv][nt][2 * r] + o[mv][nt][2 * r + 1], f, zq);
            if (OUTL) v += ocr[h * kHeadDim + ch];
            my[h * kHeadDim + ch] = v;
          }
        }
    }
  }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = 4 * nt + t4;
      ml[(warp * H + h) * 2] = w_count > 0 ? m_run[nt] : -INFINITY;
      ml[(warp * H + h) * 2 + 1] = l_run[nt];
    }
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
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[(w * H + h) * 2]);
    float ov = 0.0f, lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = ml[(w * H + h) * 2];
      const float wt = mw == -INFINITY ? 0.0f : exp2f(mw - M);
      ov = fmaf(wt, mo[(w * H + h) * kHeadDim + c], ov);
      lsum = fmaf(wt, ml[(w * H + h) * 2 + 1], lsum);
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

template <int KB, int VB, int VG, int NT, bool OUTL, int GF = 0>
cudaError_t launch_t(const LayerDev& L, const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<KB, VB, VG, NT, OUTL>;
  const size_t sm = C::smem_bytes(OUTL ? L.outliers : 0, NT == 1 && a.gqa == 1);
  auto kern = decode_tc_kernel<KB, VB, VG, NT, OUTL, GF>;
  static SmemAttr attr;
  {  // room for the most outliers a row may hold
    const cudaError_t e = attr.ensure(kern, C::smem_bytes(OUTL ? kMaxOutliers : 0));
    if (e != cudaSuccess) return e;
  }
  if (a.occupancy_out) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(a.occupancy_out, kern, kThreads, sm);
  dim3 grid(a.splits, L.n_streams);
  kern<<<grid, kThreads, sm, st>>>(L, a);
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace kvq
