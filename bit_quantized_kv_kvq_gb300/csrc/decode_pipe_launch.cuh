// Host side of the stream-K decode kernel (decode_pipe.cuh): work partition,
// shared-memory plan, tensor maps of the code arrays, launch. The including
// translation unit picks the key/value code widths with KVQ_PIPE_KB and
// KVQ_PIPE_VB.
#pragma once

#include <cstring>

#include "decode_pipe.cuh"

namespace kvq {
namespace pipe {

inline int round_up_i(int x, int m) { return (x + m - 1) / m * m; }

constexpr int kSmemMax = 232448;  // dynamic shared memory per CTA on sm_103a (227 KB)

template <int KB, int VB, int VG, bool OUTL>
struct Plan {
  static constexpr int KROW = 4 * Pack<KB>::kWords, VROW = 4 * Pack<VB>::kWords;
  static constexpr int VGPR = kHeadDim / VG;
  static constexpr int UT = 64;  // tokens per unit: two subtiles of 32 per wait and refill

  // Fills the shared-memory layout of `a` (H, kout, T set) and returns the
  // dynamic shared memory the launch needs, or 0 if it does not fit.
  static int layout(Args& a) {
    a.UT = UT;
    a.U = a.T / UT;
    const int H = a.H, kout = OUTL ? a.kout : 0;
    a.kc_bytes = UT * KROW;
    a.vc_bytes = UT * VROW;
    a.vm_bytes = UT * VGPR * 4;
    const bool swz = KB != 3 || VB != 3;
    a.off_vc = round_up_i(a.kc_bytes, VB != 3 ? 1024 : 128);
    a.off_km = round_up_i(a.off_vc + a.vc_bytes, 128);
    a.off_vm = a.off_km + kHeadDim * 4;
    a.off_out = round_up_i(a.off_vm + a.vm_bytes, 128);
    a.stage_bytes = round_up_i(a.off_out + (OUTL ? 4 * UT * kout * 2 : 0), swz ? 1024 : 128);
    a.w_qn = 0;
    a.w_frag = round_up_i(H * kHeadDim * 4, 16);
    // fragment rows of heads < H; with outliers and several heads the area
    // also holds a [32 tokens][8 heads] float exchange
    const int frag_bytes = 4 * H * kFragRow * 16;
    a.w_eq = a.w_frag + (OUTL && H > 1 && frag_bytes < 32 * kHMax * 4 ? 32 * kHMax * 4 : frag_bytes);
    a.w_kz = a.w_eq + 32;
    a.w_ocr = a.w_kz + (OUTL ? kHeadDim * 4 : 0);
    a.warp_bytes = round_up_i(a.w_ocr + (OUTL ? H * kHeadDim * 4 : 0), 128);
    a.slot_bytes = round_up_i((H * kHeadDim + 2 * kHMax) * 4, 128);
    const int fixed = 1024 /* base alignment */ + kCons * a.warp_bytes + 2 * a.slot_bytes + 128;
    int ns = (kSmemMax - fixed) / (a.stage_bytes + 16);  // + barrier and last-issue word per stage
    if (ns > 64) ns = 64;
    ns -= ns % a.U;  // a stage's next unit is then a whole number of key blocks ahead
    if (ns < a.U) return 0;  // at least one key block of stages (warps then take turns)
    a.ns = ns;
    a.ring_bytes = ns * a.stage_bytes;
    return fixed + a.ring_bytes + 16 * ns;
  }
};

template <int KB, int VB, int VG, bool OUTL>
cudaError_t launch_t(const LayerDev& L, Args a, cudaStream_t st) {
  using PL = Plan<KB, VB, VG, OUTL>;
  const int smem = PL::layout(a);
  if (smem == 0) return cudaErrorInvalidConfiguration;
  Maps maps;
  std::memset(&maps, 0, sizeof maps);
  if (KB != 3) {
    cudaError_t e = encode_rows(&maps.k, L.k.codes, PL::KROW, L.capacity, L.n_streams,
                                L.k.codes_sstride * 4, PL::UT);
    if (e != cudaSuccess) return e;
  }
  if (VB != 3) {
    cudaError_t e = encode_rows(&maps.v, L.v.codes, PL::VROW, L.capacity, L.n_streams,
                                L.v.codes_sstride * 4, PL::UT);
    if (e != cudaSuccess) return e;
  }
  auto kern = decode_pipe_kernel<KB, VB, VG, OUTL>;
  static SmemAttr attr;
  {
    const cudaError_t e = attr.ensure(kern, kSmemMax);
    if (e != cudaSuccess) return e;
  }
  kern<<<a.P, kThreads, smem, st>>>(maps, L, a);
  return cudaGetLastError();
}

}  // namespace pipe

#define KVQ_PIPE_NAME3(a, b, c) a##b##c
#define KVQ_PIPE_NAME(b, c) KVQ_PIPE_NAME3(launch_decode_pipe_k, b, c)

cudaError_t KVQ_PIPE_NAME(KVQ_PIPE_KB, KVQ_PIPE_VB)(const LayerDev& L, const pipe::Args& a, cudaStream_t st) {
  constexpr int KB = KVQ_PIPE_KB, VB = KVQ_PIPE_VB;
  const bool outl = L.outliers > 0;
  if (VB == 3 || L.v.group == 128)
    return outl ? pipe::launch_t<KB, VB, 128, true>(L, a, st) : pipe::launch_t<KB, VB, 128, false>(L, a, st);
  if constexpr (VB != 3)
    return outl ? pipe::launch_t<KB, VB, 64, true>(L, a, st) : pipe::launch_t<KB, VB, 64, false>(L, a, st);
  return cudaErrorNotSupported;
}

}  // namespace kvq
