// Tensor maps of the packed code arrays and the tiled TMA copy of a box of
// whole code rows (uint8 tensor [stream][row][byte]) into shared memory with
// the bank swizzle of the row width, shared by the decode kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace kvq {

// Byte offset of a (row, byte) position inside a tile copied with the 64- or
// 128-byte bank swizzle (16-byte chunk index XOR address bits 7..9).
template <int RB>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  return off ^ (((off >> 7) & (RB == 128 ? 7u : 3u)) << 4);
}

// 3-D tensor copy (byte 0, row, stream) of a box of code rows into shared memory.
__device__ __forceinline__ void tma_rows(void* dst, const CUtensorMap* map, int row, int stream,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(stream), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// cuTensorMapEncodeTiled from the driver, looked up once.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Code rows of one tensor as a uint8 tensor [stream][row][byte]; a box is
// `box_rows` whole rows, written to shared memory with the bank swizzle of the
// row width (64 or 128 bytes).
inline cudaError_t encode_rows(CUtensorMap* m, const void* base, int row_bytes, int cap, int n_streams,
                               int64_t stream_bytes, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)cap, (cuuint64_t)n_streams};
  const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)stream_bytes};
  const cuuint32_t box[3] = {(cuuint32_t)row_bytes, (cuuint32_t)box_rows, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  const CUtensorMapSwizzle sw = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace kvq
