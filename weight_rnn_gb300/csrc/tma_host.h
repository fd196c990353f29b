// tma_host.h -- host-side creation of TMA tensor maps.  The driver entry
// point cuTensorMapEncodeTiled is looked up through the runtime at first use,
// so the library needs no link-time dependency on libcuda.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace delta {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A 4-D bf16 tensor [d3][d2][d1][d0] (d0 innermost, contiguous) tiled with a
// box {b0, b1, b2, b3}.  swizzle128: 128-byte swizzle (b0 * 2 must be <= 128).
inline cudaError_t make_map_4d_bf16(CUtensorMap *map, const void *base, uint64_t d0,
                                    uint64_t d1, uint64_t d2, uint64_t d3, uint32_t b0,
                                    uint32_t b1, uint32_t b2, uint32_t b3, bool swizzle128) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};  // bytes, dims 1..3
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                   strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A 3-D bf16 tensor [d2][d1][d0] (d0 innermost, contiguous) tiled with a
// box {b0, b1, b2} and the 128-byte swizzle (b0 * 2 must be <= 128).
inline cudaError_t make_map_3d_bf16_sw128(CUtensorMap *map, const void *base, uint64_t d0,
                                          uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
                                          uint32_t b2) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};  // bytes, dims 1..2
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                   strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace delta
