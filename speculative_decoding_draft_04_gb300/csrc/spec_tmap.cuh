// Host-side encoding of the TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry point: the library links no driver
// library of its own).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "spec_internal.cuh"

namespace spec {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// U as [B][gamma][V] bf16, boxes of 64 columns x 1 step x 128 requests,
// 128-byte swizzle; reads outside the tensor return zeros.
inline cudaError_t encode_u_map(const Shape& sh, const void* U, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t V = (cuuint64_t)sh.V;
  const cuuint64_t dims[3] = {V, (cuuint64_t)sh.gamma, (cuuint64_t)sh.B};
  const cuuint64_t strides[2] = {V * 2, V * 2 * (cuuint64_t)sh.gamma};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// U as [B][gamma][V] bf16 in chunks of 32 columns: boxes of 32 columns x 1
// step x 128 requests, 64-byte swizzle (one 8 KB chunk of a 128-request
// tile); reads outside the tensor return zeros.
inline cudaError_t encode_u_chunk_map(const Shape& sh, const void* U, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t V = (cuuint64_t)sh.V;
  const cuuint64_t dims[3] = {V, (cuuint64_t)sh.gamma, (cuuint64_t)sh.B};
  const cuuint64_t strides[2] = {V * 2, V * 2 * (cuuint64_t)sh.gamma};
  const cuuint32_t box[3] = {32, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// The draft's A-row buffer as [rows][r] bf16, boxes of 64 columns x 128 rows
// (one K atom of the A operand), 128-byte swizzle; rows beyond `rows` read as
// zeros.
inline cudaError_t encode_abuf_map(int rows, int r, const void* abuf, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)r * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(abuf), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// W2 as [r][V] bf16, boxes of 64 columns x r rows (one MN-major operand
// atom), 128-byte swizzle; reads outside the tensor return zeros.
inline cudaError_t encode_w2_map(const Shape& sh, const void* W2, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)sh.V, (cuuint64_t)sh.r};
  const cuuint64_t strides[1] = {(cuuint64_t)sh.V * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)sh.r};
  const cuuint32_t es[2] = {1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

}  // namespace spec
