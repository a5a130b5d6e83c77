// Host-side TMA tensor-map encoding (driver API reached through the runtime's entry-point
// query, so the library needs no link-time libcuda).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace fa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// [heads x N x cols] bf16 (contiguous), loaded as boxes of 64 columns x box_rows rows of
// one head with the 128-byte swizzle. Rows past N inside a head read as zeros, so a tile
// that straddles the end of a head never picks up the next head's rows.
inline bool make_map_bf16_3d(CUtensorMap* map, const void* base, int64_t heads, int64_t N, int64_t cols,
                             int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)N * cols * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [heads x N x cols] bytes (8-bit elements, e.g. e4m3), loaded as boxes of 128 columns x
// box_rows rows of one head with the 128-byte swizzle; rows past N read as zeros.
inline bool make_map_u8_3d(CUtensorMap* map, const void* base, int64_t heads, int64_t N, int64_t cols,
                           int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)N * cols};
  cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fa
