// Host-side TMA tensor-map encoding for 2D bf16 tensors.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "status.cuh"

namespace dsa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A row-major [rows, cols] tensor of 2-byte (bf16) or 1-byte (FP8 codes) elements with the
// given row pitch. Box = box_cols x box_rows elements; swizzle one of
// CU_TENSOR_MAP_SWIZZLE_{NONE,64B,128B}. Out-of-range elements read 0.
inline int make_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                        uint64_t rows, uint64_t cols, uint64_t row_pitch_bytes, uint32_t box_cols,
                        uint32_t box_rows, CUtensorMapSwizzle swizzle);

inline int make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                             uint64_t row_pitch_bytes, uint32_t box_cols, uint32_t box_rows,
                             CUtensorMapSwizzle swizzle) {
  return make_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rows, cols, row_pitch_bytes,
                      box_cols, box_rows, swizzle);
}

inline int make_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                        uint64_t rows, uint64_t cols, uint64_t row_pitch_bytes, uint32_t box_cols,
                        uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || row_pitch_bytes % 16 != 0)
    return fail(DSA_ERR_INVALID, "tensor base must be 16-byte aligned and rows 16-byte multiples");
  const cuuint64_t dims[2] = {cols, rows == 0 ? 1 : rows};
  const cuuint64_t strides[1] = {row_pitch_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, dtype, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): rows=%llu cols=%llu box=%ux%u",
                static_cast<int>(r), static_cast<unsigned long long>(rows),
                static_cast<unsigned long long>(cols), box_cols, box_rows);
  return DSA_OK;
}

int num_sms_cached();

}  // namespace dsa
