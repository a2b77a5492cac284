// Host-side creation of TMA tensor maps (2-D, 128-byte swizzle).  The driver
// entry point is looked up through the runtime, so libdsa.so does not link
// against libcuda directly and loads on machines without a driver.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Row-major [rows, row_bytes] byte-addressed matrix (uint8 elements), tiles of
// box_rows x 128 bytes with the 128-byte swizzle.  Out-of-range rows read as
// zero.  Returns false when the driver rejects the map (e.g. misalignment).
inline bool make_tmap_rows128(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes,
                              uint32_t box_rows, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const uint32_t esize = dt == CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 ? 2u : 1u;
  cuuint64_t dims[2] = {row_bytes / esize, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128u / esize, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major bf16 matrix [rows, cols]; boxes of box_rows x box_cols elements
// (box_cols * 2 bytes = 128 with the 128-byte swizzle, 64 with the 64-byte one).
inline bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                           uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dsa
