// Host-side encoding of TMA tensor maps through the driver entry point, so the
// library links only the CUDA runtime (no -lcuda at build time).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

namespace fa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      return nullptr;
    }
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A bf16 tensor viewed as [planes][rows][cols] (cols contiguous), copied in
// boxes of box_cols x box_rows x 1 with 128-byte swizzling.  Rows and planes
// outside the tensor read as zero and are not written by stores, so a ragged
// last tile never touches the next plane.  Returns false on an encoding error.
inline bool encode_bf16_3d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                           uint64_t planes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};  // bytes, for dims 1 and 2
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A one-byte tensor (the FP8 path's e4m3 codes) viewed as
// [planes][rows][cols] (cols contiguous), in boxes of box_cols x box_rows x 1
// with 128-byte swizzling; rows outside the tensor read as zero.
inline bool encode_u8_3d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                         uint64_t planes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols, cols * rows};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An fp32 tensor viewed as [planes][rows][cols] (cols contiguous), in boxes
// of box_cols x box_rows x 1 without swizzling (the box is plain row-major in
// shared memory).  Used for reductions into it: elements outside the tensor
// are skipped.  Returns false on an encoding error.
inline bool encode_f32_3d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                          uint64_t planes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 4, cols * rows * 4};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa
