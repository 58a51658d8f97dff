// Host-side TMA descriptor encoding (cuTensorMapEncodeTiled reached through
// the runtime's driver entry point, so the library needs no link-time libcuda).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

namespace mla {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
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

// 2-D row-major tensor [rows, cols] of `elem_bytes`-byte elements with a row
// pitch of `row_stride_bytes`; boxes of box_rows x box_cols; out-of-bounds
// elements read as zero.  Returns false if the CUDA driver rejects the layout.
inline bool encode_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols,
                           uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                           CUtensorMapSwizzle swizzle) {
  auto fn = tmap_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D tensor [d2][d1][d0] (d0 contiguous) with byte strides s1 (between
// consecutive d1 indices) and s2 (between consecutive d2 indices); boxes of
// box0 x box1 x box2; out-of-bounds elements read as zero.
inline bool encode_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1,
                           uint64_t d2, uint64_t s1, uint64_t s2, uint32_t box0, uint32_t box1, uint32_t box2,
                           CUtensorMapSwizzle swizzle) {
  auto fn = tmap_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mla
