// Host-side construction of TMA tensor maps (cuTensorMapEncodeTiled, fetched from the driver at
// run time so the library loads on machines without a GPU driver).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace dit {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn();  // null when the driver entry point is unavailable

// 2-D map over a row-major matrix: `inner` elements per row (contiguous), `outer` rows,
// `row_bytes` between rows; box = box_inner x box_outer elements. Out-of-range box elements
// read as zero. swizzle128: 128-byte swizzle (box_inner * elem_bytes must be 128).
inline bool make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, long long inner,
                         long long outer, long long row_bytes, int box_inner, int box_outer, bool swizzle128) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  (void)elem_bytes;
  cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
  cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map (bf16, 128-byte swizzle): dims {d0 (contiguous), d1, d2}, strides in bytes of d1 and d2.
inline bool make_tmap_3d_bf16(CUtensorMap* m, const void* base, long long d0, long long d1, long long d2,
                              long long stride1_bytes, long long stride2_bytes, int box0, int box1) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cuuint64_t(d0), cuuint64_t(d1), cuuint64_t(d2)};
  cuuint64_t strides[2] = {cuuint64_t(stride1_bytes), cuuint64_t(stride2_bytes)};
  cuuint32_t box[3] = {cuuint32_t(box0), cuuint32_t(box1), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dit
