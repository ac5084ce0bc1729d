// sa_tma.h — host-side construction of TMA tensor maps (cuTensorMapEncodeTiled
// through the runtime's driver entry point; no link against libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <stdint.h>

namespace sa {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A bf16 matrix of `rows` rows x `d` elements (row stride d*2 bytes) seen as
// boxes of 64 elements (128 bytes) x box_rows rows, 128-byte swizzled in
// shared memory.  Out-of-range rows read as zeros.  box_rows = 1 is the form
// the 4-row gather (tile::gather4) requires.
inline bool make_rows_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t d,
                          uint32_t box_rows) {
  const EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {d, rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Every `stride`-th key row of each of BH heads of a [BH, Nk, d] bf16 tensor:
// row i of head h is key i*stride (i < nkeys), seen as boxes of 64 elements x
// 128 rows of one head, 128-byte swizzled.  Rows past nkeys read as zeros.
inline bool make_keys_map(CUtensorMap* map, const void* base, uint32_t d, uint64_t nkeys,
                          uint64_t Nk, uint64_t BH, uint64_t stride) {
  const EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d, nkeys, BH};
  const cuuint64_t strides[2] = {stride * d * 2, Nk * d * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The fp32 score matrix of B*H heads x G rows x Nk keys (row stride ld
// floats, head stride G*ld floats) seen as boxes of 32 keys x 128 rows of one
// head, unswizzled.  Stores clip at Nk, at G (never into the next head) and
// at the last head.
inline bool make_scores_map(CUtensorMap* map, void* base, uint32_t Nk, uint64_t G, uint64_t BH,
                            uint64_t ld) {
  const EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {Nk, G, BH};
  const cuuint64_t strides[2] = {ld * 4, G * ld * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sa
