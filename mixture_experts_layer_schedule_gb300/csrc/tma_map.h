// tma_map.h -- host-side construction of 2-D TMA tensor maps (driver entry
// point looked up once through the runtime, no libcuda link).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace moe {

typedef CUresult (*EncodeTiledFnT)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFnT tma_encode_fn() {
  static EncodeTiledFnT fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnT>(p);
  });
  return fn;
}

// 2-D view [outer][inner] (inner contiguous) of `elem`-byte elements, box
// box_inner x box_outer, 128-byte swizzle unless told otherwise. false if the
// view or box is not encodable (base 16-byte aligned, row pitch a multiple of
// 16 bytes, box row at most 128 bytes).
inline bool tma_map_2d(CUtensorMap* m, const void* base, int64_t inner, int64_t outer,
                       int box_outer, int box_inner, CUtensorMapDataType dtype, int elem,
                       CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFnT fn = tma_encode_fn();
  if (!fn || outer <= 0 || inner <= 0 || box_outer <= 0 || box_outer > 256) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (inner * elem) % 16 != 0) return false;
  if (box_inner * elem > 128 || (box_inner * elem) % 16 != 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * elem)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner),
                             static_cast<cuuint32_t>(box_outer)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe
