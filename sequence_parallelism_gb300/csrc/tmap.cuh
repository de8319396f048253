// tmap.cuh -- TMA tensor maps over [B][S][H][128] bf16 tensors, viewed
// blockwise for the ring schedule.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "sp_gb300.h"

namespace sp {
namespace tmap {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// [B][S][H][128] bf16 viewed as 5-D (d, H, rows-in-block, block, B) for the
// contiguous order or (d, H, block, rows-in-block, B) for the striped order,
// box = 64 columns x 1 head x box_rows rows, 128-byte swizzle.  Rows past the
// end of a block are out of bounds and read as zeros.
inline bool make_map(CUtensorMap* m, const void* base, int B, int S, int H, int P, int order,
                     int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t Lb = static_cast<cuuint64_t>(S / P);
  const cuuint64_t row = static_cast<cuuint64_t>(H) * 128 * 2;  // bytes per token
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], estr[5] = {1, 1, 1, 1, 1};
  dims[0] = 128;
  dims[1] = H;
  dims[4] = B;
  strides[0] = 128 * 2;
  strides[3] = static_cast<cuuint64_t>(S) * row;
  box[0] = 64;
  box[1] = 1;
  box[4] = 1;
  if (order == SP_ORDER_STRIPED) {
    dims[2] = P;
    dims[3] = Lb;
    strides[1] = row;
    strides[2] = row * P;
    box[2] = 1;
    box[3] = static_cast<cuuint32_t>(box_rows);
  } else {
    dims[2] = Lb;
    dims[3] = P;
    strides[1] = row;
    strides[2] = row * Lb;
    box[2] = static_cast<cuuint32_t>(box_rows);
    box[3] = 1;
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tmap
}  // namespace sp
