// tc_host.h -- host-side helpers shared by the tensor-core translation units: TMA
// tensor-map encoding (driver entry point fetched through the runtime, so no -lcuda),
// dynamic shared-memory opt-in and the stream-K grid choice.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "flashot.h"

namespace flashot {
namespace tc {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over a packed operand (rows x cols elements, row-major), box = box_rows x 128 B,
// 128-byte swizzle (the layout the UMMA K-major SW128 descriptor expects).
inline int make_map_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, bool bf16,
                         int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return FLASHOT_ERR_CUDA;
  const int es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * es)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FLASHOT_OK : FLASHOT_ERR_INVALID_ARG;
}

inline int make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, bool bf16) {
  return make_map_rows(m, base, rows, cols, bf16, 128);
}

template <typename K>
int set_smem(K kernel, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

// Number of persistent CTAs: at most one per SM, at most one per tile, and few enough that
// no row tile is split over more than max_owners CTAs.
inline int64_t choose_grid(int64_t row_tiles, int64_t NT, int sms, int max_owners) {
  const int64_t T = row_tiles * NT;
  int64_t G = std::min<int64_t>(sms, T);
  while (G > 1) {
    int64_t worst = 0;
    for (int64_t rt = 0; rt < row_tiles; ++rt) {
      const int64_t s = sk_owner((rt + 1) * NT - 1, T, G) - sk_owner(rt * NT, T, G) + 1;
      worst = std::max(worst, s);
    }
    if (worst <= max_owners) break;
    --G;
  }
  return std::max<int64_t>(G, 1);
}

}  // namespace tc
}  // namespace flashot
