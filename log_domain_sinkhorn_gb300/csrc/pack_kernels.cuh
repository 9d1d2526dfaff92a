// pack_kernels.cuh -- packing of the fp32 point clouds into padded operand copies
// (fp32 for the CUDA-core path, tf32-rounded fp32 or bf16 for the tensor-core path).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace flashot {

// Output element type of the packer.
enum class PackKind : int { F32 = 0, TF32 = 1, BF16 = 2 };

__device__ __forceinline__ uint32_t tf32_rna(float v) {
  uint32_t t;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(v));
  return t;
}

// Split-tf32 packing: row r of dst (ld elements) holds three segments of d columns each,
// back to back; segment k holds part[k] of every coordinate, where part 0 = hi = tf32(x),
// part 1 = lo = tf32(x - hi). pattern encodes the three parts (bits 0, 1, 2): 0b100 =
// [hi|hi|lo], 0b010 = [hi|lo|hi]. Zero padding from column 3d to ld and in rows >= rows.
static __global__ void pack_rows_tf32x3_kernel(const float* __restrict__ src, uint32_t* __restrict__ dst,
                                        int64_t rows, int64_t d, int64_t rows_pad, int64_t ld,
                                        int pattern) {
  const int64_t total = rows_pad * ld;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / ld;
    const int64_t cc = e - r * ld;
    if (cc >= 3 * d) {
      dst[e] = 0u;
      continue;
    }
    const int part = (int)(cc / d);
    const int64_t c = cc - part * d;
    const float v = r < rows ? src[r * d + c] : 0.0f;
    const uint32_t hi = tf32_rna(v);
    const uint32_t lo = tf32_rna(v - __uint_as_float(hi));
    dst[e] = ((pattern >> part) & 1) ? lo : hi;
  }
}

// dst (rows_pad x d_pad, row-major) = src (rows x d) zero-padded; TF32 rounds to nearest
// (cvt.rna.tf32.f32), BF16 rounds to nearest even. One thread per destination element.
template <PackKind K>
__global__ void pack_rows_kernel(const float* __restrict__ src, void* __restrict__ dst,
                                 int64_t rows, int64_t d, int64_t rows_pad, int64_t d_pad) {
  const int64_t total = rows_pad * d_pad;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / d_pad;
    const int64_t c = e - r * d_pad;
    const float v = (r < rows && c < d) ? src[r * d + c] : 0.0f;
    if constexpr (K == PackKind::BF16) {
      static_cast<__nv_bfloat16*>(dst)[e] = __float2bfloat16_rn(v);
    } else if constexpr (K == PackKind::TF32) {
      uint32_t t;
      asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(v));
      static_cast<uint32_t*>(dst)[e] = t;
    } else {
      static_cast<float*>(dst)[e] = v;
    }
  }
}

// dst (cols_pad x rows_pad, row-major) = transpose of src (rows x cols, row-major), zero
// padded; rounding as above. 32 x 32 tiles through shared memory so both the reads and the
// writes are coalesced. Block (32, 8); grid (rows_pad / 32, cols_pad / 32).
template <PackKind K>
__global__ void pack_transpose_kernel(const float* __restrict__ src, void* __restrict__ dst,
                                      int64_t rows, int64_t cols, int64_t rows_pad,
                                      int64_t cols_pad) {
  __shared__ float tile[32][33];
  const int64_t r0 = (int64_t)blockIdx.x * 32, c0 = (int64_t)blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < rows && c < cols) ? src[r * cols + c] : 0.0f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;  // dst row c, dst column r
    if (c >= cols_pad || r >= rows_pad) continue;
    const float v = tile[threadIdx.x][i];
    const int64_t e = c * rows_pad + r;
    if constexpr (K == PackKind::BF16) {
      static_cast<__nv_bfloat16*>(dst)[e] = __float2bfloat16_rn(v);
    } else if constexpr (K == PackKind::TF32) {
      uint32_t t;
      asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(v));
      static_cast<uint32_t*>(dst)[e] = t;
    } else {
      static_cast<float*>(dst)[e] = v;
    }
  }
}

}  // namespace flashot
