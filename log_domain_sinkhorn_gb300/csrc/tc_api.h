// tc_api.h -- host entry points of the tcgen05 (tensor-core) streaming passes, used by
// flashot.cu. All pointers are device pointers inside the caller's workspace or the
// caller's own buffers; every function only enqueues work on `st`.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace flashot {

// Launch the bounded-wait self-test kernel (see flashot_selftest_bounded_wait).
int tc_selftest_bounded_wait(unsigned* status, int64_t limit_ns, cudaStream_t st);

// Pack X (n x d) and Y (m x d) fp32 into row-padded, K-padded operand copies for the
// tensor cores: bf16 (round to nearest even) or tf32-rounded fp32.
// mode: 0 = tf32, 1 = bf16, 2 = split tf32 (X = [hi|hi|lo], Y = [hi|lo|hi], three segments of
// d elements back to back, padded to dpt).
int tc_pack_inputs(int mode, const float* X, const float* Y, int64_t n, int64_t m, int64_t d,
                   int64_t n_pad, int64_t m_pad, int64_t dpt, void* xq, void* yq, int sms,
                   cudaStream_t st);

// Row-wise base-2 LSE of s2_ij = kappa <p_i, q_j> + colBias_j over all columns, as
// (max, sum) partials: partial[slot * rows_pad + i], slots described by *info (stream-K).
int tc_lse_pass(bool bf16, const void* rowQ, const void* colQ, const float* colBias,
                int64_t n_rows, int64_t rows_pad, int64_t cols_pad, int64_t dpt, float kappa,
                float2* partial, int max_splits, int sms, unsigned* status, SplitInfo* info,
                cudaStream_t st);

// Weighted sums with w_ij = exp2(kappa <p_i, q_j> + colBias_j + rowBias_i); mode as in
// fma_kernels.cuh (apply / grad / Hadamard). V (n_cols x k, fp32, row stride ldv) is the
// right operand of the second contraction (the column points themselves for the
// gradient); it is transposed and packed into vtq first. X is the row points (fp32) for
// the gradient's epilogue. When one CTA per (row tile, output group) would leave a wave
// mostly empty, the column tiles are split over up to 8 CTAs whose raw sums go to split_buf
// and are added in a fixed order by a second kernel.
int tc_wsum_pass(bool bf16, int mode, const void* rowQ, const void* colQ, const float* colBias,
                 const float* rowBias, int64_t n_rows, int64_t n_cols, int64_t rows_pad,
                 int64_t cols_pad, int64_t d, int64_t dpt, float kappa, const float* V,
                 int64_t ldv, int64_t k, void* vtq, const float* rowW, const float* X,
                 float* out, int64_t ldo, int sms, unsigned* status, cudaStream_t st,
                 void* split_buf, size_t split_bytes);
// Partial-sum buffer of tc_wsum_pass's column splits (tf32): enough for up to 8 splits of
// rows_pad rows with max(k, d) output columns, capped at 64 MB; fewer splits run when the
// buffer holds fewer.
size_t tc_wsum_split_bytes(int64_t rows_pad, int64_t k_or_d);

// bf16 weighted-sum pass on 128 x 256 tiles with stream-K partials (tc_wsum2.cu). scratch
// holds tc_wsum2_scratch_bytes(rows_pad, max(k, d)) bytes for the partial sums.
size_t tc_wsum2_scratch_bytes(int64_t rows_pad, int64_t k_or_d);
int tc_wsum2_pass(int mode, const void* rowQ, const void* colQ, const float* colBias,
                  const float* rowBias, int64_t n_rows, int64_t n_cols, int64_t rows_pad,
                  int64_t cols_pad, int64_t d, int64_t dpt, float kappa, const float* V,
                  int64_t ldv, int64_t k, void* vtq, void* scratch, const float* rowW,
                  const float* X, float* out, int64_t ldo, int sms, unsigned* status,
                  cudaStream_t st);

}  // namespace flashot
