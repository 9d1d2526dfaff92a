// tc_wsum_pair.h -- host entry points of the CTA-pair weighted-sum pass (tc_wsum_pair.cu),
// used by flashot.cu. All pointers are device pointers inside the caller's workspace or the
// caller's own buffers; every function only enqueues work on `st`.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace flashot {

// Weighted-sum pass on CTA pairs: bf16, tf32 or split tf32 (prec is the FLASHOT_PREC_*
// value), 256-row x 256-column units, W kept in tensor memory as the A operand of the
// second contraction. rows_pad must be a multiple of 256. vtq holds
// tc_wsum_pair_vt_bytes(prec, cols_pad, max(k, d)) bytes for the V^T planes, scratch
// tc_wsum_pair_scratch_bytes(rows_pad, max(k, d)) bytes for the partial sums.
size_t tc_wsum_pair_scratch_bytes(int64_t rows_pad, int64_t k_or_d);
size_t tc_wsum_pair_vt_bytes(int prec, int64_t rows_pad, int64_t k_or_d);
// Whether enough 2-CTA clusters of the pass fit on this device (queried once).
bool tc_wsum_pair_available(int sms);
int tc_wsum_pair_pass(int prec, int mode, const void* rowQ, const void* colQ,
                      const float* colBias, const float* rowBias, int64_t n_rows, int64_t n_cols,
                      int64_t rows_pad, int64_t cols_pad, int64_t d, int64_t dpt, float kappa,
                      const float* V, int64_t ldv, int64_t k, void* vtq, void* scratch,
                      const float* rowW, const float* X, float* out, int64_t ldo, int sms,
                      unsigned* status, cudaStream_t st);

}  // namespace flashot
