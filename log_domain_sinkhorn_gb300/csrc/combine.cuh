// combine.cuh -- the end of a log-sum-exp half-step: merge the per-split (max, sum)
// partials of the base-2 LSE of one row and write the new potential and the next pass's
// bias (lse_combine_kernel, one thread per row).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace flashot {

// What a half-step writes besides the partials it reads (pointers may be NULL):
//   L_i  = M + log2 S,   pot_i = norm_i - eps ln2 L_i   (averaged with the previous out_pot
//   when `average` is set: the symmetric schedule),
//   next_bias_i = lw2_i - L_i * (eps / eps_next)   (= (pot_i - norm_i) log2e/eps_next + lw2_i)
// next_bias is the bias the following pass (the other side's update at eps_next) needs;
// its padding entries [rows, rows_pad) are set to -inf so padded points carry no mass.
// err_rows != NULL (the convergence check): before out_pot is overwritten, the row's share
// of the L1 marginal error of the previous iterate,
//   err_rows_i = w_i |exp((old_i - new_i) / eps) - 1|  (= |sum_j P_ij(old) - w_i|),
// is written, with 0 for padding rows.
struct CombineArgs {
  int64_t rows, rows_pad;
  const float* norms;
  float eps;
  const float* lw2;
  float eps_ratio;
  float* out_pot;
  float* next_bias;
  float* out_lse2;
  int average;
  const float* err_w;
  float* err_rows;
};

// Number of partial slots of row i.
__device__ __forceinline__ int combine_slots(const SplitInfo& split, int64_t i) {
  if (split.n_splits != 0) return split.n_splits;
  const int64_t rt = i / split.unit_rows;
  return split.slots_per_owner *
         (int)(sk_owner((rt + 1) * split.sk_NT - 1, split.sk_T, split.sk_G) -
               sk_owner(rt * split.sk_NT, split.sk_T, split.sk_G) + 1);
}

// Row i (0 <= i < rows_pad). kL2: read the partials from L2 (ld.global.cg), for a caller
// inside the kernel whose other CTAs wrote them (a stale L1 line must not be read).
template <bool kL2 = false>
__device__ __forceinline__ void combine_row(const float2* __restrict__ partial, int64_t ld,
                                            const SplitInfo& split, int64_t i,
                                            const CombineArgs& a) {
  if (i >= a.rows) {
    if (i < a.rows_pad && a.next_bias) a.next_bias[i] = neg_inf();
    if (i < a.rows_pad && a.err_rows) a.err_rows[i] = 0.0f;
    return;
  }
  const int n_splits = combine_slots(split, i);
  auto load = [&](int s) { return kL2 ? __ldcg(partial + s * ld + i) : partial[s * ld + i]; };
  float M = kNegBig;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, load(s).x);
  float S = 0.0f;
  for (int s = 0; s < n_splits; ++s) {
    const float2 p = load(s);
    S += p.y * ex2(p.x - M);
  }
  const float L = M + log2f(S);  // S == 0 (no mass) gives -inf, so pot = +inf
  const float fresh = a.norms[i] - a.eps * kLn2 * L;
  // Symmetric schedule: the new potential is the mean of the previous one and the update.
  const float pot = a.average ? 0.5f * (a.out_pot[i] + fresh) : fresh;
  if (a.err_rows) {
    const float w = a.err_w[i];
    a.err_rows[i] = w > 0.0f ? w * fabsf(expm1f((a.out_pot[i] - fresh) / a.eps)) : 0.0f;
  }
  if (a.out_pot) a.out_pot[i] = pot;
  if (a.next_bias) a.next_bias[i] = a.lw2[i] - L * a.eps_ratio;
  if (a.out_lse2) a.out_lse2[i] = L;
}

}  // namespace flashot
