// common.cuh -- shared device helpers for the streaming log-domain Sinkhorn kernels.
//
// All kernels work in base 2: for an F-type pass (rows = X, columns = Y) the score is
//   s2_ij = kappa * <x_i, y_j> + c_j,   kappa = 2 log2(e) / eps,
//   c_j   = (g_j - |y_j|^2) log2(e) / eps + log2 b_j,
// so that f_i = |x_i|^2 - eps ln2 * LSE2_j(s2_ij) (FlashSinkhorn: IO-Aware Entropic
// Optimal Transport on GPU, SAI replication review, "Summary": the Sinkhorn update as a
// row-wise log-sum-exp of biased dot-product scores). A G-type pass swaps the roles of
// X and Y. Padded columns carry c_j = -inf and contribute exactly zero.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace flashot {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
// Finite floor for running maxima: exp2(x - kNegBig) never produces NaN from -inf - -inf.
constexpr float kNegBig = -1.0e30f;

// SFU base-2 exponential (MUFU.EX2), flush-to-zero; exp2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Programmatic dependent launch (sm_90+). A kernel launched with the programmatic
// stream-serialization attribute may start before the kernel ahead of it in the stream has
// finished; griddep_wait() blocks the calling thread until that kernel (and so every
// earlier one) has completed and its writes are visible. griddep_launch_dependents() lets
// the next such kernel start early. Both are no-ops for a kernel launched normally.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// What a weighted-sum pass produces: transport application P V, the barycentric gradient,
// the Hadamard-weighted transport (P .* X Y^T) 1, or the Hadamard-weighted transport
// matrix application (P .* U Q^T) Q (weights P_ij <u_i, q_j> applied to the column points;
// the curvature term of the Hessian-vector product).
enum WsumMode : int { kWsumApply = 0, kWsumGrad = 1, kWsumHadamard = 2, kWsumHessT = 3 };

// Status bits written into the workspace status word by kernels that give up a wait.
constexpr unsigned kErrTimeout = 1u;

// Stream-K split of T tiles over G persistent CTAs: CTA c owns tiles [c*T/G, (c+1)*T/G).
__host__ __device__ __forceinline__ int64_t sk_begin(int64_t c, int64_t T, int64_t G) {
  return c * T / G;
}
// The CTA whose range contains tile v (largest c with sk_begin(c) <= v).
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t v, int64_t T, int64_t G) {
  return ((v + 1) * G + T - 1) / T - 1;
}

// How the partials of one LSE pass are laid out: either n_splits fixed splits per row, or
// (n_splits == 0) stream-K over T = row_tiles * NT tiles (row tiles of unit_rows rows: 128
// for single CTAs, 256 for CTA pairs) with G owners (CTAs or CTA pairs), where the row
// tile rt has slots_per_owner * (owner((rt+1)NT-1) - owner(rt NT) + 1) slots.
struct SplitInfo {
  int n_splits;
  int slots_per_owner;  // stream-K: partial slots each owner writes per row tile
  int64_t sk_T, sk_G, sk_NT;
  int unit_rows;        // stream-K: rows per row tile
};

}  // namespace flashot
