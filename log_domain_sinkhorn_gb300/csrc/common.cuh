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

// The row-tile segments of a stream-K range [tb, te) of row-tile-major units (NT units per
// row tile), in the order the CTA-pair passes walk them: the last segment (the head of the
// last row tile, columns from 0) first, then the others in order. Every owner's range then
// starts at column 0 and, after its first segment, runs about T/G mod NT columns behind,
// so the owners sweep the column tiles nearly in step: each column tile is read by all of
// them within a short window, and the column operand's L2 working set stays a few tiles
// instead of the whole cloud (a row-major walk spreads the owners' columns over all of
// it). The segments and their partial slots are those of the row-major walk.
struct SegOrder {
  int64_t tb, te, NT, v0, n;
  __device__ __forceinline__ SegOrder(int64_t tb_, int64_t te_, int64_t nt)
      : tb(tb_), te(te_), NT(nt), v0(tb_ / nt), n(te_ > tb_ ? (te_ - 1) / nt - tb_ / nt + 1 : 0) {}
  // Segment i (0 <= i < n) as the unit range [a, b) of one row tile.
  __device__ __forceinline__ void get(int64_t i, int64_t& a, int64_t& b) const {
    const int64_t j = n >= 2 ? (i == 0 ? n - 1 : i - 1) : i;
    const int64_t v = v0 + j;
    a = tb > v * NT ? tb : v * NT;
    b = te < (v + 1) * NT ? te : (v + 1) * NT;
  }
};

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
