// prep_kernels.cuh -- packing, norms, log-weights, score biases, LSE combine and loss.
//
// These are the O((n + m) d) steps around the streaming passes: they fold the norms
// |x|^2, |y|^2 and the log-weights into per-row / per-column biases (FlashSinkhorn, SAI
// replication review, "Weaknesses": cost of the form c_ij = alpha_i + beta_j - Q_i^T K_j).
#pragma once

#include "combine.cuh"
#include "common.cuh"
#include "pack_kernels.cuh"

namespace flashot {

// norms[r] = |src_r|^2 from the fp32 input (one warp per row); 0 for padding rows.
__global__ void row_norms_kernel(const float* __restrict__ src, int64_t rows, int64_t d,
                                 int64_t rows_pad, float* __restrict__ norms) {
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows_pad) return;
  float s = 0.0f;
  if (warp < rows) {
    const float* p = src + warp * d;
    for (int64_t c = lane; c < d; c += 32) s = fmaf(p[c], p[c], s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) norms[warp] = s;
}

// w_out[i] = w[i] (or 1/rows if w == NULL), lw2[i] = log2 w_out[i]; padding: 0 and -inf.
// The first thread also clears the workspace status word.
__global__ void weights_kernel(const float* __restrict__ w, int64_t rows, int64_t rows_pad,
                               float* __restrict__ w_out, float* __restrict__ lw2,
                               unsigned* __restrict__ status) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i == 0 && status != nullptr) *status = 0u;
  if (i >= rows_pad) return;
  if (i < rows) {
    const float v = w ? w[i] : (float)(1.0 / (double)rows);
    w_out[i] = v;
    lw2[i] = v > 0.0f ? log2f(v) : neg_inf();
  } else {
    w_out[i] = 0.0f;
    lw2[i] = neg_inf();
  }
}

// Column (or row) bias of a pass whose "other side" has potential pot:
//   bias_i = (pot_i - norm_i) log2(e) / eps + lw2_i ;  pot == NULL means pot = 0.
// Padding entries get -inf so they never contribute.
__global__ void bias_kernel(const float* __restrict__ pot, const float* __restrict__ norms,
                            const float* __restrict__ lw2, int64_t rows, int64_t rows_pad,
                            float inv_eps_log2e, float* __restrict__ bias) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= rows_pad) return;
  if (i < rows) {
    const float p = pot ? pot[i] : 0.0f;
    bias[i] = (p - norms[i]) * inv_eps_log2e + lw2[i];
  } else {
    bias[i] = neg_inf();
  }
}

// Merge per-split (max, sum) partials of the base-2 LSE and finish the half-step (see
// combine_row): one thread per row of rows_pad.
__global__ void lse_combine_kernel(const float2* __restrict__ partial, SplitInfo split,
                                   int64_t ld, CombineArgs args) {
  // Launched as a programmatic dependent of the LSE pass: everything below reads its
  // partials, so wait for it first; the next pass may then start its own prologue.
  griddep_wait();
  griddep_launch_dependents();
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < args.rows_pad) combine_row(partial, ld, split, i, args);
}

// Input check (FLASHOT_VALIDATE): bit 1 of *flag if a coordinate of X or Y is not finite,
// bit 2 if a weight is negative or not finite.
__global__ void validate_kernel(const float* __restrict__ X, int64_t nx,
                                const float* __restrict__ Y, int64_t ny,
                                const float* __restrict__ a, int64_t na,
                                const float* __restrict__ b, int64_t nb,
                                unsigned* __restrict__ flag) {
  unsigned bad = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nx + ny; i += stride) {
    const float v = i < nx ? X[i] : Y[i - nx];
    if (!isfinite(v)) bad |= 1u;
  }
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < na + nb; i += stride) {
    const float w = i < na ? a[i] : b[i - na];
    if (!(w >= 0.0f) || !isfinite(w)) bad |= 2u;
  }
  if (bad) atomicOr(flag, bad);
}

// Plan diagnostics from the marginals r = P 1, c = P^T 1 and the Hadamard sums
// h_i = sum_j P_ij <x_i, y_j> (one block, fp64, fixed order). With <C, P> = sum r alpha +
// sum c beta - 2 sum h and sum P log(P / (a b)) = (sum r f + sum c g - <C, P>) / eps:
//   out = {primal = sum r f + sum c g - eps (sum P - sum a sum b),
//          dual = sum a f + sum b g - eps (sum P - sum a sum b),
//          <C, P>, sum |r - a|, sum |c - b|, sum P}.
__global__ void __launch_bounds__(1024)
diagnostics_kernel(const float* __restrict__ r, const float* __restrict__ c,
                   const float* __restrict__ h, const float* __restrict__ alpha,
                   const float* __restrict__ beta, const float* __restrict__ wa,
                   const float* __restrict__ wb, const float* __restrict__ f,
                   const float* __restrict__ g, int64_t n, int64_t m, double eps,
                   double* __restrict__ out) {
  __shared__ double red[8][33];
  double v[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // rf+cg, af+bg, cost, row_err, col_err, mass, suma, sumb
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const double ri = r[i], ai = wa[i];
    v[0] += ri == 0.0 ? 0.0 : ri * (double)f[i];
    v[1] += ai == 0.0 ? 0.0 : ai * (double)f[i];
    v[2] += ri * (double)alpha[i] - 2.0 * (double)h[i];
    v[3] += fabs(ri - ai);
    v[5] += ri;
    v[6] += ai;
  }
  for (int64_t j = threadIdx.x; j < m; j += blockDim.x) {
    const double cj = c[j], bj = wb[j];
    v[0] += cj == 0.0 ? 0.0 : cj * (double)g[j];
    v[1] += bj == 0.0 ? 0.0 : bj * (double)g[j];
    v[2] += cj * (double)beta[j];
    v[4] += fabs(cj - bj);
    v[7] += bj;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    if ((threadIdx.x & 31) == 0) red[k][threadIdx.x >> 5] = v[k];
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    double t[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      t[k] = (threadIdx.x < (blockDim.x >> 5)) ? red[k][threadIdx.x] : 0.0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t[k] += __shfl_xor_sync(0xffffffffu, t[k], o);
    }
    if (threadIdx.x == 0) {
      const double excess = t[5] - t[6] * t[7];
      out[0] = t[0] - eps * excess;
      out[1] = t[1] - eps * excess;
      out[2] = t[2];
      out[3] = t[3];
      out[4] = t[4];
      out[5] = t[5];
    }
  }
}

__global__ void fill_kernel(float* __restrict__ p, int64_t count, float v) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

// loss = sum_i wa_i f_i + sum_j wb_j g_j in fp64; one block, deterministic order.
__global__ void __launch_bounds__(1024)
dual_loss_kernel(const float* __restrict__ wa, const float* __restrict__ f, int64_t n,
                 const float* __restrict__ wb, const float* __restrict__ g, int64_t m,
                 double* __restrict__ loss) {
  __shared__ double red[32];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) s += (double)wa[i] * (double)f[i];
  for (int64_t j = threadIdx.x; j < m; j += blockDim.x) s += (double)wb[j] * (double)g[j];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) *loss = s;
  }
}

// out = sum_i v_i in fp64; one block, deterministic order (the convergence check's error).
__global__ void __launch_bounds__(1024)
sum_rows_kernel(const float* __restrict__ v, int64_t rows, double* __restrict__ out) {
  __shared__ double red[32];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < rows; i += blockDim.x) s += (double)v[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) *out = s;
  }
}

}  // namespace flashot

namespace flashot {
// out[0] = out[1] - out[2] / 2 - out[3] / 2 (the debiased divergence from its three terms).
__global__ void divergence_combine_kernel(double* __restrict__ out) {
  if (threadIdx.x == 0 && blockIdx.x == 0) out[0] = out[1] - 0.5 * out[2] - 0.5 * out[3];
}
}  // namespace flashot
