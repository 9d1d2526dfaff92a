// hvp_kernels.cuh -- the O((n + m) d) steps of the streaming Hessian-vector product of the
// OT loss w.r.t. X (FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, SAI
// replication review, "Summary" (iii): an HVP oracle built from streaming transport
// applications and a Schur solve, for O((n + m) d)-memory Newton-CG).
//
// At potentials (f, g), with P_ij = a_i b_j exp((f_i + g_j - |x_i - y_j|^2)/eps), r = P 1,
// c = P^T 1, s_i = <x_i, v_i>, (PY)_i = sum_j P_ij y_j and T_i = sum_j P_ij <v_i, y_j> y_j:
//   w_f,i = (2/eps) (r_i s_i - <v_i, (PY)_i>)
//   w_g,j = (2/eps) ((P^T s)_j - <y_j, (P^T V)_j>)
//   K (u, z) = (w_f, w_g),  K = [[diag r, P], [P^T, diag c]]  (solved through the Schur
//      complement S = diag c - P^T diag(1/r) P on z, then u = (w_f - P z) / r)
//   (H V)_i = 2 r_i v_i - (4/eps) (x_i (eps/2) w_f,i - s_i (PY)_i + T_i)
//             + 2 ((r_i x_i - (PY)_i) u_i + x_i (P z)_i - (P diag(z) Y)_i).
// The streaming passes (P [Y | 1], P^T [V | s | 1], T, the CG's P p and P^T t, and
// P [diag(z) Y | z]) run in the weighted-sum kernels; the kernels here assemble their
// inputs and outputs. Every reduction runs in a fixed order (deterministic).
#pragma once

#include "common.cuh"

namespace flashot {

// Scalars the CG keeps on the device (doubles).
enum HvpScalar : int {
  kHvpRho = 0, kHvpRR = 1, kHvpRR0 = 2, kHvpBreak = 3, kHvpRhoOld = 4, kHvpScalars = 8
};
// A CG step runs on up to kCgMaxBlocks CTAs of kCgThreads threads; each writes its block's
// partial sums, and every CTA of the next kernel reduces all of them in the same order.
constexpr int kCgMaxBlocks = 256;
constexpr int kCgThreads = 256;
static_assert(kCgMaxBlocks <= kCgThreads, "one block partial per thread of the reducing CTA");

// VA (m x (d+1)) = [Y | 1];  VB (n x (d+2)) = [V | s | 1] with s_i = <x_i, v_i>.
__global__ void hvp_prep_kernel(const float* __restrict__ X, const float* __restrict__ Y,
                                const float* __restrict__ V, int64_t n, int64_t m, int64_t d,
                                float* __restrict__ VA, float* __restrict__ VB) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t < m) {
    for (int64_t k = 0; k < d; ++k) VA[t * (d + 1) + k] = Y[t * d + k];
    VA[t * (d + 1) + d] = 1.0f;
  }
  if (t < n) {
    float s = 0.0f;
    for (int64_t k = 0; k < d; ++k) {
      const float v = V[t * d + k];
      VB[t * (d + 2) + k] = v;
      s = fmaf(X[t * d + k], v, s);
    }
    VB[t * (d + 2) + d] = s;
    VB[t * (d + 2) + d + 1] = 1.0f;
  }
}

// w_f,i from OA = [PY | r] and VB; t1_i = w_f,i / r_i (0 for rows without mass).
__global__ void hvp_rhs_kernel(const float* __restrict__ OA, const float* __restrict__ VB,
                               int64_t n, int64_t d, float eps, float* __restrict__ wf,
                               float* __restrict__ t1) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float* pa = OA + i * (d + 1);
  const float* vb = VB + i * (d + 2);
  float vpy = 0.0f;
  for (int64_t k = 0; k < d; ++k) vpy = fmaf(vb[k], pa[k], vpy);
  const float r = pa[d];
  const float w = (2.0f / eps) * (r * vb[d] - vpy);
  wf[i] = w;
  t1[i] = r > 0.0f ? w / r : 0.0f;
}

// y = a / b elementwise (0 where b <= 0), reading b with a stride (a column of a matrix).
__global__ void hvp_div_kernel(const float* __restrict__ a, const float* __restrict__ b,
                               int64_t ldb, int64_t n, float* __restrict__ y) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float bi = b[i * ldb];
  y[i] = bi > 0.0f ? a[i] / bi : 0.0f;
}

// Per-thread running sum in fp32 with Neumaier compensation (the pair s + c carries about
// twice fp32's precision). The CG's single-block reductions accumulate their ~m / 1024 terms
// per thread this way and combine only the 1024 partials in fp64: GB300's fp64 pipe is a
// small fraction of its fp32 one, and fp64 per element made these one-SM kernels the
// largest cost of a CG step after the streaming passes.
struct Sum32 {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float x) {
    const float t = s + x;
    c += (fabsf(s) >= fabsf(x)) ? (s - t) + x : (x - t) + s;
    s = t;
  }
  __device__ __forceinline__ double value() const { return (double)s + (double)c; }
};

// Block-wide fp64 sum (blockDim.x a multiple of 32, at most 1024); every thread receives
// the result. The tree is fixed, so every block reducing the same values gets the same sum.
__device__ __forceinline__ double block_sum(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    double s = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) red[32] = s;
  }
  __syncthreads();
  return red[32];
}

// S is singular: S 1 = 0, and rows / columns of points without mass (c_j = 0) are zero. Its
// range is {v : v_j = 0 where c_j = 0, sum of the other v_j = 0}. The right-hand side lies
// there analytically, but for smooth V it is a small difference of large terms, and fp32
// rounding leaves a null-space component that CG cannot remove (the residual stalls). So
// the right-hand side and every S p are projected onto the range: the mean over the
// columns with mass is subtracted from them.

// CG start on S z = rhs, rhs_j = w_g,j - PtT_j (projected), w_g from OB = [P^T V | P^T s | c];
// preconditioner diag(c). z = 0, res = rhs, yv = res / c, p = yv.
__global__ void __launch_bounds__(1024)
hvp_cg_init_kernel(const float* __restrict__ Y, const float* __restrict__ OB,
                   const float* __restrict__ PtT, int64_t m, int64_t d, float eps,
                   float* __restrict__ z, float* __restrict__ res, float* __restrict__ yv,
                   float* __restrict__ p, double* __restrict__ sc) {
  __shared__ double red[33];
  Sum32 s_sum;
  int n_mass = 0;
  for (int64_t j = threadIdx.x; j < m; j += blockDim.x) {
    const float* ob = OB + j * (d + 2);
    float rhs = 0.0f;
    if (ob[d + 1] > 0.0f) {
      float yptv = 0.0f;
      for (int64_t k = 0; k < d; ++k) yptv = fmaf(Y[j * d + k], ob[k], yptv);
      rhs = (2.0f / eps) * (ob[d] - yptv) - PtT[j];
      s_sum.add(rhs);
      ++n_mass;
    }
    res[j] = rhs;
  }
  const double sum = block_sum(s_sum.value(), red);
  const double cnt = block_sum((double)n_mass, red);
  const float mean = cnt > 0.0 ? (float)(sum / cnt) : 0.0f;
  Sum32 s_rho, s_rr;
  for (int64_t j = threadIdx.x; j < m; j += blockDim.x) {
    const float cj = OB[j * (d + 2) + d + 1];
    const float r = cj > 0.0f ? res[j] - mean : 0.0f;
    const float y = cj > 0.0f ? r / cj : 0.0f;
    z[j] = 0.0f;
    res[j] = r;
    yv[j] = y;
    p[j] = y;
    s_rho.add(r * y);
    s_rr.add(r * r);
  }
  const double rho = block_sum(s_rho.value(), red);
  const double rr = block_sum(s_rr.value(), red);
  if (threadIdx.x == 0) {
    sc[kHvpRho] = rho;
    sc[kHvpRR] = rr;
    sc[kHvpRR0] = rr;
    sc[kHvpBreak] = 0.0;
  }
}

// One preconditioned CG step given PtT = P^T diag(1/r) P p:
//   q = c p - PtT (projected), alpha = rho / <p, q>, z += alpha p, res -= alpha q,
//   yv = res / c, rho' = <res, yv>, p = yv + (rho'/rho) p.  <p, q> <= 0 (S is PSD, so only
//   round-off gives it) stops the iteration (kHvpBreak = 1) without changing z.
// Three kernels over the same grid of G CTAs, each global sum taken between two of them:
//   hvp_cg_q_kernel      partial sums of q, p q, p and the count of columns with mass;
//   hvp_cg_update_kernel alpha from those; z, res, yv; partial sums of res yv and res^2;
//   hvp_cg_dir_kernel    beta from those; p.
// Per thread Sum32, fp64 across the block, fp64 across the G block partials.
__global__ void __launch_bounds__(kCgThreads)
hvp_cg_q_kernel(const float* __restrict__ OB, const float* __restrict__ PtT, int64_t m,
                int64_t d, const float* __restrict__ p, double* __restrict__ part) {
  __shared__ double red[33];
  Sum32 s_q, s_pq, s_p;
  int n_mass = 0;
  for (int64_t j = blockIdx.x * (int64_t)kCgThreads + threadIdx.x; j < m;
       j += (int64_t)gridDim.x * kCgThreads) {
    const float cj = OB[j * (d + 2) + d + 1], pj = p[j], tj = PtT[j];
    if (cj > 0.0f) {
      const float q = cj * pj - tj;
      s_q.add(q);
      s_pq.add(pj * q);
      s_p.add(pj);
      ++n_mass;
    }
  }
  const double sq = block_sum(s_q.value(), red);
  const double spq = block_sum(s_pq.value(), red);
  const double sp = block_sum(s_p.value(), red);
  const double cnt = block_sum((double)n_mass, red);
  if (threadIdx.x == 0) {
    double* o = part + 4 * (int64_t)blockIdx.x;
    o[0] = sq;
    o[1] = spq;
    o[2] = sp;
    o[3] = cnt;
  }
}

__global__ void __launch_bounds__(kCgThreads)
hvp_cg_update_kernel(const float* __restrict__ OB, const float* __restrict__ PtT, int64_t m,
                     int64_t d, float* __restrict__ z, float* __restrict__ res,
                     float* __restrict__ yv, const float* __restrict__ p,
                     const double* __restrict__ part, double* __restrict__ part2,
                     double* __restrict__ sc) {
  __shared__ double red[33];
  const int G = gridDim.x;  // <= kCgThreads: one partial per thread
  const int t = threadIdx.x;
  const double sq = block_sum(t < G ? part[4 * t + 0] : 0.0, red);
  const double spq = block_sum(t < G ? part[4 * t + 1] : 0.0, red);
  const double sp = block_sum(t < G ? part[4 * t + 2] : 0.0, red);
  const double cnt = block_sum(t < G ? part[4 * t + 3] : 0.0, red);
  const double qbar = cnt > 0.0 ? sq / cnt : 0.0;
  const double pq = spq - qbar * sp;
  const double rho = sc[kHvpRho];
  if (!(pq > 0.0) || !(rho > 0.0)) {  // the same decision in every block
    if (blockIdx.x == 0 && t == 0) sc[kHvpBreak] = 1.0;
    return;
  }
  const float alpha = (float)(rho / pq);
  const float qb = (float)qbar;
  Sum32 s_rho, s_rr;
  for (int64_t j = blockIdx.x * (int64_t)kCgThreads + t; j < m;
       j += (int64_t)gridDim.x * kCgThreads) {
    const float cj = OB[j * (d + 2) + d + 1], pj = p[j], tj = PtT[j];
    if (cj > 0.0f) {
      const float q = (cj * pj - tj) - qb;
      z[j] = fmaf(alpha, pj, z[j]);
      const float rj = fmaf(-alpha, q, res[j]);
      res[j] = rj;
      const float y = rj / cj;
      yv[j] = y;
      s_rho.add(rj * y);
      s_rr.add(rj * rj);
    }
  }
  const double r0 = block_sum(s_rho.value(), red);
  const double r1 = block_sum(s_rr.value(), red);
  if (t == 0) {
    part2[2 * (int64_t)blockIdx.x + 0] = r0;
    part2[2 * (int64_t)blockIdx.x + 1] = r1;
    // kHvpRho itself is rewritten by the next kernel while its blocks still need the old one
    if (blockIdx.x == 0) sc[kHvpRhoOld] = rho;
  }
}

__global__ void __launch_bounds__(kCgThreads)
hvp_cg_dir_kernel(int64_t m, float* __restrict__ p, const float* __restrict__ yv,
                  const double* __restrict__ part2, double* __restrict__ sc) {
  __shared__ double red[33];
  if (sc[kHvpBreak] != 0.0) return;
  const int G = gridDim.x;
  const int t = threadIdx.x;
  const double rho_new = block_sum(t < G ? part2[2 * t + 0] : 0.0, red);
  const double rr = block_sum(t < G ? part2[2 * t + 1] : 0.0, red);
  const float beta = (float)(rho_new / sc[kHvpRhoOld]);
  for (int64_t j = blockIdx.x * (int64_t)kCgThreads + t; j < m;
       j += (int64_t)gridDim.x * kCgThreads)
    p[j] = fmaf(beta, p[j], yv[j]);
  if (blockIdx.x == 0 && t == 0) {
    sc[kHvpRho] = rho_new;
    sc[kHvpRR] = rr;
  }
}

// VD (m x (d+1)) = [diag(z) Y | z].
__global__ void hvp_vd_kernel(const float* __restrict__ Y, const float* __restrict__ z,
                              int64_t m, int64_t d, float* __restrict__ VD) {
  const int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (j >= m) return;
  const float zj = z[j];
  for (int64_t k = 0; k < d; ++k) VD[j * (d + 1) + k] = zj * Y[j * d + k];
  VD[j * (d + 1) + d] = zj;
}

// (H V)_i from the pass outputs: OA = [PY | r], VB = [V | s | 1], T, wf, OD = [P diag(z) Y | P z].
__global__ void hvp_final_kernel(const float* __restrict__ X, const float* __restrict__ OA,
                                 const float* __restrict__ VB, const float* __restrict__ T,
                                 const float* __restrict__ wf, const float* __restrict__ OD,
                                 int64_t n, int64_t d, float eps, float* __restrict__ out) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float* pa = OA + i * (d + 1);
  const float* vb = VB + i * (d + 2);
  const float* od = OD + i * (d + 1);
  const float r = pa[d], s = vb[d], w = wf[i], pz = od[d];
  const float u = r > 0.0f ? (w - pz) / r : 0.0f;
  const float c4 = 4.0f / eps;
  for (int64_t k = 0; k < d; ++k) {
    const float x = X[i * d + k], py = pa[k];
    const float lxx = 2.0f * r * vb[k] - c4 * (x * (0.5f * eps * w) - s * py + T[i * d + k]);
    const float lxp = 2.0f * ((r * x - py) * u + x * pz - od[k]);
    out[i * d + k] = lxx + lxp;
  }
}

}  // namespace flashot
