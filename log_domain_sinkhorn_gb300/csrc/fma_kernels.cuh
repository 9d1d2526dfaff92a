// fma_kernels.cuh -- CUDA-core (fp32 FMA) streaming passes.
//
// Used for small d (d < 32, where a tensor-core tile would be mostly padding and the
// epilogue dominates anyway) and for the FP32 precision option at any d. Like the
// tensor-core kernels they never form the n x m score matrix: each CTA keeps its rows'
// online (max, sum) state in registers and streams column tiles through shared memory
// (FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract: tiles streamed
// through on-chip SRAM, potentials updated in a single pass).
//
// Two families:
//  * lse_*   : one half-step's row-wise base-2 log-sum-exp, split over column ranges;
//              each split writes a (max, sum) partial, lse_combine_kernel merges them.
//  * wsum_*  : weighted sums with weights w_ij = exp2(kappa <p_i, q_j> + c_j + r_i):
//              transport application (P V), the barycentric gradient (softmax-weighted
//              Y), the Hadamard-weighted transport (sum_j P_ij <x_i, y_j>) and the
//              Hessian curvature term (sum_j P_ij <u_i, y_j> y_j).
#pragma once

#include "common.cuh"

namespace flashot {

constexpr int kFmaThreads = 128;
constexpr int kFmaBN = 128;  // columns per shared-memory tile, small-d LSE kernel
constexpr int kFmaJ = 8;     // columns per online-LSE chunk

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

// Online base-2 LSE update of (M, S) with a chunk of J scores.
template <int J>
__device__ __forceinline__ void lse_chunk(const float (&s)[J], float& M, float& S) {
  float mx = s[0];
#pragma unroll
  for (int j = 1; j < J; ++j) mx = fmaxf(mx, s[j]);
  if (mx > M) {
    S *= ex2(M - mx);
    M = mx;
  }
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < J; ++j) acc += ex2(s[j] - M);
  S += acc;
}

// ---------------------------------------------------------------------------------------
// LSE pass, d_pad = DP <= 32 (multiple of 4): each thread owns R rows, x in registers.
// rowP: n_rows x DP, colP: (n_col_tiles*kFmaBN) x DP, packed fp32 (zero padded).
// Grid: (row blocks, splits). Split s covers column tiles [s*tps, (s+1)*tps).
// ---------------------------------------------------------------------------------------
template <int DP, int R>
__global__ void __launch_bounds__(kFmaThreads)
lse_fma_small_kernel(const float* __restrict__ rowP, const float* __restrict__ colP,
                     const float* __restrict__ colBias, int64_t n_rows, int n_col_tiles,
                     int tiles_per_split, float kappa, float2* __restrict__ partial,
                     int64_t ld) {
  static_assert(DP % 4 == 0 && DP <= 32, "DP must be a multiple of 4, at most 32");
  static_assert(kFmaBN == kFmaThreads, "one bias entry per thread");
  constexpr int Q = DP / 4;
  __shared__ float4 ys[kFmaBN * Q];
  __shared__ float cs[kFmaBN];
  const int tid = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * (kFmaThreads * R) + tid;

  float4 x[R][Q];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = row0 + (int64_t)r * kFmaThreads;
    const float4* src = reinterpret_cast<const float4*>(rowP + (row < n_rows ? row : 0) * DP);
#pragma unroll
    for (int q = 0; q < Q; ++q) x[r][q] = src[q];
  }
  float M[R], S[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    M[r] = kNegBig;
    S[r] = 0.0f;
  }

  const int t0 = blockIdx.y * tiles_per_split;
  const int t1 = min(t0 + tiles_per_split, n_col_tiles);
  for (int t = t0; t < t1; ++t) {
    __syncthreads();
    const float4* src = reinterpret_cast<const float4*>(colP + (int64_t)t * kFmaBN * DP);
    for (int e = tid; e < kFmaBN * Q; e += kFmaThreads) ys[e] = src[e];
    cs[tid] = colBias[(int64_t)t * kFmaBN + tid];
    __syncthreads();
#pragma unroll 1
    for (int jc = 0; jc < kFmaBN; jc += kFmaJ) {
      float s[R][kFmaJ];
#pragma unroll
      for (int jj = 0; jj < kFmaJ; ++jj) {
        float acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = 0.0f;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const float4 y = ys[(jc + jj) * Q + q];
#pragma unroll
          for (int r = 0; r < R; ++r) acc[r] = dot4(x[r][q], y, acc[r]);
        }
        const float c = cs[jc + jj];
#pragma unroll
        for (int r = 0; r < R; ++r) s[r][jj] = fmaf(kappa, acc[r], c);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) lse_chunk<kFmaJ>(s[r], M[r], S[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = row0 + (int64_t)r * kFmaThreads;
    if (row < n_rows) partial[blockIdx.y * ld + row] = make_float2(M[r], S[r]);
  }
}

// ---------------------------------------------------------------------------------------
// LSE pass, any d_pad (multiple of 32): one row per thread; dots for 32 columns are
// accumulated over 32-wide k-chunks staged in shared memory.
// colP has n_col_tiles*32 rows.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kFmaThreads)
lse_fma_generic_kernel(const float* __restrict__ rowP, const float* __restrict__ colP,
                       const float* __restrict__ colBias, int64_t n_rows, int64_t d_pad,
                       int n_col_tiles, int tiles_per_split, float kappa,
                       float2* __restrict__ partial, int64_t ld) {
  __shared__ float4 ys[32 * 8];
  __shared__ float cs[32];
  const int tid = threadIdx.x;
  const int64_t row = (int64_t)blockIdx.x * kFmaThreads + tid;
  const float4* xr = reinterpret_cast<const float4*>(rowP + (row < n_rows ? row : 0) * d_pad);
  const int nkc = (int)(d_pad / 32);
  float M = kNegBig, S = 0.0f;
  const int t0 = blockIdx.y * tiles_per_split;
  const int t1 = min(t0 + tiles_per_split, n_col_tiles);
  for (int t = t0; t < t1; ++t) {
    float acc[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) acc[c] = 0.0f;
    for (int kc = 0; kc < nkc; ++kc) {
      __syncthreads();
      for (int e = tid; e < 256; e += kFmaThreads) {
        const int c = e >> 3, q = e & 7;
        ys[e] = reinterpret_cast<const float4*>(colP + ((int64_t)t * 32 + c) * d_pad +
                                                (int64_t)kc * 32)[q];
      }
      if (kc == 0 && tid < 32) cs[tid] = colBias[(int64_t)t * 32 + tid];
      __syncthreads();
      float4 xv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) xv[q] = xr[kc * 8 + q];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[c] = dot4(xv[q], ys[c * 8 + q], acc[c]);
      }
    }
#pragma unroll
    for (int c0 = 0; c0 < 32; c0 += kFmaJ) {
      float s[kFmaJ];
#pragma unroll
      for (int j = 0; j < kFmaJ; ++j) s[j] = fmaf(kappa, acc[c0 + j], cs[c0 + j]);
      lse_chunk<kFmaJ>(s, M, S);
    }
  }
  if (row < n_rows) partial[blockIdx.y * ld + row] = make_float2(M, S);
}

// Final write of a weighted-sum row (shared by the two wsum kernels); KO output columns.
template <int MODE, int KO>
__device__ __forceinline__ void wsum_store(const float (&acc)[KO], float sumw, float had,
                                           int64_t row, int64_t o0, int64_t k,
                                           const float* __restrict__ rowW,
                                           const float* __restrict__ Xrow, int64_t d,
                                           float* __restrict__ out, int64_t ldo) {
  if constexpr (MODE == kWsumHadamard) {
    out[row] = had;
  } else if constexpr (MODE == kWsumGrad) {
    // grad_i = 2 a_i (x_i - yhat_i), yhat_i = sum_j w_ij y_j / sum_j w_ij
    const float a = rowW[row];
    const float inv = sumw > 0.0f ? 1.0f / sumw : 0.0f;
#pragma unroll
    for (int o = 0; o < KO; ++o) {
      const int64_t oo = o0 + o;
      if (oo < d) out[row * ldo + oo] = a > 0.0f ? 2.0f * a * (Xrow[row * d + oo] - acc[o] * inv)
                                                 : 0.0f;
    }
  } else {
#pragma unroll
    for (int o = 0; o < KO; ++o) {
      const int64_t oo = o0 + o;
      if (oo < k) out[row * ldo + oo] = acc[o];
    }
  }
}

// Stage a 32-column x KO-output tile of V (rows of V are the pass's columns j), zero
// padded in both directions.
template <int KO>
__device__ __forceinline__ void stage_v_tile(float (*vs)[KO + 1], const float* __restrict__ V,
                                             int64_t ldv, int64_t n_cols, int64_t k,
                                             int64_t j0, int64_t o0, int tid) {
  for (int e = tid; e < 32 * KO; e += kFmaThreads) {
    const int c = e / KO, o = e % KO;
    const int64_t j = j0 + c, oo = o0 + o;
    vs[c][o] = (j < n_cols && oo < k) ? V[j * ldv + oo] : 0.0f;
  }
}

// ---------------------------------------------------------------------------------------
// Weighted sums, d_pad = DP <= 32. One row per thread; output columns [o0, o0+KO) per
// blockIdx.y. w_ij = exp2(kappa <p_i, q_j> + c_j + r_i).
//  Apply:    out_i[o] = sum_j w_ij V_j[o]
//  Grad:     V = packed column points; out_i = 2 a_i (x_i - sum_j w_ij q_j / sum_j w_ij)
//  Hadamard: out_i = sum_j w_ij <p_i, q_j>
//  HessT:    out_i[o] = sum_j w_ij <u_i, q_j> V_j[o], u_i the rows of rowU (packed like
//            rowP) and V the column points
// ---------------------------------------------------------------------------------------
// Column splits: with part != NULL, CTA (x, y, z) covers the column tiles
// [z tps, (z+1) tps) and writes its raw sums to part[(z rows_pad + row) kp + o] (and sum w
// or the Hadamard sum to column kp - 1); wsum_split_reduce_kernel adds the splits in a fixed
// order and applies the mode's epilogue. This gives the small-d passes enough CTAs when the
// rows alone would leave most SMs idle.
template <int DP, int MODE, int KO = 32, int R = 1>
__global__ void __launch_bounds__(kFmaThreads)
wsum_fma_small_kernel(const float* __restrict__ rowP, const float* __restrict__ colP,
                      const float* __restrict__ colBias, const float* __restrict__ rowBias,
                      int64_t n_rows, int64_t n_cols, int n_col_tiles, float kappa,
                      const float* __restrict__ V, int64_t ldv, int64_t k,
                      const float* __restrict__ rowW, const float* __restrict__ Xrow,
                      int64_t d, float* __restrict__ out, int64_t ldo,
                      const float* __restrict__ rowU, int tiles_per_split = 0,
                      float* __restrict__ part = nullptr, int64_t rows_pad = 0, int kp = 0) {
  // R rows per thread (rows tid + r kFmaThreads of the CTA's block of kFmaThreads R rows):
  // every staged column is read from shared memory once for R rows.
  constexpr int Q = DP / 4;
  constexpr bool kHess = (MODE == kWsumHessT);
  __shared__ float4 ys[32 * Q];
  __shared__ float cs[32];
  __shared__ float vs[32][KO + 1];
  const int tid = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * kFmaThreads * R + tid;
  const int64_t o0 = (int64_t)blockIdx.y * KO;
  float4 x[R][Q], u[R][kHess ? Q : 1];
  float rb[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = row0 + (int64_t)r * kFmaThreads;
    const int64_t rr = row < n_rows ? row : 0;
    const float4* xr = reinterpret_cast<const float4*>(rowP + rr * DP);
#pragma unroll
    for (int q = 0; q < Q; ++q) x[r][q] = xr[q];
    if constexpr (kHess) {
      const float4* ur = reinterpret_cast<const float4*>(rowU + rr * DP);
#pragma unroll
      for (int q = 0; q < Q; ++q) u[r][q] = ur[q];
    }
    rb[r] = row < n_rows ? rowBias[row] : neg_inf();
  }
  float acc[R][KO];
  float sumw[R], had[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    sumw[r] = 0.0f;
    had[r] = 0.0f;
#pragma unroll
    for (int o = 0; o < KO; ++o) acc[r][o] = 0.0f;
  }
  int t_begin = 0, t_end = n_col_tiles;
  if (part != nullptr) {
    t_begin = (int)blockIdx.z * tiles_per_split;
    t_end = min(n_col_tiles, t_begin + tiles_per_split);
  }
  for (int t = t_begin; t < t_end; ++t) {
    __syncthreads();
    const float4* src = reinterpret_cast<const float4*>(colP + (int64_t)t * 32 * DP);
    for (int e = tid; e < 32 * Q; e += kFmaThreads) ys[e] = src[e];
    if (tid < 32) cs[tid] = colBias[(int64_t)t * 32 + tid];
    if constexpr (MODE != kWsumHadamard)
      stage_v_tile<KO>(vs, V, ldv, n_cols, k, (int64_t)t * 32, o0, tid);
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < 32; ++c) {
      float4 y[Q];
#pragma unroll
      for (int q = 0; q < Q; ++q) y[q] = ys[c * Q + q];
      const float cc = cs[c];
      float vv[MODE == kWsumHadamard ? 1 : KO];
      if constexpr (MODE != kWsumHadamard) {
#pragma unroll
        for (int o = 0; o < KO; ++o) vv[o] = vs[c][o];
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float dot = 0.0f;
#pragma unroll
        for (int q = 0; q < Q; ++q) dot = dot4(x[r][q], y[q], dot);
        float w = ex2(fmaf(kappa, dot, cc) + rb[r]);
        if constexpr (MODE == kWsumHadamard) {
          had[r] = fmaf(w, dot, had[r]);
        } else {
          if constexpr (kHess) {
            float tu = 0.0f;
#pragma unroll
            for (int q = 0; q < Q; ++q) tu = dot4(u[r][q], y[q], tu);
            w *= tu;
          }
#pragma unroll
          for (int o = 0; o < KO; ++o) acc[r][o] = fmaf(w, vv[o], acc[r][o]);
          if constexpr (MODE == kWsumGrad) sumw[r] += w;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = row0 + (int64_t)r * kFmaThreads;
    if (row >= n_rows) continue;
    if (part != nullptr) {
      float* pr = part + ((int64_t)blockIdx.z * rows_pad + row) * kp;
      if constexpr (MODE != kWsumHadamard) {
#pragma unroll
        for (int o = 0; o < KO; ++o)
          if (o0 + o < kp - 1) pr[o0 + o] = acc[r][o];
      }
      if (blockIdx.y == 0) pr[kp - 1] = (MODE == kWsumHadamard) ? had[r] : sumw[r];
    } else {
      wsum_store<MODE, KO>(acc[r], sumw[r], had[r], row, o0, k, rowW, Xrow, d, out, ldo);
    }
  }
}

// Sum of the column splits of a weighted-sum pass (fixed order) and the mode's epilogue
// (see wsum_store). One thread per (row, output column); column kp - 1 holds sum w or the
// Hadamard sum.
template <int MODE>
__global__ void wsum_split_reduce_kernel(const float* __restrict__ part, int n_splits,
                                         int64_t rows_pad, int kp, int64_t n_rows, int64_t k,
                                         const float* __restrict__ rowW,
                                         const float* __restrict__ Xrow, int64_t d,
                                         float* __restrict__ out, int64_t ldo) {
  const int64_t kk = (MODE == kWsumHadamard) ? 1 : k;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n_rows * kk;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / kk, o = e - row * kk;
    const int col = (MODE == kWsumHadamard) ? kp - 1 : (int)o;
    float acc = 0.0f;
    for (int sp = 0; sp < n_splits; ++sp) acc += part[((int64_t)sp * rows_pad + row) * kp + col];
    if constexpr (MODE == kWsumGrad) {
      float sumw = 0.0f;
      for (int sp = 0; sp < n_splits; ++sp)
        sumw += part[((int64_t)sp * rows_pad + row) * kp + kp - 1];
      const float a = rowW[row];
      const float inv = sumw > 0.0f ? 1.0f / sumw : 0.0f;
      out[row * ldo + o] = a > 0.0f ? 2.0f * a * (Xrow[row * d + o] - acc * inv) : 0.0f;
    } else if constexpr (MODE == kWsumHadamard) {
      out[row] = acc;
    } else {
      out[row * ldo + o] = acc;
    }
  }
}

// Weighted sums, any d_pad (multiple of 32): dots for 32 columns accumulated over 32-wide
// k-chunks, then the same epilogue as the small-d kernel.
template <int MODE, int KO = 32>
__global__ void __launch_bounds__(kFmaThreads)
wsum_fma_generic_kernel(const float* __restrict__ rowP, const float* __restrict__ colP,
                        const float* __restrict__ colBias, const float* __restrict__ rowBias,
                        int64_t n_rows, int64_t n_cols, int n_col_tiles, int64_t d_pad,
                        float kappa, const float* __restrict__ V, int64_t ldv, int64_t k,
                        const float* __restrict__ rowW, const float* __restrict__ Xrow,
                        int64_t d, float* __restrict__ out, int64_t ldo,
                        const float* __restrict__ rowU) {
  constexpr bool kHess = (MODE == kWsumHessT);
  __shared__ float4 ys[32 * 8];
  __shared__ float cs[32];
  __shared__ float vs[32][KO + 1];
  const int tid = threadIdx.x;
  const int64_t row = (int64_t)blockIdx.x * kFmaThreads + tid;
  const int64_t o0 = (int64_t)blockIdx.y * KO;
  const int64_t rr = row < n_rows ? row : 0;
  const float4* xr = reinterpret_cast<const float4*>(rowP + rr * d_pad);
  const float4* ur = kHess ? reinterpret_cast<const float4*>(rowU + rr * d_pad) : nullptr;
  const int nkc = (int)(d_pad / 32);
  const float rb = row < n_rows ? rowBias[row] : neg_inf();
  float out_acc[KO];
#pragma unroll
  for (int o = 0; o < KO; ++o) out_acc[o] = 0.0f;
  float sumw = 0.0f, had = 0.0f;
  for (int t = 0; t < n_col_tiles; ++t) {
    float acc[32], tacc[kHess ? 32 : 1];
#pragma unroll
    for (int c = 0; c < 32; ++c) acc[c] = 0.0f;
    if constexpr (kHess) {
#pragma unroll
      for (int c = 0; c < 32; ++c) tacc[c] = 0.0f;
    }
    for (int kc = 0; kc < nkc; ++kc) {
      __syncthreads();
      for (int e = tid; e < 256; e += kFmaThreads) {
        const int c = e >> 3, q = e & 7;
        ys[e] = reinterpret_cast<const float4*>(colP + ((int64_t)t * 32 + c) * d_pad +
                                                (int64_t)kc * 32)[q];
      }
      if (kc == 0) {
        if (tid < 32) cs[tid] = colBias[(int64_t)t * 32 + tid];
        if constexpr (MODE != kWsumHadamard)
          stage_v_tile<KO>(vs, V, ldv, n_cols, k, (int64_t)t * 32, o0, tid);
      }
      __syncthreads();
      float4 xv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) xv[q] = xr[kc * 8 + q];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[c] = dot4(xv[q], ys[c * 8 + q], acc[c]);
      }
      if constexpr (kHess) {
#pragma unroll
        for (int q = 0; q < 8; ++q) xv[q] = ur[kc * 8 + q];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
#pragma unroll
          for (int q = 0; q < 8; ++q) tacc[c] = dot4(xv[q], ys[c * 8 + q], tacc[c]);
        }
      }
    }
#pragma unroll 4
    for (int c = 0; c < 32; ++c) {
      float w = ex2(fmaf(kappa, acc[c], cs[c]) + rb);
      if constexpr (MODE == kWsumHadamard) {
        had = fmaf(w, acc[c], had);
      } else {
        if constexpr (kHess) w *= tacc[c];
#pragma unroll
        for (int o = 0; o < KO; ++o) out_acc[o] = fmaf(w, vs[c][o], out_acc[o]);
        if constexpr (MODE == kWsumGrad) sumw += w;
      }
    }
  }
  if (row < n_rows)
    wsum_store<MODE, KO>(out_acc, sumw, had, row, o0, k, rowW, Xrow, d, out, ldo);
}

}  // namespace flashot
