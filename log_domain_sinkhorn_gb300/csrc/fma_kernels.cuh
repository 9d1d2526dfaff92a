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
#include "ptx.cuh"

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

// Online base-2 LSE update of two rows at once, (M0, S0) and (M1, S1), with a chunk of J
// score pairs s2[j] = (row 0's score, row 1's score) (packed fp32x2): per-row maxima, then
// the shift, the sum of exponentials and its accumulation on packed instructions.
template <int J>
__device__ __forceinline__ void lse_chunk_pair(const uint64_t (&s2)[J], float& M0, float& S0,
                                               float& M1, float& S1) {
  float a[J], b[J];
#pragma unroll
  for (int j = 0; j < J; ++j) ptx::unpack2(s2[j], a[j], b[j]);
  float mx0 = a[0], mx1 = b[0];
#pragma unroll
  for (int j = 1; j + 1 < J; j += 2) {
    mx0 = ptx::max3(mx0, a[j], a[j + 1]);
    mx1 = ptx::max3(mx1, b[j], b[j + 1]);
  }
  if constexpr (J % 2 == 0) {
    mx0 = fmaxf(mx0, a[J - 1]);
    mx1 = fmaxf(mx1, b[J - 1]);
  }
  if (mx0 > M0) {
    S0 *= ex2(M0 - mx0);
    M0 = mx0;
  }
  if (mx1 > M1) {
    S1 *= ex2(M1 - mx1);
    M1 = mx1;
  }
  const uint64_t nm2 = ptx::pack2(-M0, -M1);
  uint64_t acc2 = 0ull;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    float d0, d1;
    ptx::unpack2(ptx::add2(s2[j], nm2), d0, d1);
    acc2 = ptx::add2(acc2, ptx::pack2(ex2(d0), ex2(d1)));
  }
  float t0, t1;
  ptx::unpack2(acc2, t0, t1);
  S0 += t0;
  S1 += t1;
}

// ---------------------------------------------------------------------------------------
// LSE pass, d_pad = DP <= 32 (multiple of 4): each thread owns R rows (R even), x in
// registers as row pairs: x2[p][k] = (x_{2p,k}, x_{2p+1,k}). The staged column tile keeps
// every coordinate and bias duplicated, (y_k, y_k), so one packed FMA (fma.rn.f32x2)
// advances the dot products of two rows: half the issue slots of scalar FMAs for the same
// FMA-pipe work.
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
  static_assert(R % 2 == 0, "rows are processed in pairs");
  static_assert(kFmaBN == kFmaThreads, "one bias entry per thread");
  constexpr int Q = DP / 4;
  constexpr int P = R / 2;
  __shared__ __align__(16) float2 ys2[kFmaBN * DP];  // (y_k, y_k) per column and coordinate
  __shared__ __align__(16) float2 cs2[kFmaBN];
  const int tid = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * (kFmaThreads * R) + tid;

  uint64_t x2[P][DP];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int64_t ra = row0 + (int64_t)(2 * p) * kFmaThreads;
    const int64_t rb = ra + kFmaThreads;
    const float4* sa = reinterpret_cast<const float4*>(rowP + (ra < n_rows ? ra : 0) * DP);
    const float4* sb = reinterpret_cast<const float4*>(rowP + (rb < n_rows ? rb : 0) * DP);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float4 a = sa[q], b = sb[q];
      x2[p][4 * q + 0] = ptx::pack2(a.x, b.x);
      x2[p][4 * q + 1] = ptx::pack2(a.y, b.y);
      x2[p][4 * q + 2] = ptx::pack2(a.z, b.z);
      x2[p][4 * q + 3] = ptx::pack2(a.w, b.w);
    }
  }
  float M[R], S[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    M[r] = kNegBig;
    S[r] = 0.0f;
  }
  const uint64_t k2 = ptx::pack2(kappa, kappa);

  const int t0 = blockIdx.y * tiles_per_split;
  const int t1 = min(t0 + tiles_per_split, n_col_tiles);
  for (int t = t0; t < t1; ++t) {
    __syncthreads();
    const float* src = colP + (int64_t)t * kFmaBN * DP;
    for (int e = tid; e < kFmaBN * DP; e += kFmaThreads) {
      const float v = src[e];
      ys2[e] = make_float2(v, v);
    }
    const float cb = colBias[(int64_t)t * kFmaBN + tid];
    cs2[tid] = make_float2(cb, cb);
    __syncthreads();
    const uint64_t* ysp = reinterpret_cast<const uint64_t*>(ys2);
    const uint64_t* csp = reinterpret_cast<const uint64_t*>(cs2);
#pragma unroll 1
    for (int jc = 0; jc < kFmaBN; jc += kFmaJ) {
      uint64_t s2[P][kFmaJ];
#pragma unroll
      for (int jj = 0; jj < kFmaJ; ++jj) {
        const uint64_t* y2 = ysp + (jc + jj) * DP;
        uint64_t acc[P];
#pragma unroll
        for (int p = 0; p < P; ++p) acc[p] = 0ull;
#pragma unroll
        for (int k = 0; k < DP; ++k) {
          const uint64_t yk = y2[k];
#pragma unroll
          for (int p = 0; p < P; ++p) acc[p] = ptx::fma2(x2[p][k], yk, acc[p]);
        }
        const uint64_t c2 = csp[jc + jj];
#pragma unroll
        for (int p = 0; p < P; ++p) s2[p][jj] = ptx::fma2(k2, acc[p], c2);
      }
#pragma unroll
      for (int p = 0; p < P; ++p)
        lse_chunk_pair<kFmaJ>(s2[p], M[2 * p], S[2 * p], M[2 * p + 1], S[2 * p + 1]);
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
// static: this header is included by more than one translation unit
static __global__ void __launch_bounds__(kFmaThreads)
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

// The same weighted sums with R (even) rows per thread processed as row pairs on packed
// fp32x2 instructions, as in lse_fma_small_kernel: the row points (and the u_i of HessT) are
// held as pairs x2[p][k] = (x_{2p,k}, x_{2p+1,k}); the staged column coordinates, biases and
// values of V are duplicated, (v, v), so every packed operand is one shared-memory load.
// Same arguments, grid and outputs as wsum_fma_small_kernel.
// kFoldRow (d < DP, Apply and HessT only): the whole exponent comes out of the dot product.
// kappa is applied to the row coordinates once at load, the row bias rides in the first
// padding lane (x_{i,d} = r_i against y_{j,d} = 1 in the staged column tile) and the dot
// starts from c_j, so s_ij = c_j + sum_k (kappa x_ik) y_jk + r_i with no epilogue
// arithmetic: d_pad + 1 FMA-pipe operations per score instead of d_pad + 2.
// Column tiles are double-buffered: the next tile's loads are issued before the current
// tile's scores and stored to the other buffer after them, one barrier per tile.
template <int DP, int MODE, int KO, int R, bool kFoldRow = false>
__global__ void __launch_bounds__(kFmaThreads, DP <= 4 ? 8 : 1)  // 8 CTAs per SM at d_pad 4
wsum_fma_pair_kernel(const float* __restrict__ rowP, const float* __restrict__ colP,
                     const float* __restrict__ colBias, const float* __restrict__ rowBias,
                     int64_t n_rows, int64_t n_cols, int n_col_tiles, float kappa,
                     const float* __restrict__ V, int64_t ldv, int64_t k,
                     const float* __restrict__ rowW, const float* __restrict__ Xrow,
                     int64_t d, float* __restrict__ out, int64_t ldo,
                     const float* __restrict__ rowU, int tiles_per_split = 0,
                     float* __restrict__ part = nullptr, int64_t rows_pad = 0, int kp = 0) {
  static_assert(R % 2 == 0, "rows are processed in pairs");
  constexpr int Q = DP / 4;
  constexpr int P = R / 2;
  constexpr bool kHess = (MODE == kWsumHessT);
  constexpr bool kHad = (MODE == kWsumHadamard);
  constexpr int KV = kHad ? 1 : KO;
  static_assert(!(kFoldRow && kHad), "the Hadamard sum needs the plain dot product");
  static_assert((32 * DP) % kFmaThreads == 0, "whole column tiles per thread");
  constexpr int kYPer = 32 * DP / kFmaThreads;               // staged coordinates per thread
  constexpr int kVPer = (32 * KV + kFmaThreads - 1) / kFmaThreads;  // staged V entries
  __shared__ __align__(16) float2 ys2[2][32 * DP];
  __shared__ __align__(16) float2 cs2[2][32];
  __shared__ __align__(16) float2 vs2[2][32][KV];
  const int tid = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * kFmaThreads * R + tid;
  const int64_t o0 = (int64_t)blockIdx.y * KO;
  const uint64_t k2 = ptx::pack2(kappa, kappa);
  uint64_t x2[P][DP], u2[P][kHess ? DP : 1], rb2[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int64_t ra = row0 + (int64_t)(2 * p) * kFmaThreads;
    const int64_t rb = ra + kFmaThreads;
    const int64_t qa = ra < n_rows ? ra : 0, qb = rb < n_rows ? rb : 0;
    const float4* xa = reinterpret_cast<const float4*>(rowP + qa * DP);
    const float4* xb = reinterpret_cast<const float4*>(rowP + qb * DP);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float4 a = xa[q], b = xb[q];
      x2[p][4 * q + 0] = ptx::pack2(a.x, b.x);
      x2[p][4 * q + 1] = ptx::pack2(a.y, b.y);
      x2[p][4 * q + 2] = ptx::pack2(a.z, b.z);
      x2[p][4 * q + 3] = ptx::pack2(a.w, b.w);
    }
    if constexpr (kHess) {
      const float4* ua = reinterpret_cast<const float4*>(rowU + qa * DP);
      const float4* ub = reinterpret_cast<const float4*>(rowU + qb * DP);
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const float4 a = ua[q], b = ub[q];
        u2[p][4 * q + 0] = ptx::pack2(a.x, b.x);
        u2[p][4 * q + 1] = ptx::pack2(a.y, b.y);
        u2[p][4 * q + 2] = ptx::pack2(a.z, b.z);
        u2[p][4 * q + 3] = ptx::pack2(a.w, b.w);
      }
    }
    const float rba = ra < n_rows ? rowBias[ra] : neg_inf();
    const float rbb = rb < n_rows ? rowBias[rb] : neg_inf();
    rb2[p] = ptx::pack2(rba, rbb);
    if constexpr (kFoldRow) {
      const uint64_t f2 = ptx::pack2(rba, rbb);
#pragma unroll
      for (int kk = 0; kk < DP; ++kk) x2[p][kk] = (kk == d) ? f2 : ptx::mul2(k2, x2[p][kk]);
    }
  }
  uint64_t acc2[P][KV], sw2[P], hd2[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    sw2[p] = 0ull;
    hd2[p] = 0ull;
#pragma unroll
    for (int o = 0; o < KV; ++o) acc2[p][o] = 0ull;
  }
  int t_begin = 0, t_end = n_col_tiles;
  if (part != nullptr) {
    t_begin = (int)blockIdx.z * tiles_per_split;
    t_end = min(n_col_tiles, t_begin + tiles_per_split);
  }
  // staging of column tile t: global loads into registers (fetch), then duplicated into
  // buffer b of shared memory (put)
  float ypre[kYPer], cpre = 0.0f, vpre[kVPer];
  auto fetch = [&](int t) {
    const float* src = colP + (int64_t)t * 32 * DP;
#pragma unroll
    for (int i = 0; i < kYPer; ++i) {
      const int e = tid + i * kFmaThreads;
      ypre[i] = (kFoldRow && e % DP == d) ? 1.0f : src[e];
    }
    if (tid < 32) cpre = colBias[(int64_t)t * 32 + tid];
    if constexpr (!kHad) {
#pragma unroll
      for (int i = 0; i < kVPer; ++i) {
        const int e = tid + i * kFmaThreads;
        const int c = e / KO, o = e % KO;
        const int64_t j = (int64_t)t * 32 + c, oo = o0 + o;
        vpre[i] = (e < 32 * KO && j < n_cols && oo < k) ? V[j * ldv + oo] : 0.0f;
      }
    }
  };
  auto put = [&](int b) {
#pragma unroll
    for (int i = 0; i < kYPer; ++i) ys2[b][tid + i * kFmaThreads] = make_float2(ypre[i], ypre[i]);
    if (tid < 32) cs2[b][tid] = make_float2(cpre, cpre);
    if constexpr (!kHad) {
#pragma unroll
      for (int i = 0; i < kVPer; ++i) {
        const int e = tid + i * kFmaThreads;
        if (e < 32 * KO) vs2[b][e / KO][e % KO] = make_float2(vpre[i], vpre[i]);
      }
    }
  };
  if (t_begin < t_end) {
    fetch(t_begin);
    put(0);
  }
  __syncthreads();
  for (int t = t_begin; t < t_end; ++t) {
    const int b = (t - t_begin) & 1;
    const bool more = t + 1 < t_end;
    if (more) fetch(t + 1);
    const uint64_t* ysp = reinterpret_cast<const uint64_t*>(ys2[b]);
    const uint64_t* csp = reinterpret_cast<const uint64_t*>(cs2[b]);
#pragma unroll 2
    for (int c = 0; c < 32; ++c) {
      const uint64_t* y2 = ysp + c * DP;
      const uint64_t c2 = csp[c];
      uint64_t vv[KV];
      if constexpr (!kHad) {
        const uint64_t* vp = reinterpret_cast<const uint64_t*>(vs2[b][c]);
#pragma unroll
        for (int o = 0; o < KV; ++o) vv[o] = vp[o];
      }
      uint64_t dot[P], tu[P];
#pragma unroll
      for (int p = 0; p < P; ++p) {
        dot[p] = kFoldRow ? c2 : 0ull;
        tu[p] = 0ull;
      }
#pragma unroll
      for (int kk = 0; kk < DP; ++kk) {
        const uint64_t yk = y2[kk];
#pragma unroll
        for (int p = 0; p < P; ++p) {
          dot[p] = ptx::fma2(x2[p][kk], yk, dot[p]);
          if constexpr (kHess) tu[p] = ptx::fma2(u2[p][kk], yk, tu[p]);
        }
      }
#pragma unroll
      for (int p = 0; p < P; ++p) {
        float e0, e1;
        if constexpr (kFoldRow)
          ptx::unpack2(dot[p], e0, e1);
        else
          ptx::unpack2(ptx::add2(ptx::fma2(k2, dot[p], c2), rb2[p]), e0, e1);
        uint64_t w2 = ptx::pack2(ex2(e0), ex2(e1));
        if constexpr (kHad) {
          hd2[p] = ptx::fma2(w2, dot[p], hd2[p]);
        } else {
          if constexpr (kHess) w2 = ptx::mul2(w2, tu[p]);
#pragma unroll
          for (int o = 0; o < KV; ++o) acc2[p][o] = ptx::fma2(w2, vv[o], acc2[p][o]);
          if constexpr (MODE == kWsumGrad) sw2[p] = ptx::add2(sw2[p], w2);
        }
      }
    }
    // buffer b ^ 1 was last read in the previous tile, before the previous barrier
    if (more) put(b ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int p = 0; p < P; ++p) {
    float accA[KV], accB[KV];
#pragma unroll
    for (int o = 0; o < KV; ++o) ptx::unpack2(acc2[p][o], accA[o], accB[o]);
    float swA, swB, hdA, hdB;
    ptx::unpack2(sw2[p], swA, swB);
    ptx::unpack2(hd2[p], hdA, hdB);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t row = row0 + (int64_t)(2 * p + h) * kFmaThreads;
      if (row >= n_rows) continue;
      // h is a compile-time constant in each unrolled copy: the selections stay in registers
      float acc[KO];
#pragma unroll
      for (int o = 0; o < KO; ++o) acc[o] = kHad ? 0.0f : (h ? accB[o < KV ? o : 0] : accA[o < KV ? o : 0]);
      const float sumw = h ? swB : swA, had = h ? hdB : hdA;
      if (part != nullptr) {
        float* pr = part + ((int64_t)blockIdx.z * rows_pad + row) * kp;
        if constexpr (!kHad) {
#pragma unroll
          for (int o = 0; o < KO; ++o)
            if (o0 + o < kp - 1) pr[o0 + o] = acc[o];
        }
        if (blockIdx.y == 0) pr[kp - 1] = kHad ? had : sumw;
      } else {
        wsum_store<MODE, KO>(acc, sumw, had, row, o0, k, rowW, Xrow, d, out, ldo);
      }
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

// The same sum with kSplitLanes consecutive threads per (row, output column): lane l adds
// splits l, l + 8, ... and the lanes combine by a fixed xor tree, so each thread waits on
// n_splits / 8 loads instead of n_splits (the CUDA-core passes split their columns up to
// 64 ways). blockDim.x must be a multiple of 32; any grid size (grid-stride).
constexpr int kSplitLanes = 8;
template <int MODE>
__global__ void wsum_split_reduce_lanes_kernel(const float* __restrict__ part, int n_splits,
                                               int64_t rows_pad, int kp, int64_t n_rows,
                                               int64_t k, const float* __restrict__ rowW,
                                               const float* __restrict__ Xrow, int64_t d,
                                               float* __restrict__ out, int64_t ldo) {
  const int64_t kk = (MODE == kWsumHadamard) ? 1 : k;
  const int64_t n_el = n_rows * kk;
  const int l = threadIdx.x % kSplitLanes;
  // the loop bound depends on the block only: every lane of a warp runs every shuffle
  for (int64_t base = blockIdx.x * (int64_t)blockDim.x; base < n_el * kSplitLanes;
       base += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = (base + threadIdx.x) / kSplitLanes;
    const bool valid = e < n_el;
    const int64_t row = valid ? e / kk : 0, o = valid ? e - row * kk : 0;
    const int col = (MODE == kWsumHadamard) ? kp - 1 : (int)o;
    float acc = 0.0f, sumw = 0.0f;
    if (valid) {
      for (int sp = l; sp < n_splits; sp += kSplitLanes) {
        const float* pr = part + ((int64_t)sp * rows_pad + row) * kp;
        acc += pr[col];
        if constexpr (MODE == kWsumGrad) sumw += pr[kp - 1];
      }
    }
#pragma unroll
    for (int x = kSplitLanes / 2; x > 0; x >>= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, x);
      if constexpr (MODE == kWsumGrad) sumw += __shfl_xor_sync(0xffffffffu, sumw, x);
    }
    if (!valid || l != 0) continue;
    if constexpr (MODE == kWsumGrad) {
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
