// small_solve.cu -- the whole alternating solve in one launch, for small fp32 problems.
//
// When both clouds, all potentials and the score biases fit in one SM's shared memory, the
// iteration is bound by launch latency (four launches per iteration on the streaming path).
// Here one thread-block cluster (16 CTAs where the GPU can co-schedule that many, else 8)
// runs every stage and iteration inside a single kernel (FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract: the
// f- and g-updates as row-wise log-sum-exps; arithmetic identical to the CUDA-core path):
//  - every CTA keeps X, Y, |x|^2, |y|^2, log2 a, log2 b and full copies of f and g;
//  - for an f-update each CTA computes its slice of rows: lanes own rows, warps own slices
//    of the columns, and the per-warp (max, sum) pairs of a row are merged through shared
//    memory; the CTA then stores its f values into the shared memory of every CTA of the
//    cluster (DSMEM);
//  - a cluster barrier (release / acquire) separates the half-steps.
// All CTAs of a cluster are co-scheduled, and every CTA reaches every barrier, so the
// barriers need no time limit.
#include <cuda_runtime.h>

#include <cstdint>

#include "flashot.h"
#include "common.cuh"
#include "small_solve.h"
#include "trace.h"

namespace flashot {
namespace small {

constexpr int kClusterPortable = 8;  // the portable cluster size
constexpr int kClusterLarge = 16;    // non-portable (opt-in) cluster size
constexpr int kThreads = 512;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Store v into the same shared-memory location of CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster(float* local, uint32_t rank, float v) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

// Rows per lane in a half-step when a CTA owns more than 32 rows (registers hold R points
// of DP floats); with at most 32 rows one row per lane keeps every lane busy.
template <int DP>
constexpr int rows_per_lane() {
  return DP <= 16 ? 2 : 1;
}

// One half-step for the rows [r0, r1) of the side P against the nq points of the other
// side Q, whose column biases cq fold in their potential, norm and log-weight:
// out_i = nrmp_i - eps ln2 LSE2_j(kappa <p_i, q_j> + cq_j), stored into every CTA.
// Lanes own rows (R per lane, 32 R per group) and warps own column slices, so each column's
// point and bias are one broadcast shared-memory read per warp; each warp keeps an online
// (max, sum) per row over its slice in chunks of 8 columns, and the kWarps partials of a row
// are merged through shared memory before the row's value is broadcast to the cluster.
template <int DP, int R>
__device__ __forceinline__ void half_step(const float* __restrict__ P, const float* __restrict__ Q,
                                          int nq, const float* __restrict__ cq,
                                          const float* __restrict__ nrmp, int r0, int r1,
                                          float kappa, float eps, float* out, float2* red) {
  constexpr int kWarps = kThreads / 32;
  const uint32_t ncta = gridDim.x;  // the grid is one cluster
  constexpr int Q4 = DP / 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cs = (nq + kWarps - 1) / kWarps;
  const int j0 = min(nq, warp * cs), j1 = min(nq, j0 + cs);
  for (int base = r0; base < r1; base += 32 * R) {
    float4 x[R][Q4];
    float M[R], S[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int i = base + lane + 32 * r;
      const float4* src = reinterpret_cast<const float4*>(P + (i < r1 ? i : r0) * DP);
#pragma unroll
      for (int q = 0; q < Q4; ++q) x[r][q] = src[q];
      M[r] = kNegBig;
      S[r] = 0.0f;
    }
    for (int j = j0; j < j1; j += 8) {
      float sc[R][8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int jj = j + u;
        if (jj < j1) {
          const float4* yq = reinterpret_cast<const float4*>(Q + jj * DP);
          float4 y[Q4];
#pragma unroll
          for (int q = 0; q < Q4; ++q) y[q] = yq[q];
          const float c = cq[jj];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float dot = 0.0f;
#pragma unroll
            for (int q = 0; q < Q4; ++q) {
              dot = fmaf(x[r][q].x, y[q].x, dot);
              dot = fmaf(x[r][q].y, y[q].y, dot);
              dot = fmaf(x[r][q].z, y[q].z, dot);
              dot = fmaf(x[r][q].w, y[q].w, dot);
            }
            sc[r][u] = fmaf(kappa, dot, c);
          }
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) sc[r][u] = neg_inf();
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float mx = sc[r][0];
#pragma unroll
        for (int u = 1; u < 8; ++u) mx = fmaxf(mx, sc[r][u]);
        if (mx > M[r]) {
          S[r] *= ex2(M[r] - mx);
          M[r] = mx;
        }
        float acc = 0.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += ex2(sc[r][u] - M[r]);
        S[r] += acc;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) red[warp * 32 * R + lane + 32 * r] = make_float2(M[r], S[r]);
    __syncthreads();
    if (tid < 32 * R) {
      const int i = base + tid;
      if (i < r1) {
        float Mx = kNegBig;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) Mx = fmaxf(Mx, red[w * 32 * R + tid].x);
        float Sm = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float2 p = red[w * 32 * R + tid];
          Sm += p.y * ex2(p.x - Mx);
        }
        const float L = Mx + log2f(Sm);
        const float v = nrmp[i] - eps * kLn2 * L;
        for (uint32_t rk = 0; rk < ncta; ++rk) st_cluster(out + i, rk, v);
      }
    }
    __syncthreads();
  }
}

// Launched as a single cluster of gridDim.x CTAs (the cluster size is set at launch).
template <int DP>
__global__ void __launch_bounds__(kThreads, 1)
small_solve_kernel(const float* __restrict__ X, const float* __restrict__ Y,
                   const float* __restrict__ a, const float* __restrict__ b, int n, int m, int d,
                   EpsSchedule sched, int iters, int warm, float* __restrict__ f_out,
                   float* __restrict__ g_out, double* __restrict__ loss_out) {
  extern __shared__ float sm[];
  float* Xs = sm;                 // n x DP
  float* Ys = Xs + n * DP;        // m x DP
  float* fa = Ys + m * DP;        // n
  float* ga = fa + n;             // m
  float* al = ga + m;             // n  |x|^2
  float* be = al + n;             // m  |y|^2
  float* la = be + m;             // n  log2 a
  float* lb = la + n;             // m  log2 b
  float* wa = lb + m;             // n
  float* wb = wa + n;             // m
  float* cb = wb + m;             // max(n, m): bias of the current pass
  // kThreads/32 x 32 R (max, sum) partials of a row group, 8-byte aligned after cb.
  float2* red = reinterpret_cast<float2*>(cb + ((n > m ? n : m) + 1) / 2 * 2);
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();

  for (int e = tid; e < n * DP; e += kThreads) {
    const int i = e / DP, c = e % DP;
    Xs[e] = c < d ? X[(int64_t)i * d + c] : 0.0f;
  }
  for (int e = tid; e < m * DP; e += kThreads) {
    const int j = e / DP, c = e % DP;
    Ys[e] = c < d ? Y[(int64_t)j * d + c] : 0.0f;
  }
  for (int i = tid; i < n; i += kThreads) {
    float s = 0.0f;
    for (int c = 0; c < d; ++c) s = fmaf(X[(int64_t)i * d + c], X[(int64_t)i * d + c], s);
    al[i] = s;
    const float w = a ? a[i] : (float)(1.0 / (double)n);
    wa[i] = w;
    la[i] = w > 0.0f ? log2f(w) : neg_inf();
  }
  for (int j = tid; j < m; j += kThreads) {
    float s = 0.0f;
    for (int c = 0; c < d; ++c) s = fmaf(Y[(int64_t)j * d + c], Y[(int64_t)j * d + c], s);
    be[j] = s;
    const float w = b ? b[j] : (float)(1.0 / (double)m);
    wb[j] = w;
    lb[j] = w > 0.0f ? log2f(w) : neg_inf();
    ga[j] = warm ? g_out[j] : 0.0f;
  }
  __syncthreads();
  cluster_sync();  // every CTA's shared memory is initialised before any remote store

  const int ncta = (int)gridDim.x;
  const int fr0 = (int)(((int64_t)n * rank) / ncta), fr1 = (int)(((int64_t)n * (rank + 1)) / ncta);
  const int gr0 = (int)(((int64_t)m * rank) / ncta), gr1 = (int)(((int64_t)m * (rank + 1)) / ncta);
  constexpr int R2 = rows_per_lane<DP>();
  // every CTA has the same row counts to within one: the choice is uniform over the cluster
  const bool f_one = fr1 - fr0 <= 32, g_one = gr1 - gr0 <= 32;
  for (int s = 0; s < sched.n_stages; ++s) {
    const float eps = sched.eps[s];
    const float kappa = 2.0f * kLog2e / eps;
    const float inv = kLog2e / eps;
    for (int it = 0; it < iters; ++it) {
      // f-update: bias of the columns (Y side) from g
      for (int j = tid; j < m; j += kThreads) cb[j] = (ga[j] - be[j]) * inv + lb[j];
      __syncthreads();
      if (f_one) half_step<DP, 1>(Xs, Ys, m, cb, al, fr0, fr1, kappa, eps, fa, red);
      else half_step<DP, R2>(Xs, Ys, m, cb, al, fr0, fr1, kappa, eps, fa, red);
      cluster_sync();
      // g-update: bias of the columns (X side) from f
      for (int i = tid; i < n; i += kThreads) cb[i] = (fa[i] - al[i]) * inv + la[i];
      __syncthreads();
      if (g_one) half_step<DP, 1>(Ys, Xs, n, cb, be, gr0, gr1, kappa, eps, ga, red);
      else half_step<DP, R2>(Ys, Xs, n, cb, be, gr0, gr1, kappa, eps, ga, red);
      cluster_sync();
    }
  }

  if (rank == 0) {
    for (int i = tid; i < n; i += kThreads) f_out[i] = fa[i];
    for (int j = tid; j < m; j += kThreads) g_out[j] = ga[j];
    if (loss_out) {
      __shared__ double red[kThreads / 32];
      double acc = 0.0;
      for (int i = tid; i < n; i += kThreads) acc += (double)wa[i] * (double)fa[i];
      for (int j = tid; j < m; j += kThreads) acc += (double)wb[j] * (double)ga[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if ((tid & 31) == 0) red[tid >> 5] = acc;
      __syncthreads();
      if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) t += red[w];
        *loss_out = t;
      }
    }
  }
}

size_t smem_bytes(int64_t n, int64_t m, int dp) {
  const int64_t mx = n > m ? n : m;
  const int64_t floats = (n + m) * dp + 5 * (n + m) + (mx + 1) / 2 * 2;
  // partials: kThreads/32 warps x 32 rows-per-group x up to 2 rows per lane, float2 each
  return (size_t)floats * sizeof(float) + (size_t)(kThreads / 32) * 64 * sizeof(float2);
}

// Cluster size for a problem: 16 CTAs (non-portable) when the clouds are large enough to
// use them and the GPU can co-schedule a 16-CTA cluster of this kernel, else 8.
template <int DP>
int cluster_size(int n, int m, size_t bytes) {
  if ((n > m ? n : m) <= 256) return kClusterPortable;
  static int can16 = -1;  // per DP instantiation, decided once per process
  if (can16 < 0) {
    can16 = 0;
    // the query needs the kernel's dynamic shared-memory limit raised to `bytes` first
    if (cudaFuncSetAttribute(small_solve_kernel<DP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
            cudaSuccess &&
        cudaFuncSetAttribute(small_solve_kernel<DP>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kClusterLarge);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = bytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kClusterLarge;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, small_solve_kernel<DP>, &cfg) ==
              cudaSuccess &&
          clusters >= 1)
        can16 = 1;
    }
    cudaGetLastError();  // a refused query leaves no error behind
  }
  return can16 ? kClusterLarge : kClusterPortable;
}

template <int DP>
int launch(const float* X, const float* Y, const float* a, const float* b, int n, int m, int d,
           const EpsSchedule& sched, int iters, int warm, float* f, float* g, double* loss,
           cudaStream_t st) {
  const size_t bytes = smem_bytes(n, m, DP);
  cudaError_t e = cudaFuncSetAttribute(small_solve_kernel<DP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return FLASHOT_ERR_CUDA;
  const int ncta = cluster_size<DP>(n, m, bytes);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ncta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    TraceScope ts_(FLASHOT_KERNEL_LSE, st);
    e = cudaLaunchKernelEx(&cfg, small_solve_kernel<DP>, X, Y, a, b, n, m, d, sched, iters, warm,
                           f, g, loss);
  }
  if (e != cudaSuccess) return FLASHOT_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

}  // namespace small

bool small_solve_eligible(int64_t n, int64_t m, int64_t dp, int n_stages) {
  // Up to n m = 2^20 the single launch is ahead of the streaming path, which is bound by
  // launch latency here (about 21 us per iteration up to 2048^2 at d = 3; the 16-CTA
  // cluster takes 11 us at 1024^2). Just above, a CTA of the 16-CTA cluster owns more than
  // 64 rows and needs a second pass over its row group (1040^2: 23 us per iteration).
  return n_stages <= kSmallMaxStages && dp <= 32 && dp % 4 == 0 && n * m <= (int64_t(1) << 20) &&
         small::smem_bytes(n, m, (int)dp) <= (size_t)200 * 1024;
}

int small_solve(const float* X, const float* Y, const float* a, const float* b, int64_t n,
                int64_t m, int64_t d, int64_t dp, const float* eps_sched, int n_stages,
                int iters, bool warm, float* f, float* g, double* loss, cudaStream_t st) {
  EpsSchedule sched;
  sched.n_stages = n_stages;
  for (int s = 0; s < n_stages; ++s) sched.eps[s] = eps_sched[s];
  const int ni = (int)n, mi = (int)m, di = (int)d, w = warm ? 1 : 0;
  switch (dp) {
    case 4: return small::launch<4>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    case 8: return small::launch<8>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    case 12: return small::launch<12>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    case 16: return small::launch<16>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    case 20: return small::launch<20>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    case 24: return small::launch<24>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    case 28: return small::launch<28>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    case 32: return small::launch<32>(X, Y, a, b, ni, mi, di, sched, iters, w, f, g, loss, st);
    default: return FLASHOT_ERR_INVALID_ARG;
  }
}

}  // namespace flashot
