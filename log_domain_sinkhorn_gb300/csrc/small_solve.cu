// small_solve.cu -- the whole alternating solve in one launch, for small fp32 problems.
//
// When both clouds, all potentials and the score biases fit in one SM's shared memory, the
// iteration is bound by launch latency (four launches per iteration on the streaming path).
// Here one thread-block cluster of kCluster CTAs runs every stage and iteration inside a
// single kernel (FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract: the
// f- and g-updates as row-wise log-sum-exps; arithmetic identical to the CUDA-core path):
//  - every CTA keeps X, Y, |x|^2, |y|^2, log2 a, log2 b and full copies of f and g;
//  - for an f-update each CTA computes its slice of rows, each row split over kTPR threads
//    whose (max, sum) pairs are merged with warp shuffles, and stores its f values into the
//    shared memory of every CTA of the cluster (DSMEM);
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

constexpr int kCluster = 8;
constexpr int kThreads = 512;
constexpr int kTPR = 4;  // threads per row

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

// One half-step for the rows [r0, r1) of the side P against the nq points of the other
// side Q, whose column biases cq fold in their potential, norm and log-weight:
// out_i = nrmp_i - eps ln2 LSE2_j(kappa <p_i, q_j> + cq_j), stored into every CTA.
template <int DP>
__device__ __forceinline__ void half_step(const float* __restrict__ P, const float* __restrict__ Q,
                                          int nq, const float* __restrict__ cq,
                                          const float* __restrict__ nrmp, int r0, int r1,
                                          float kappa, float eps, float* out) {
  const int tid = threadIdx.x;
  for (int base = r0; base < r1; base += kThreads / kTPR) {
    const int i = base + tid / kTPR;
    const int part = tid % kTPR;
    float M = kNegBig, S = 0.0f;
    if (i < r1) {
      float x[DP];
#pragma unroll
      for (int c = 0; c < DP; ++c) x[c] = P[i * DP + c];
      for (int j0 = part * 8; j0 < nq; j0 += kTPR * 8) {
        float s[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + u;
          float dot = 0.0f;
          if (j < nq) {
#pragma unroll
            for (int c = 0; c < DP; ++c) dot = fmaf(x[c], Q[j * DP + c], dot);
            s[u] = fmaf(kappa, dot, cq[j]);
          } else {
            s[u] = neg_inf();
          }
        }
        float mx = s[0];
#pragma unroll
        for (int u = 1; u < 8; ++u) mx = fmaxf(mx, s[u]);
        if (mx > M) {
          S *= ex2(M - mx);
          M = mx;
        }
        float acc = 0.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += ex2(s[u] - M);
        S += acc;
      }
    }
    // Merge the kTPR partial (max, sum) pairs of a row (adjacent lanes).
#pragma unroll
    for (int o = 1; o < kTPR; o <<= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
      const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const float Mn = fmaxf(M, M2);
      S = S * ex2(M - Mn) + S2 * ex2(M2 - Mn);
      M = Mn;
    }
    if (i < r1 && part == 0) {
      const float L = M + log2f(S);
      const float v = nrmp[i] - eps * kLn2 * L;
      for (uint32_t r = 0; r < (uint32_t)kCluster; ++r) st_cluster(out + i, r, v);
    }
  }
}

template <int DP>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
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

  const int fr0 = (int)(((int64_t)n * rank) / kCluster), fr1 = (int)(((int64_t)n * (rank + 1)) / kCluster);
  const int gr0 = (int)(((int64_t)m * rank) / kCluster), gr1 = (int)(((int64_t)m * (rank + 1)) / kCluster);
  for (int s = 0; s < sched.n_stages; ++s) {
    const float eps = sched.eps[s];
    const float kappa = 2.0f * kLog2e / eps;
    const float inv = kLog2e / eps;
    for (int it = 0; it < iters; ++it) {
      // f-update: bias of the columns (Y side) from g
      for (int j = tid; j < m; j += kThreads) cb[j] = (ga[j] - be[j]) * inv + lb[j];
      __syncthreads();
      half_step<DP>(Xs, Ys, m, cb, al, fr0, fr1, kappa, eps, fa);
      cluster_sync();
      // g-update: bias of the columns (X side) from f
      for (int i = tid; i < n; i += kThreads) cb[i] = (fa[i] - al[i]) * inv + la[i];
      __syncthreads();
      half_step<DP>(Ys, Xs, n, cb, be, gr0, gr1, kappa, eps, ga);
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
  return (size_t)((n + m) * dp + 5 * (n + m) + (n > m ? n : m)) * sizeof(float);
}

template <int DP>
int launch(const float* X, const float* Y, const float* a, const float* b, int n, int m, int d,
           const EpsSchedule& sched, int iters, int warm, float* f, float* g, double* loss,
           cudaStream_t st) {
  const size_t bytes = smem_bytes(n, m, DP);
  cudaError_t e = cudaFuncSetAttribute(small_solve_kernel<DP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return FLASHOT_ERR_CUDA;
  {
    TraceScope ts_(FLASHOT_KERNEL_LSE, st);
    small_solve_kernel<DP><<<kCluster, kThreads, bytes, st>>>(X, Y, a, b, n, m, d, sched, iters,
                                                              warm, f, g, loss);
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

}  // namespace small

bool small_solve_eligible(int64_t n, int64_t m, int64_t dp, int n_stages) {
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
