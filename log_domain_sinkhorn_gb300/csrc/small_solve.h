// small_solve.h -- single-launch cluster solver for small fp32 problems (small_solve.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace flashot {

constexpr int kSmallMaxStages = 32;

// The eps schedule passed by value to the kernel.
struct EpsSchedule {
  float eps[kSmallMaxStages];
  int n_stages;
};

// True when the whole problem (both clouds padded to dp, potentials, norms, log-weights and
// biases) fits in one SM's shared memory and the problem is small enough that launch
// latency, not arithmetic, bounds the streaming path (n * m <= 2^20).
bool small_solve_eligible(int64_t n, int64_t m, int64_t dp, int n_stages);

// Runs all stages and iterations of the alternating solve in one launch of one cluster
// (16 CTAs where possible, else 8); writes f, g and (if loss != NULL) the dual loss. a / b NULL = uniform.
int small_solve(const float* X, const float* Y, const float* a, const float* b, int64_t n,
                int64_t m, int64_t d, int64_t dp, const float* eps_sched, int n_stages,
                int iters, bool warm, float* f, float* g, double* loss, cudaStream_t st);

}  // namespace flashot
