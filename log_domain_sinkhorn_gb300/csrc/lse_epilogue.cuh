// lse_epilogue.cuh -- the online base-2 log-sum-exp of one row segment of a score tile,
// shared by the tensor-core LSE passes (tc_kernels.cu) and the persistent short solve
// (tc_solve_short.cu): each thread holds kN scores of one row in registers (a tcgen05.ld of
// the fp32 accumulator), adds the column biases and folds them into its running (max, sum).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace flashot {
namespace tc {

// Lazy rescaling of the online (max, sum), without a max pass: a chunk is exponentiated
// against the running max M of the earlier chunks, and its sum alone tells whether that was
// safe. When the sum is at most kLazyLimit = 2^64 (so every term is), the chunk is added as
// it is; otherwise (a score more than 64 above M, a sum that overflowed to inf, or the first
// chunk of a row segment, where M is at its floor) the chunk's max is taken, M is raised to
// it and the chunk's terms are taken again. The terms kept are at most 2^64 times the term
// of the row's running max, so S stays far inside fp32 range (below 2^64 times the number of
// columns), and M + log2 S is the same log-sum-exp; a term of the row's true max is never
// flushed, since M never exceeds it.
constexpr float kLazyLimit = 18446744073709551616.0f;  // 2^64

// kN (a multiple of 8) columns of one S-tile row: scores s2 = kappa * dot + bias and the online
// base-2 (max, sum) update. Pairs of scores go through packed fp32x2 instructions: per
// score half an FFMA2, half an FADD2, one SFU ex2 and half an FADD2.
// kLdg: read the biases through the read-only path (global memory) rather than as plain
// loads (biases staged in shared memory).
template <int kN, bool kLdg>
__device__ __forceinline__ void lse_chunk(float (&v)[kN], const float4* __restrict__ cb,
                                          float kappa, float& M, float& S) {
  const uint64_t k2 = ptx::pack2(kappa, kappa);
  uint64_t nm2 = ptx::pack2(-M, -M);
  // Four packed sums keep the dependency chains short.
  uint64_t s2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int j = 0; j < kN; j += 8) {
    const float4 b4 = kLdg ? __ldg(cb + j / 4) : cb[j / 4];
    const float4 b5 = kLdg ? __ldg(cb + j / 4 + 1) : cb[j / 4 + 1];
    ptx::unpack2(ptx::fma2(k2, ptx::pack2(v[j + 0], v[j + 1]), ptx::pack2(b4.x, b4.y)),
                 v[j + 0], v[j + 1]);
    ptx::unpack2(ptx::fma2(k2, ptx::pack2(v[j + 2], v[j + 3]), ptx::pack2(b4.z, b4.w)),
                 v[j + 2], v[j + 3]);
    ptx::unpack2(ptx::fma2(k2, ptx::pack2(v[j + 4], v[j + 5]), ptx::pack2(b5.x, b5.y)),
                 v[j + 4], v[j + 5]);
    ptx::unpack2(ptx::fma2(k2, ptx::pack2(v[j + 6], v[j + 7]), ptx::pack2(b5.z, b5.w)),
                 v[j + 6], v[j + 7]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float d0, d1;
      ptx::unpack2(ptx::add2(ptx::pack2(v[j + 2 * u], v[j + 2 * u + 1]), nm2), d0, d1);
      s2[u] = ptx::add2(s2[u], ptx::pack2(ex2(d0), ex2(d1)));
    }
  }
  uint64_t t2 = ptx::add2(ptx::add2(s2[0], s2[1]), ptx::add2(s2[2], s2[3]));
  float t0, t1;
  ptx::unpack2(t2, t0, t1);
  float t = t0 + t1;
  if (!(t <= kLazyLimit)) {  // rare: raise the max to the chunk's and take the sums again
    float m0 = M, m1 = M, m2 = M, m3 = M;
#pragma unroll
    for (int j = 0; j < kN; j += 8) {
      m0 = ptx::max3(m0, v[j + 0], v[j + 1]);
      m1 = ptx::max3(m1, v[j + 2], v[j + 3]);
      m2 = ptx::max3(m2, v[j + 4], v[j + 5]);
      m3 = ptx::max3(m3, v[j + 6], v[j + 7]);
    }
    const float mx = fmaxf(ptx::max3(m0, m1, m2), m3);
    S *= ex2(M - mx);
    M = mx;
    nm2 = ptx::pack2(-M, -M);
#pragma unroll
    for (int u = 0; u < 4; ++u) s2[u] = 0ull;
#pragma unroll
    for (int j = 0; j < kN; j += 8) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float d0, d1;
        ptx::unpack2(ptx::add2(ptx::pack2(v[j + 2 * u], v[j + 2 * u + 1]), nm2), d0, d1);
        s2[u] = ptx::add2(s2[u], ptx::pack2(ex2(d0), ex2(d1)));
      }
    }
    t2 = ptx::add2(ptx::add2(s2[0], s2[1]), ptx::add2(s2[2], s2[3]));
    ptx::unpack2(t2, t0, t1);
    t = t0 + t1;
  }
  S += t;
}

}  // namespace tc
}  // namespace flashot
