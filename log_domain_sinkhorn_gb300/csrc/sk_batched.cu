// sk_batched.cu -- batched Sinkhorn-Knopp projection of tiny matrices onto the Birkhoff
// polytope ("Fused & Furious: Sinkhorn Triton Kernels", section II: P = diag(u) M diag(v)
// with M = exp(H), u = 1 / (M v), v = 1 / (M^T u) alternated n_iter times from v = 1;
// section III: one n x n matrix per token, n = 4, n_iter = 20, batches up to 2^24).
//
// Each matrix is read once and written once; everything in between stays in registers.
// At n = 4 and 20 iterations the arithmetic, not HBM, bounds it: per matrix 672 FMA-pipe
// operations and 176 SFU operations (16 exp, 160 reciprocals) against 128 bytes of
// traffic, and the SFU runs reciprocals at 16 per clock per SM. The reciprocals are
// therefore taken in pairs (rcp_pairs), and even n use packed fp32x2 arithmetic to save
// issue slots. Layout of the kernel:
//  - one matrix per thread; a warp owns a chunk of 32 consecutive matrices;
//  - the chunk moves between HBM and registers through a per-warp shared-memory slab with
//    fully coalesced 16-byte loads and stores, the slab padded so that each thread's
//    16-byte reads of its own matrix are free of bank conflicts;
//  - the next chunk's loads are issued before the current chunk is computed, so loads
//    stay in flight during the arithmetic;
//  - a persistent grid (a multiple of the SM count) walks the chunks.
// exp(H) is taken in registers after subtracting the matrix's largest logit (diagonal
// scaling makes P invariant to a constant factor on M, and the shift keeps M <= 1).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "flashot.h"
#include "common.cuh"
#include "ptx.cuh"
#include "trace.h"

namespace flashot {
namespace sk {

constexpr int kMaxN = 8;

// Warps per CTA: 8, or 4 for n >= 7 (keeps the static slab under 48 KB).
template <int N>
constexpr int warps_for() {
  return N >= 7 ? 4 : 8;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// out[k] = 1 / s[k] with one SFU reciprocal per pair: 1/s0 = s1 / (s0 s1), 1/s1 = s0 / (s0 s1).
// The SFU delivers 16 reciprocals per clock per SM against 128 FP32 lanes, so with one
// reciprocal per sum it would bound the kernel; the pairing moves half of that work onto
// the FMA pipe. Exact in real arithmetic; valid while s0 s1 stays in the fp32 normal range.
template <int K>
__device__ __forceinline__ void rcp_pairs(const float (&s)[K], float (&out)[K]) {
#pragma unroll
  for (int k = 0; k + 1 < K; k += 2) {
    const float r = rcp_approx(s[k] * s[k + 1]);
    out[k] = s[k + 1] * r;
    out[k + 1] = s[k] * r;
  }
  if constexpr (K % 2 == 1) out[K - 1] = rcp_approx(s[K - 1]);
}

// Floats per matrix in the slab: a multiple of 4 whose quarter is odd, so that the 16-byte
// reads of 8 consecutive lanes fall into 8 different bank quads.
template <int N>
constexpr int slab_stride() {
  constexpr int s = (N * N + 3) / 4 * 4;
  return ((s / 4) % 2 == 0) ? s + 4 : s;
}

// n_iter Sinkhorn-Knopp alternations on M (registers, row-major), overwritten with P.
// Scalar form (any n).
template <int N>
__device__ __forceinline__ void sk_scalar(float (&m)[N * N], int n_iter) {
  float u[N], v[N], s[N];
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = 1.0f;
  for (int it = 0; it < n_iter; ++it) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      s[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < N; ++j) s[i] = fmaf(m[i * N + j], v[j], s[i]);
    }
    rcp_pairs<N>(s, u);
#pragma unroll
    for (int j = 0; j < N; ++j) {
      s[j] = 0.0f;
#pragma unroll
      for (int i = 0; i < N; ++i) s[j] = fmaf(m[i * N + j], u[i], s[j]);
    }
    rcp_pairs<N>(s, v);
  }
#pragma unroll
  for (int i = 0; i < N; ++i)
#pragma unroll
    for (int j = 0; j < N; ++j) m[i * N + j] = u[i] * m[i * N + j] * v[j];
}

// Packed form for even n: each row of M is held as n/2 fp32 pairs (m_i,2p, m_i,2p+1), and
// the products run two lanes per instruction (fma.rn.f32x2). Row sums accumulate their
// even and odd terms in the two lanes (added at the end); column sums come out in pairs
// (t_2p, t_2p+1) against the broadcast u_i.
template <int N>
__device__ __forceinline__ void sk_packed(float (&m)[N * N], int n_iter) {
  constexpr int H = N / 2;
  uint64_t MR[N][H];
#pragma unroll
  for (int i = 0; i < N; ++i)
#pragma unroll
    for (int p = 0; p < H; ++p) MR[i][p] = ptx::pack2(m[i * N + 2 * p], m[i * N + 2 * p + 1]);
  uint64_t VP[H];
#pragma unroll
  for (int p = 0; p < H; ++p) VP[p] = ptx::pack2(1.0f, 1.0f);
  float u[N];
  for (int it = 0; it < n_iter; ++it) {
    float s[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
      uint64_t acc = ptx::mul2(MR[i][0], VP[0]);
#pragma unroll
      for (int p = 1; p < H; ++p) acc = ptx::fma2(MR[i][p], VP[p], acc);
      float lo, hi;
      ptx::unpack2(acc, lo, hi);
      s[i] = lo + hi;
    }
    rcp_pairs<N>(s, u);
    uint64_t UU[N];
#pragma unroll
    for (int i = 0; i < N; ++i) UU[i] = ptx::pack2(u[i], u[i]);
#pragma unroll
    for (int p = 0; p < H; ++p) {
      uint64_t acc = ptx::mul2(MR[0][p], UU[0]);
#pragma unroll
      for (int i = 1; i < N; ++i) acc = ptx::fma2(MR[i][p], UU[i], acc);
      float t0, t1;
      ptx::unpack2(acc, t0, t1);
      const float r = rcp_approx(t0 * t1);
      VP[p] = ptx::pack2(t1 * r, t0 * r);
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint64_t ui = ptx::pack2(u[i], u[i]);
#pragma unroll
    for (int p = 0; p < H; ++p)
      ptx::unpack2(ptx::mul2(MR[i][p], ptx::mul2(ui, VP[p])), m[i * N + 2 * p],
                   m[i * N + 2 * p + 1]);
  }
}

template <int N>
__global__ void __launch_bounds__(warps_for<N>() * 32)
sk_batched_kernel(const float* H, int64_t B, int n_iter, float* P) {  // P may alias H
  constexpr int kWarps = warps_for<N>();
  constexpr int NN = N * N;
  constexpr int S = slab_stride<N>();
  constexpr bool kVec = (NN % 4) == 0;
  constexpr int kChunkFloats = 32 * NN;
  constexpr int kVecPerLane = kVec ? kChunkFloats / 4 / 32 : 1;  // float4 per lane per chunk
  __shared__ __align__(16) float slab[kWarps][32 * S];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* my = slab[warp];
  const int64_t n_chunks = (B + 31) / 32;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  int64_t c = (int64_t)blockIdx.x * kWarps + warp;

  // Registers holding the next chunk in flight (coalesced layout: lane-strided float4s).
  float4 buf[kVecPerLane];
  auto load_chunk = [&](int64_t ch) {
    const int64_t f0 = ch * kChunkFloats;
    const int64_t avail = (B - ch * 32) * NN;  // floats of this chunk that exist
    if constexpr (kVec) {
#pragma unroll
      for (int q = 0; q < kVecPerLane; ++q) {
        const int e = (q * 32 + lane) * 4;
        buf[q] = e < avail ? __ldcs(reinterpret_cast<const float4*>(H + f0 + e))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  if constexpr (kVec) {
    if (c < n_chunks) load_chunk(c);
  }
  for (; c < n_chunks; c += stride) {
    const int64_t f0 = c * kChunkFloats;
    const int64_t avail = std::min<int64_t>((B - c * 32) * NN, kChunkFloats);
    // ---- chunk -> slab ----------------------------------------------------------------
    if constexpr (kVec) {
#pragma unroll
      for (int q = 0; q < kVecPerLane; ++q) {
        const int e = (q * 32 + lane) * 4;  // float index in the chunk
        *reinterpret_cast<float4*>(my + (e / NN) * S + e % NN) = buf[q];
      }
      if (c + stride < n_chunks) load_chunk(c + stride);  // next chunk in flight
    } else {
      for (int e = lane; e < kChunkFloats; e += 32)
        my[(e / NN) * S + e % NN] = e < avail ? H[f0 + e] : 0.0f;
    }
    __syncwarp();
    // ---- one matrix per lane ------------------------------------------------------------
    float m[NN];
    if constexpr (kVec) {  // 16-byte slab accesses: conflict-free by the slab stride
      const float4* src = reinterpret_cast<const float4*>(my + lane * S);
#pragma unroll
      for (int q = 0; q < NN / 4; ++q) {
        const float4 t = src[q];
        m[4 * q] = t.x;
        m[4 * q + 1] = t.y;
        m[4 * q + 2] = t.z;
        m[4 * q + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < NN; ++k) m[k] = my[lane * S + k];
    }
    float hmax = m[0];
#pragma unroll
    for (int k = 1; k < NN; ++k) hmax = fmaxf(hmax, m[k]);
#pragma unroll
    for (int k = 0; k < NN; ++k) m[k] = ex2((m[k] - hmax) * kLog2e);
    if constexpr (N % 2 == 0) {
      sk_packed<N>(m, n_iter);
    } else {
      sk_scalar<N>(m, n_iter);
    }
    if constexpr (kVec) {
      float4* dst = reinterpret_cast<float4*>(my + lane * S);
#pragma unroll
      for (int q = 0; q < NN / 4; ++q)
        dst[q] = make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < NN; ++k) my[lane * S + k] = m[k];
    }
    __syncwarp();
    // ---- slab -> chunk ----------------------------------------------------------------
    if constexpr (kVec) {
#pragma unroll
      for (int q = 0; q < kVecPerLane; ++q) {
        const int e = (q * 32 + lane) * 4;
        if (e < avail)
          __stcs(reinterpret_cast<float4*>(P + f0 + e),
                 *reinterpret_cast<const float4*>(my + (e / NN) * S + e % NN));
      }
    } else {
      for (int e = lane; e < avail; e += 32) P[f0 + e] = my[(e / NN) * S + e % NN];
    }
    __syncwarp();
  }
}

template <int N>
int launch(const float* H, int64_t B, int n_iter, float* P, int sms, cudaStream_t st) {
  constexpr int kWarps = warps_for<N>();
  const int64_t n_chunks = (B + 31) / 32;
  const int64_t blocks_needed = (n_chunks + kWarps - 1) / kWarps;
  // Persistent: as many CTAs as fit on every SM at once (a multiple of the SM count).
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sk_batched_kernel<N>,
                                                    kWarps * 32, 0) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int64_t grid =
      std::max<int64_t>(1, std::min<int64_t>(blocks_needed, (int64_t)sms * per_sm));
  TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
  sk_batched_kernel<N><<<(unsigned)grid, kWarps * 32, 0, st>>>(H, B, n_iter, P);
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

}  // namespace sk
}  // namespace flashot

extern "C" int flashot_sinkhorn_knopp_batched(const float* H, int64_t B, int n, int n_iter,
                                              float* P, flashot_stream_t stream) {
  using namespace flashot::sk;
  if (B < 0 || n < 1 || n > kMaxN || n_iter < 1 || n_iter > (1 << 20))
    return FLASHOT_ERR_INVALID_ARG;
  if (B == 0) return FLASHOT_OK;
  if (B > (int64_t(1) << 40) / ((int64_t)n * n)) return FLASHOT_ERR_INVALID_ARG;
  for (const void* p : {static_cast<const void*>(H), static_cast<const void*>(P)}) {
    cudaPointerAttributes at;
    if (p == nullptr || cudaPointerGetAttributes(&at, p) != cudaSuccess ||
        (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)) {
      cudaGetLastError();
      return FLASHOT_ERR_INVALID_ARG;
    }
    if ((n * n) % 4 == 0 && (reinterpret_cast<uintptr_t>(p) & 15u) != 0)
      return FLASHOT_ERR_ALIGNMENT;
  }
  int dev = 0, maj = 0, mnr = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&mnr, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return FLASHOT_ERR_CUDA;
  }
  if (maj != 10 || mnr != 3) return FLASHOT_ERR_UNSUPPORTED_DEVICE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  switch (n) {
    case 1: return launch<1>(H, B, n_iter, P, sms, st);
    case 2: return launch<2>(H, B, n_iter, P, sms, st);
    case 3: return launch<3>(H, B, n_iter, P, sms, st);
    case 4: return launch<4>(H, B, n_iter, P, sms, st);
    case 5: return launch<5>(H, B, n_iter, P, sms, st);
    case 6: return launch<6>(H, B, n_iter, P, sms, st);
    case 7: return launch<7>(H, B, n_iter, P, sms, st);
    default: return launch<8>(H, B, n_iter, P, sms, st);
  }
}
