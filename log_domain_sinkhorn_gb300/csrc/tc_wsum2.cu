// tc_wsum2.cu -- bf16 tensor-core weighted-sum pass: transport application P V / P^T U,
// the barycentric gradient and the Hadamard-weighted transport (FlashSinkhorn: IO-Aware
// Entropic Optimal Transport on GPU, SAI replication review, "Summary" (i)-(ii)).
//
// For every (row tile i, column tile j) of 128 x 256:
//   S   = rows * cols^T                               tcgen05.mma M=128 N=256 -> TMEM[0:256)
//   w_ij = exp2(kappa S_ij + colBias_j + rowBias_i)   8 epilogue warps, fp32 + SFU ex2
//   O  += W * V^T-tile                                tcgen05.mma M=128 N=kKV -> TMEM[384:)
// W is written by the epilogue as bf16 into tensor memory (TMEM[256:384), two weights per
// 32-bit column) and is the A operand of the second MMA, read from there; V^T is loaded by
// TMA. Keeping W out of shared memory leaves room for four operand stages instead of two.
// The S MMA of tile j+1 overlaps the epilogue of tile j.
// The weights are plan entries (or a_i times softmax weights), all <= 1, so no running max.
//
// Work split: the (output-column group, row tile, column tile) triples are cut into
// gridDim.x contiguous ranges (stream-K), one per persistent CTA. A CTA writes, per row
// tile it touched, a partial O (128 x kKV) and partial (sum w, sum w S) per column half;
// wsum2_reduce_kernel adds the partials in a fixed order and finishes the output.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "flashot.h"
#include "common.cuh"
#include "pack_kernels.cuh"
#include "ptx.cuh"
#include "tc_api.h"
#include "tc_host.h"
#include "trace.h"

namespace flashot {
namespace tc2 {

constexpr int kBM = 128;
constexpr int kSBN = 256;                 // S tile width (MMA N)
constexpr int kChunk = 128 * 128;         // 128 rows x 128 bytes
constexpr int kThreads = 320;             // TMA warp, MMA warp, 8 epilogue warps
constexpr int kEpi = 256;
constexpr int kMaxStages = 4;
constexpr int kMaxOwners = 4;             // partial slots per (group, row tile)
constexpr int kSmemLimit = 232448;

struct __align__(128) W2Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t s_full, s_empty, w_full, w_empty, v_full, v_empty, o_full, o_empty, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void flag_error(W2Ctrl& ctl, unsigned* status) {
  atomicOr(status, kErrTimeout);
  ctl.abort_flag = 1;
}

// Parity of the n-th completion (0-based) of a barrier that is waited on by its consumer.
__device__ __forceinline__ uint32_t par(int64_t n) { return (uint32_t)(n & 1); }

template <int kKV>  // output columns per group: 64 or 128; 0 = Hadamard only
__global__ void __launch_bounds__(kThreads, 1)
wsum2_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
             const __grid_constant__ CUtensorMap mapV, const float* __restrict__ colBias,
             const float* __restrict__ rowBias, int64_t n_rows, int64_t row_tiles, int64_t NT,
             int64_t T, int kc_count, int n_st, float kappa, float* __restrict__ pO,
             float2* __restrict__ pW, int64_t ldp, unsigned* __restrict__ status) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ W2Ctrl ctl;
  constexpr bool kHad = (kKV == 0);
  constexpr uint32_t kBChunk = 2u * kChunk;            // 256 rows x 128 B
  constexpr uint32_t kStage = kChunk + kBChunk;        // A chunk + B chunk
  constexpr uint32_t kVChunk = (uint32_t)(kHad ? 1 : kKV) * 128u;  // kKV rows x 128 B
  constexpr uint32_t kVBytes = kHad ? 0u : 4u * kVChunk;
  constexpr uint32_t kTmemCols = 512;  // S at [0, 256), W at [256, 384), O at [384, 384 + kKV)
  constexpr uint32_t kTmemW = 256, kTmemO = 384;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = ptx::smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = dyn_smem + (base - raw);
  const uint32_t v_base = (uint32_t)n_st * kStage;
  const int64_t G = gridDim.x, cta = blockIdx.x;
  const int64_t t_begin = sk_begin(cta, T, G), t_end = sk_begin(cta + 1, T, G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < n_st; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    ptx::mbar_init(&ctl.s_full, 1);
    ptx::mbar_init(&ctl.s_empty, kEpi);
    ptx::mbar_init(&ctl.w_full, kEpi);
    ptx::mbar_init(&ctl.w_empty, 1);
    ptx::mbar_init(&ctl.v_full, 1);
    ptx::mbar_init(&ctl.v_empty, 1);
    ptx::mbar_init(&ctl.o_full, 1);
    ptx::mbar_init(&ctl.o_empty, kEpi);
    ptx::mbar_init(&ctl.mma_done, 1);
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&mapA);
    ptx::tma_prefetch_desc(&mapB);
    if constexpr (!kHad) ptx::tma_prefetch_desc(&mapV);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------- TMA producer -------------------------------------
      uint32_t stage = 0, ph = 0;
      int64_t issued = 0, v_issued = 0;
      bool ok = true;
      for (int64_t t = t_begin; ok && t < t_end; ++t) {
        const int64_t vr = t / NT;
        const int jt = (int)(t - vr * NT);
        const int64_t grp = vr / row_tiles, rt = vr - grp * row_tiles;
        for (int kc = 0; kc < kc_count; ++kc) {
          if (!ptx::mbar_wait(&ctl.empty[stage], ph ^ 1u)) { ok = false; break; }
          uint8_t* st = smem + (size_t)stage * kStage;
          ptx::mbar_arrive_expect_tx(&ctl.full[stage], kStage);
          ptx::tma_load_2d(&mapA, &ctl.full[stage], st, kc * 64, (int)(rt * kBM));
          ptx::tma_load_2d(&mapB, &ctl.full[stage], st + kChunk, kc * 64, jt * kSBN);
          ++issued;
          if (++stage == (uint32_t)n_st) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        if constexpr (!kHad) {
          if (!ptx::mbar_wait(&ctl.v_empty, par(v_issued) ^ 1u)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&ctl.v_full, kVBytes);
          for (int vc = 0; vc < 4; ++vc)
            ptx::tma_load_2d(&mapV, &ctl.v_full, smem + v_base + (size_t)vc * kVChunk,
                             jt * kSBN + vc * 64, (int)(grp * kKV));
          ++v_issued;
        }
      }
      if (!ok) flag_error(ctl, status);
      for (int s = 0; s < n_st; ++s) {
        const int64_t arms = issued / n_st + (s < issued % n_st ? 1 : 0);
        if (arms > 0) ptx::mbar_wait(&ctl.full[s], par(arms - 1));
      }
      if (v_issued > 0) ptx::mbar_wait(&ctl.v_full, par(v_issued - 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------- MMA issuer ----------------------------------------
      constexpr uint32_t idesc_s = ptx::make_idesc<true>(kBM, kSBN);
      constexpr uint32_t idesc_o = ptx::make_idesc<true>(kBM, kHad ? 64 : kKV);
      uint32_t stage = 0, ph = 0;
      int64_t s_uses = 0, w_uses = 0, segs = 0;
      bool ok = true;
      for (int64_t t = t_begin; ok && t < t_end;) {
        const int64_t vr = t / NT;
        const int64_t seg_end = min(t_end, (vr + 1) * NT);
        const int64_t L = seg_end - t;
        for (int64_t u = 0; ok && u <= L; ++u) {
          if (u < L) {  // S(u)
            if (!ptx::mbar_wait(&ctl.s_empty, par(s_uses) ^ 1u)) { ok = false; break; }
            ptx::tc_fence_after();
            for (int kc = 0; kc < kc_count; ++kc) {
              if (!ptx::mbar_wait(&ctl.full[stage], ph)) { ok = false; break; }
              ptx::tc_fence_after();
              const uint32_t st = base + stage * kStage;
              const uint64_t a_desc = ptx::sdesc_k128(st);
              const uint64_t b_desc = ptx::sdesc_k128(st + kChunk);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::umma<true>(tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc_s,
                                (kc | kk) != 0 ? 1u : 0u);
              ptx::umma_commit(&ctl.empty[stage]);
              if (++stage == (uint32_t)n_st) { stage = 0; ph ^= 1u; }
            }
            if (!ok) break;
            ptx::umma_commit(&ctl.s_full);
            ++s_uses;
          }
          if constexpr (!kHad) {
            if (u >= 1) {  // O(u-1) += W(u-1) V(u-1)
              if (u == 1 && !ptx::mbar_wait(&ctl.o_empty, par(segs) ^ 1u)) { ok = false; break; }
              if (!ptx::mbar_wait(&ctl.w_full, par(w_uses))) { ok = false; break; }
              if (!ptx::mbar_wait(&ctl.v_full, par(w_uses))) { ok = false; break; }
              ptx::tc_fence_after();
              const uint64_t v_desc = ptx::sdesc_k128(base + v_base);
              // K = 256 in steps of 16: W columns advance by 8 (two bf16 per column), the V
              // descriptor by 32 bytes inside each 64-element swizzled chunk.
#pragma unroll
              for (int vc = 0; vc < 4; ++vc) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  ptx::umma_ts_bf16(tmem + kTmemO, tmem + kTmemW + (uint32_t)(vc * 4 + kk) * 8u,
                                    v_desc + (uint64_t)(vc * (kVChunk >> 4) + 2 * kk), idesc_o,
                                    (u > 1 || vc > 0 || kk > 0) ? 1u : 0u);
              }
              ptx::umma_commit(&ctl.w_empty);
              ptx::umma_commit(&ctl.v_empty);
              ++w_uses;
            }
          }
        }
        if (!ok) break;
        if constexpr (!kHad) ptx::umma_commit(&ctl.o_full);
        ++segs;
        t = seg_end;
      }
      if (!ok) flag_error(ctl, status);
      ptx::umma_commit(&ctl.mma_done);
      ptx::mbar_wait(&ctl.mma_done, 0);
    }
  } else {
    // --------------------------------- epilogue ------------------------------------------
    // Warp w reads TMEM lane quarter (w % 4) and column half h = (w - 2) / 4 of each S tile.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int rloc = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int64_t s_uses = 0, w_uses = 0, segs = 0;
    bool ok = true;
    for (int64_t t = t_begin; ok && t < t_end;) {
      const int64_t vr = t / NT;
      const int64_t seg_end = min(t_end, (vr + 1) * NT);
      const int64_t grp = vr / row_tiles, rt = vr - grp * row_tiles;
      const int64_t row = rt * kBM + rloc;
      const float rb = row < n_rows ? rowBias[row] : neg_inf();
      const uint64_t rb2 = ptx::pack2(rb, rb), k2 = ptx::pack2(kappa, kappa);
      float sumw = 0.0f, had = 0.0f;
      for (int64_t tt = t; tt < seg_end; ++tt) {
        const int jt = (int)(tt - vr * NT);
        const float4* cb =
            reinterpret_cast<const float4*>(colBias + (int64_t)jt * kSBN + h * 128);
        if (!ptx::mbar_wait(&ctl.s_full, par(s_uses))) { ok = false; break; }
        ptx::tc_fence_after();
        float v[128];
        {
          float* v0 = v;
          ptx::tmem_ld_x64_sync(tmem + lane_base + h * 128, *reinterpret_cast<float(*)[64]>(v0));
          ptx::tmem_ld_x64_sync(tmem + lane_base + h * 128 + 64,
                                *reinterpret_cast<float(*)[64]>(v0 + 64));
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.s_empty);   // S may now be overwritten by the next tile
        ++s_uses;
        // Pairs of scores through packed fp32x2 instructions: w = 2^((kappa S + b_j) + b_i).
        // For the second MMA each pair is rounded to bf16 at once (wp[c] holds the weights
        // of K = 128h + 2c, 2c + 1), so the fp32 scores die as they are consumed.
        uint64_t sw2 = 0ull, hd2 = 0ull;
        uint32_t wp[kHad ? 1 : 64];
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
          const float4 b4 = __ldg(cb + j / 4);
          const uint64_t e01 = ptx::add2(ptx::fma2(k2, ptx::pack2(v[j + 0], v[j + 1]),
                                                   ptx::pack2(b4.x, b4.y)), rb2);
          const uint64_t e23 = ptx::add2(ptx::fma2(k2, ptx::pack2(v[j + 2], v[j + 3]),
                                                   ptx::pack2(b4.z, b4.w)), rb2);
          float x0, x1, x2, x3;
          ptx::unpack2(e01, x0, x1);
          ptx::unpack2(e23, x2, x3);
          const float w0 = ex2(x0), w1 = ex2(x1), w2 = ex2(x2), w3 = ex2(x3);
          const uint64_t w01 = ptx::pack2(w0, w1);
          const uint64_t w23 = ptx::pack2(w2, w3);
          if constexpr (kHad) {
            hd2 = ptx::fma2(w01, ptx::pack2(v[j + 0], v[j + 1]), hd2);
            hd2 = ptx::fma2(w23, ptx::pack2(v[j + 2], v[j + 3]), hd2);
          } else {
            __nv_bfloat162 h01 = __floats2bfloat162_rn(w0, w1);
            __nv_bfloat162 h23 = __floats2bfloat162_rn(w2, w3);
            wp[j / 2] = *reinterpret_cast<uint32_t*>(&h01);
            wp[j / 2 + 1] = *reinterpret_cast<uint32_t*>(&h23);
          }
          sw2 = ptx::add2(sw2, ptx::add2(w01, w23));
        }
        {
          float a0, a1;
          ptx::unpack2(sw2, a0, a1);
          sumw += a0 + a1;
          if constexpr (kHad) {
            ptx::unpack2(hd2, a0, a1);
            had += a0 + a1;
          }
        }
        if constexpr (!kHad) {
          // This warp's 128 weights are W row rloc, K = 128h .. 128h + 127: 64 columns of
          // bf16 pairs at TMEM column 256 + 64h.
          if (!ptx::mbar_wait(&ctl.w_empty, par(w_uses) ^ 1u)) { ok = false; break; }
          ptx::tc_fence_after();
          ptx::tmem_st_x64_sync(tmem + lane_base + kTmemW + (uint32_t)h * 64u, wp);
          ptx::tc_fence_before();
          ptx::mbar_arrive(&ctl.w_full);
          ++w_uses;
        }
      }
      if (!ok) break;
      const int64_t slot = cta - sk_owner(vr * NT, T, G);
      const int64_t prow = vr * kBM + rloc;  // row of the partial buffers
      if constexpr (!kHad) {
        if (!ptx::mbar_wait(&ctl.o_full, par(segs))) { ok = false; break; }
        ptx::tc_fence_after();
        float* dst = pO + ((size_t)slot * ldp + (size_t)prow) * kKV + h * (kKV / 2);
#pragma unroll 1
        for (int c = 0; c < kKV / 64; ++c) {
          float o[32];
          ptx::tmem_ld_x32_sync(tmem + lane_base + kTmemO + h * (kKV / 2) + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.o_empty);
      }
      pW[((size_t)(2 * slot + h)) * ldp + (size_t)prow] = make_float2(sumw, had);
      ++segs;
      t = seg_end;
    }
    if (!ok) flag_error(ctl, status);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Adds the partial slots of one (group, row tile) in a fixed order and finishes the output:
// apply: out = O; gradient: out = 2 a (x - O / sum w); Hadamard: out = sum w S.
template <int kMode>
__global__ void wsum2_reduce_kernel(const float* __restrict__ pO, const float2* __restrict__ pW,
                                    int64_t ldp, int kKV, int64_t row_tiles, int64_t NT,
                                    int64_t T, int64_t G, int64_t n_rows,
                                    const float* __restrict__ rowW, const float* __restrict__ X,
                                    int64_t d, int64_t k, float* __restrict__ out, int64_t ldo) {
  const int64_t per_row = (kMode == kWsumHadamard) ? 1 : kKV;
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (idx >= ldp * per_row) return;
  const int64_t prow = idx / per_row;
  const int64_t o = idx - prow * per_row;
  const int64_t vr = prow / kBM;
  const int64_t grp = vr / row_tiles;
  const int64_t row = (vr - grp * row_tiles) * kBM + (prow - vr * kBM);
  if (row >= n_rows) return;
  const int slots = (int)(sk_owner((vr + 1) * NT - 1, T, G) - sk_owner(vr * NT, T, G) + 1);
  if constexpr (kMode == kWsumHadamard) {
    float hsum = 0.0f;
    for (int s = 0; s < slots; ++s)
      hsum += pW[(size_t)(2 * s) * ldp + prow].y + pW[(size_t)(2 * s + 1) * ldp + prow].y;
    out[row] = hsum;
  } else {
    float acc = 0.0f;
    for (int s = 0; s < slots; ++s) acc += pO[((size_t)s * ldp + prow) * kKV + o];
    const int64_t oo = grp * kKV + o;
    if constexpr (kMode == kWsumGrad) {
      if (oo >= d) return;
      float sumw = 0.0f;
      for (int s = 0; s < slots; ++s)
        sumw += pW[(size_t)(2 * s) * ldp + prow].x + pW[(size_t)(2 * s + 1) * ldp + prow].x;
      const float a = rowW[row];
      out[row * ldo + oo] =
          (a > 0.0f && sumw > 0.0f) ? 2.0f * a * (X[row * d + oo] - acc / sumw) : 0.0f;
    } else {
      if (oo < k) out[row * ldo + oo] = acc;
    }
  }
}

template <int kKV>
static int launch(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mV,
                  const float* colBias, const float* rowBias, int64_t n_rows, int64_t row_tiles,
                  int64_t NT, int64_t T, int64_t G, int kc, float kappa, float* pO, float2* pW,
                  int64_t ldp, unsigned* status, cudaStream_t st) {
  const int fixed = (kKV == 0) ? 0 : 4 * kKV * 128;  // the V^T tile
  const int budget = kSmemLimit - (int)sizeof(W2Ctrl) - 1024 - fixed;
  const int n_st = std::min(kMaxStages, budget / (3 * kChunk));
  if (n_st < 2) return FLASHOT_ERR_INVALID_ARG;
  const int dyn = n_st * 3 * kChunk + fixed + 1024;
  auto kern = wsum2_kernel<kKV>;
  int rc = tc::set_smem(kern, dyn);
  if (rc != FLASHOT_OK) return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_WSUM, st);
    kern<<<(unsigned)G, kThreads, dyn, st>>>(mA, mB, mV, colBias, rowBias, n_rows, row_tiles, NT,
                                            T, kc, n_st, kappa, pO, pW, ldp, status);
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

}  // namespace tc2

size_t tc_wsum2_scratch_bytes(int64_t rows_pad, int64_t k_or_d) {
  // pO: kMaxOwners slots x rows_pad x (groups x kKV) floats, where groups x kKV is 64 for
  // k <= 64 and round_up(k, 128) otherwise; pW: 2 kMaxOwners slots x groups x rows_pad
  // float2, groups <= kk / 64.
  const int64_t kk = k_or_d <= 64 ? 64 : (k_or_d + 127) / 128 * 128;
  return (size_t)tc2::kMaxOwners * rows_pad * kk * sizeof(float) +
         (size_t)2 * tc2::kMaxOwners * (kk / 64) * rows_pad * sizeof(float2) + 1024;
}

int tc_wsum2_pass(int mode, const void* rowQ, const void* colQ, const float* colBias,
                  const float* rowBias, int64_t n_rows, int64_t n_cols, int64_t rows_pad,
                  int64_t cols_pad, int64_t d, int64_t dpt, float kappa, const float* V,
                  int64_t ldv, int64_t k, void* vtq, void* scratch, const float* rowW,
                  const float* X, float* out, int64_t ldo, int sms, unsigned* status,
                  cudaStream_t st) {
  using namespace tc2;
  const int kc = (int)(dpt * 2 / 128);
  if (rows_pad % kBM != 0 || cols_pad % kSBN != 0) return FLASHOT_ERR_INVALID_ARG;
  const int64_t row_tiles = rows_pad / kBM, NT = cols_pad / kSBN;
  const bool had = (mode == kWsumHadamard);
  if (!had && ldv != k) return FLASHOT_ERR_INVALID_ARG;
  const int kv = had ? 0 : (k <= 64 ? 64 : 128);
  const int64_t groups = had ? 1 : (k + kv - 1) / kv;
  const int64_t vrows = groups * row_tiles;
  const int64_t T = vrows * NT;
  const int64_t G = tc::choose_grid(vrows, NT, sms, kMaxOwners);
  const int64_t ldp = vrows * kBM;
  float* pO = static_cast<float*>(scratch);
  const size_t po_bytes = (size_t)kMaxOwners * ldp * (had ? 0 : kv) * sizeof(float);
  float2* pW = reinterpret_cast<float2*>(static_cast<char*>(scratch) + (po_bytes + 255) / 256 * 256);
  CUtensorMap mA, mB, mV;
  int rc = tc::make_map(&mA, rowQ, rows_pad, dpt, true);
  if (rc == FLASHOT_OK) rc = tc::make_map_rows(&mB, colQ, cols_pad, dpt, true, kSBN);
  if (rc != FLASHOT_OK) return rc;
  if (!had) {
    const int64_t out_rows_pad = groups * kv;
    {
      dim3 blk(32, 8), grd((unsigned)(cols_pad / 32), (unsigned)(out_rows_pad / 32));
      TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      pack_transpose_kernel<PackKind::BF16><<<grd, blk, 0, st>>>(V, vtq, n_cols, k, cols_pad,
                                                                 out_rows_pad);
    }
    if (cudaGetLastError() != cudaSuccess) return FLASHOT_ERR_CUDA;
    rc = tc::make_map_rows(&mV, vtq, out_rows_pad, cols_pad, true, kv);
    if (rc != FLASHOT_OK) return rc;
  } else {
    mV = mB;  // unused
  }
  if (had)
    rc = launch<0>(mA, mB, mV, colBias, rowBias, n_rows, row_tiles, NT, T, G, kc, kappa, pO, pW,
                   ldp, status, st);
  else if (kv == 64)
    rc = launch<64>(mA, mB, mV, colBias, rowBias, n_rows, row_tiles, NT, T, G, kc, kappa, pO, pW,
                    ldp, status, st);
  else
    rc = launch<128>(mA, mB, mV, colBias, rowBias, n_rows, row_tiles, NT, T, G, kc, kappa, pO,
                     pW, ldp, status, st);
  if (rc != FLASHOT_OK) return rc;
  const int64_t total = ldp * (had ? 1 : kv);
  const unsigned blocks = (unsigned)((total + 255) / 256);
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
    if (mode == kWsumGrad)
      wsum2_reduce_kernel<kWsumGrad><<<blocks, 256, 0, st>>>(pO, pW, ldp, kv, row_tiles, NT, T, G,
                                                            n_rows, rowW, X, d, k, out, ldo);
    else if (mode == kWsumApply)
      wsum2_reduce_kernel<kWsumApply><<<blocks, 256, 0, st>>>(pO, pW, ldp, kv, row_tiles, NT, T,
                                                             G, n_rows, rowW, X, d, k, out, ldo);
    else
      wsum2_reduce_kernel<kWsumHadamard><<<blocks, 256, 0, st>>>(pO, pW, ldp, 1, row_tiles, NT, T,
                                                                G, n_rows, rowW, X, d, k, out, ldo);
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

}  // namespace flashot
