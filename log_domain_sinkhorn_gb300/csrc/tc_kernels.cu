// tc_kernels.cu -- tcgen05 (5th-generation tensor core) streaming passes for sm_103a.
//
// The half-step of stabilized log-domain Sinkhorn is a row-wise log-sum-exp of biased
// dot-product scores (FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract;
// SAI replication review, "Summary": tiles of Q and K streamed through on-chip memory,
// scores formed on the fly, running row-wise LSE statistics, only potentials written
// back). On sm_103a the score tile S = P_rows * Q_cols^T is a dense contraction, so it
// runs on tcgen05.mma with the 128 x 128 fp32 accumulator in Tensor Memory:
//
//   warp 0      TMA producer: row tile (resident when it fits) + column-tile K-chunks
//               into a ring of shared-memory stages (128-byte swizzle);
//   warp 1      MMA issuer: one elected thread issues tcgen05.mma into one of two TMEM
//               accumulators and tcgen05.commit's stage / accumulator barriers;
//   warps 2..5  epilogue: tcgen05.ld the S tile (one row per thread), add the column
//               bias, online base-2 max / sum-exp (MUFU ex2), while the MMA fills the
//               other accumulator.
//
// Work split: the (row tile, column tile) pairs are linearised row-tile-major and cut
// into gridDim.x contiguous ranges, one per persistent CTA ("stream-K"), so every SM
// gets the same number of tiles to within one. A CTA emits one (max, sum) partial per
// row tile it touches; lse_combine_kernel merges them (at most kMaxSplits per row).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cstdlib>

#include "flashot.h"
#include "common.cuh"
#include "fma_kernels.cuh"  // wsum_split_reduce_kernel
#include "lse_epilogue.cuh"
#include "pack_kernels.cuh"
#include "ptx.cuh"
#include "tc_api.h"
#include "tc_host.h"
#include "trace.h"

namespace flashot {
namespace tc {

constexpr int kBM = 128;                 // rows per tile (MMA M)
constexpr int kBN = 128;                 // columns per tile of the weighted-sum pass (MMA N)
constexpr int kLseBN = 256;              // columns per tile of the LSE pass (MMA N)
constexpr int kChunk = 128 * 128;        // bytes of one 128-row x 128-byte K-chunk box
constexpr int kThreads = 192;            // weighted-sum pass: 6 warps
constexpr int kLseThreads = 320;         // LSE pass: TMA warp, MMA warp, 8 epilogue warps
constexpr int kLseEpiThreads = 256;
constexpr int kMaxStages = 8;
constexpr uint32_t kLseTmemCols = 512;   // two 256-column fp32 accumulators
constexpr int kSmemLimit = 232448;       // 227 KB per block (opt-in maximum)

struct __align__(128) Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t a_full[2];   // resident row tile, up to two buffers (a_bufs)
  uint64_t a_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void flag_error(Ctrl& ctl, unsigned* status) {
  atomicOr(status, kErrTimeout);
  ctl.abort_flag = 1;
}

// ---------------------------------------------------------------------------------------
// LSE pass: partial[slot * ld + row] = (max_j s2_ij, sum_j 2^(s2_ij - max)) over the
// column tiles of this CTA's range, s2_ij = kappa <p_i, q_j> + colBias_j.
// Tiles are 128 rows x 256 columns (tcgen05.mma M = 128, N = 256).
// kARes: the row tile (all K-chunks) stays in shared memory for a whole segment, and each
// stage holds one 256-row x 128-byte K-chunk of the column cloud; otherwise each stage
// holds a K-chunk of both.
// ---------------------------------------------------------------------------------------
// kStageBias: the epilogue copies each tile's column biases into shared memory one tile
// ahead (cp.async). Used for short contractions, where the epilogue bounds a tile and a
// direct read would wait on L2 (L1 is small next to the operand stages); long contractions
// keep all shared memory for operand stages and read the biases directly.
template <bool kBF16, bool kARes, bool kStageBias>
__global__ void __launch_bounds__(kLseThreads, 1)
lse_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
              const float* __restrict__ colBias, int64_t n_rows, int64_t NT, int64_t T,
              int kc_count, int stages, int a_bufs, float kappa, float2* __restrict__ partial,
              int64_t ld, unsigned* __restrict__ status) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctrl ctl;
  constexpr int kGroups = 2;               // partial slots per CTA and row tile
  constexpr int kCols = kLseBN / kGroups;  // columns of a tile per epilogue warp (direct biases)
  // kStageBias: column biases of the warp's current and next tile (all 256 columns).
  __shared__ __align__(16) float bias_s[kStageBias ? kLseEpiThreads / 32 : 1][2]
                                       [kStageBias ? kLseBN : 4];
  constexpr int kElems = kBF16 ? 64 : 32;  // elements per 128-byte K-chunk row
  constexpr uint32_t kBChunk = 2u * kChunk;  // 256 rows x 128 bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = ptx::smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = dyn_smem + (base - raw);
  const uint32_t a_bytes = kARes ? (uint32_t)kc_count * kChunk : 0u;
  const uint32_t stage_bytes = kARes ? kBChunk : kChunk + kBChunk;
  const uint32_t b_off = kARes ? 0u : (uint32_t)kChunk;  // B chunk offset within a stage
  const int64_t G = gridDim.x, cta = blockIdx.x;
  const int64_t t_begin = sk_begin(cta, T, G), t_end = sk_begin(cta + 1, T, G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl.acc_full[b], 1);
      // staged biases: the four warps of one tile parity read a tile; otherwise all eight
      ptx::mbar_init(&ctl.acc_empty[b], kStageBias ? kLseEpiThreads / 2 : kLseEpiThreads);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl.a_full[b], 1);
      ptx::mbar_init(&ctl.a_empty[b], 1);
    }
    ptx::mbar_init(&ctl.mma_done, 1);
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&mapA);
    ptx::tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, kLseTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  // Short contractions run as programmatic dependents of the previous combine: let the
  // next kernel (this pass's combine) get ready now. The operand loads and MMAs below read
  // only the packed clouds, which no kernel of the solve writes; the epilogue waits for
  // the previous kernel before it reads the biases that kernel wrote.
  if constexpr (kStageBias) griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------- TMA producer -------------------------------------
      uint32_t stage = 0, ph = 0;
      int64_t issued = 0, segs = 0;
      bool ok = true;
      for (int64_t t = t_begin; ok && t < t_end;) {
        const int64_t rt = t / NT;
        const int64_t seg_end = min(t_end, (rt + 1) * NT);
        if constexpr (kARes) {
          // segment s uses row-tile buffer s % a_bufs (its (s / a_bufs)-th use): with two
          // buffers the next segment's rows load while the current one is still in use
          const int ab = (int)(segs % a_bufs);
          const uint32_t use = (uint32_t)(segs / a_bufs);
          if (!ptx::mbar_wait(&ctl.a_empty[ab], (use & 1u) ^ 1u)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&ctl.a_full[ab], a_bytes);
          for (int kc = 0; kc < kc_count; ++kc)
            ptx::tma_load_2d(&mapA, &ctl.a_full[ab],
                             smem + (size_t)ab * a_bytes + (size_t)kc * kChunk, kc * kElems,
                             (int)(rt * kBM));
          ++segs;
        }
        for (int64_t tt = t; ok && tt < seg_end; ++tt) {
          const int jt = (int)(tt - rt * NT);
          for (int kc = 0; kc < kc_count; ++kc) {
            if (!ptx::mbar_wait(&ctl.empty[stage], ph ^ 1u)) { ok = false; break; }
            uint8_t* st = smem + (size_t)a_bufs * a_bytes + (size_t)stage * stage_bytes;
            ptx::mbar_arrive_expect_tx(&ctl.full[stage], stage_bytes);
            if constexpr (!kARes)
              ptx::tma_load_2d(&mapA, &ctl.full[stage], st, kc * kElems, (int)(rt * kBM));
            ptx::tma_load_2d(&mapB, &ctl.full[stage], st + b_off, kc * kElems, jt * kLseBN);
            ++issued;
            if (++stage == (uint32_t)stages) { stage = 0; ph ^= 1u; }
          }
        }
        t = seg_end;
      }
      if (!ok) flag_error(ctl, status);
      // Drain: every copy issued must have landed before the CTA may exit.
      for (int s = 0; s < stages; ++s) {
        const int64_t arms = issued / stages + (s < issued % stages ? 1 : 0);
        if (arms > 0) ptx::mbar_wait(&ctl.full[s], (uint32_t)((arms - 1) & 1));
      }
      for (int b = 0; b < a_bufs && b < 2; ++b) {
        const int64_t uses = segs / a_bufs + (b < segs % a_bufs ? 1 : 0);
        if (uses > 0) ptx::mbar_wait(&ctl.a_full[b], (uint32_t)((uses - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------- MMA issuer ----------------------------------------
      constexpr uint32_t idesc = ptx::make_idesc<kBF16>(kBM, kLseBN);
      uint32_t stage = 0, ph = 0, ab = 0, acc_ph = 0;
      int64_t segs = 0;
      bool ok = true;
      for (int64_t t = t_begin; ok && t < t_end;) {
        const int64_t rt = t / NT;
        const int64_t seg_end = min(t_end, (rt + 1) * NT);
        const int abuf = kARes ? (int)(segs % a_bufs) : 0;
        if constexpr (kARes) {
          if (!ptx::mbar_wait(&ctl.a_full[abuf], (uint32_t)((segs / a_bufs) & 1))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
        }
        for (int64_t tt = t; ok && tt < seg_end; ++tt) {
          if (!ptx::mbar_wait(&ctl.acc_empty[ab], acc_ph ^ 1u)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem + ab * kLseBN;
          for (int kc = 0; kc < kc_count; ++kc) {
            if (!ptx::mbar_wait(&ctl.full[stage], ph)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t st = base + (uint32_t)a_bufs * a_bytes + stage * stage_bytes;
            const uint32_t a_addr =
                kARes ? base + (uint32_t)abuf * a_bytes + (uint32_t)kc * kChunk : st;
            const uint64_t a_desc = ptx::sdesc_k128(a_addr);
            const uint64_t b_desc = ptx::sdesc_k128(st + b_off);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K advance: 32 bytes = 2 in the address field
              ptx::umma<kBF16>(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                               (kc | kk) != 0 ? 1u : 0u);
            ptx::umma_commit(&ctl.empty[stage]);
            if (++stage == (uint32_t)stages) { stage = 0; ph ^= 1u; }
          }
          if (!ok) break;
          ptx::umma_commit(&ctl.acc_full[ab]);
          if (++ab == 2) { ab = 0; acc_ph ^= 1u; }
        }
        if constexpr (kARes) ptx::umma_commit(&ctl.a_empty[abuf]);
        ++segs;
        t = seg_end;
      }
      if (!ok) flag_error(ctl, status);
      // Every MMA issued must have retired before Tensor Memory is released.
      ptx::umma_commit(&ctl.mma_done);
      ptx::mbar_wait(&ctl.mma_done, 0);
    }
  } else {
    // --------------------------------- epilogue ------------------------------------------
    // Warps 2..9: warp w reads TMEM lane quarter (w % 4) (rows 32q .. 32q+31) and column
    // half h = (w - 2) / 4 of every 256-column tile; each (row, half) keeps its own online
    // (max, sum) and becomes its own partial slot, merged later by the combine kernel.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    if constexpr (kStageBias) {
    // Short contractions: the two warps of a sub-partition take alternate tiles (warp of
    // parity p = h reads every tile k = p, p + 2, ... of the CTA's range, all 256 columns,
    // from accumulator p), so their SFU bursts and their loads and max phases interleave
    // instead of coinciding. Each (row, parity) keeps its own online (max, sum) and becomes
    // its own partial slot.
    const int par = h;
    uint32_t acc_ph = 0;
    bool ok = true;
    // The warp's 256 biases of a tile (1 KB, 32 per lane) are copied global -> shared with
    // cp.async one own tile ahead into one of two slots.
    float (*bslot)[kStageBias ? kLseBN : 4] = bias_s[kStageBias ? warp - 2 : 0];
    auto stage_bias = [&](int64_t tile, int slot) {
      const float* src = colBias + (tile % NT) * kLseBN + lane * 4;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                       ptx::smem_u32(&bslot[slot][lane * 4])),
                   "l"(src)
                   : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                       ptx::smem_u32(&bslot[slot][128 + lane * 4])),
                   "l"(src + 128)
                   : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    int bs = 0;
    griddep_wait();  // the biases (and the partial buffer) belong to the previous kernel
    if (t_begin + par < t_end) stage_bias(t_begin + par, 0);
    for (int64_t t = t_begin; ok && t < t_end;) {
      const int64_t rt = t / NT;
      const int64_t seg_end = min(t_end, (rt + 1) * NT);
      float M = kNegBig, S = 0.0f;
      // this warp's first tile of the segment: (tt - t_begin) % 2 == par
      for (int64_t tt = t + (((t - t_begin) & 1) != par ? 1 : 0); tt < seg_end; tt += 2) {
        if (tt + 2 < t_end) {
          stage_bias(tt + 2, bs ^ 1);
          asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
          asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncwarp();
        const float4* cb = reinterpret_cast<const float4*>(bslot[bs]);
        if (!ptx::mbar_wait(&ctl.acc_full[par], acc_ph)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t taddr = tmem + lane_base + (uint32_t)par * kLseBN;
        float v[64];
#pragma unroll 1
        for (int c = 0; c < 3; ++c) {
          ptx::tmem_ld_x64_sync(taddr + c * 64, v);
          lse_chunk<64, false>(v, cb + c * 16, kappa, M, S);
        }
        ptx::tmem_ld_x64_sync(taddr + 192, v);
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.acc_empty[par]);   // this warp's part of the tile is read
        acc_ph ^= 1u;
        lse_chunk<64, false>(v, cb + 48, kappa, M, S);
        __syncwarp();  // every lane is done with bslot[bs] before it is refilled
        bs ^= 1;
      }
      if (!ok) break;
      const int64_t row = rt * kBM + q * 32 + lane;
      const int64_t slot = kGroups * (cta - sk_owner(rt * NT, T, G)) + par;
      if (row < n_rows) partial[slot * ld + row] = make_float2(M, S);
      t = seg_end;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy outlives the CTA
    if (!ok) flag_error(ctl, status);
    } else {
    uint32_t ab = 0, acc_ph = 0;
    bool ok = true;
    if (t_begin < t_end && lane < 4)   // 512 B of bias per half-tile: one line per lane
      ptx::prefetch_l1(colBias + (t_begin % NT) * kLseBN + h * 128 + lane * 32);
    for (int64_t t = t_begin; ok && t < t_end;) {
      const int64_t rt = t / NT;
      const int64_t seg_end = min(t_end, (rt + 1) * NT);
      float M = kNegBig, S = 0.0f;
      for (int64_t tt = t; tt < seg_end; ++tt) {
        const float4* cb =
            reinterpret_cast<const float4*>(colBias + (tt % NT) * kLseBN + h * 128);
        if (tt + 1 < t_end && lane < 4)
          ptx::prefetch_l1(colBias + ((tt + 1) % NT) * kLseBN + h * 128 + lane * 32);
        if (!ptx::mbar_wait(&ctl.acc_full[ab], acc_ph)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t taddr = tmem + lane_base + ab * kLseBN + h * 128;
        float v[64];
        ptx::tmem_ld_x64_sync(taddr, v);
        lse_chunk<64, true>(v, cb, kappa, M, S);
        ptx::tmem_ld_x64_sync(taddr + 64, v);
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.acc_empty[ab]);   // this warp's part of the tile is read
        if (++ab == 2) { ab = 0; acc_ph ^= 1u; }
        lse_chunk<64, true>(v, cb + 16, kappa, M, S);
      }
      if (!ok) break;
      const int64_t row = rt * kBM + q * 32 + lane;
      const int64_t slot = kGroups * (cta - sk_owner(rt * NT, T, G)) + h;
      if (row < n_rows) partial[slot * ld + row] = make_float2(M, S);
      t = seg_end;
    }
    if (!ok) flag_error(ctl, status);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kLseTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// LSE pass on CTA pairs (long contractions): two CTAs of a cluster run one cta_group::2 MMA
// per K step, M = 256 rows (128 from each CTA's resident or streamed row tile) x N = 256
// columns, each CTA holding the K-chunk of 128 of the 256 column points. Per SM this halves
// the column operand's share of the shared-memory traffic (TMA writes and MMA reads) and of
// the stage ring, so more stages fit and the tensor pipe is not starved by operand
// delivery; a stage carries two K-chunks when the contraction has an even number of them,
// which halves the barrier and commit traffic per MMA. Each CTA's Tensor Memory receives
// the scores of its own 128 rows, and its eight epilogue warps run the same online LSE as
// the single-CTA pass.
//
// Units are (256-row pair tile, 256-column tile); the pairs (gridDim.x / 2) split the
// unit list stream-K. Roles in each CTA: warp 0 lane 0 loads this CTA's operand halves
// (the byte counts complete on the even CTA's barriers), warp 1 lane 0 of the even CTA
// issues the MMAs and commits to the barriers of both CTAs, warps 2..9 are the epilogue
// (local arrivals on "accumulator drained"; in the odd CTA, lane 0 of the MMA warp forwards
// them to the even CTA's barrier once all eight warps have arrived).
// ---------------------------------------------------------------------------------------
template <bool kBF16, bool kARes>
__global__ void __launch_bounds__(kLseThreads, 1)
lse_pair_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const float* __restrict__ colBias, int64_t n_rows, int64_t NT, int64_t T,
                int kc_count, int stages, int kps, float kappa, float2* __restrict__ partial,
                int64_t ld, unsigned* __restrict__ status) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctrl ctl;
  constexpr int kGroups = 2;               // partial slots per CTA pair and row tile
  constexpr int kElems = kBF16 ? 64 : 32;  // elements per 128-byte K-chunk row
  constexpr int kEpiWarps = kLseEpiThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: the pair's MMA issuer
  const uint32_t raw = ptx::smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = dyn_smem + (base - raw);
  const uint32_t a_bytes = kARes ? (uint32_t)kc_count * kChunk : 0u;
  // A stage holds kps K-chunks, each [A chunk +] B half chunk.
  const uint32_t chunk_bytes = kARes ? kChunk : 2u * kChunk;
  const uint32_t stage_bytes = (uint32_t)kps * chunk_bytes;
  const uint32_t b_off = kARes ? 0u : (uint32_t)kChunk;
  const uint32_t abase = base;  // the resident row tile (one buffer)
  const uint32_t sbase = base + a_bytes;
  const int64_t G = gridDim.x / 2, pair = blockIdx.x / 2;
  const int64_t t_begin = sk_begin(pair, T, G), t_end = sk_begin(pair + 1, T, G);
  const SegOrder so(t_begin, t_end, NT);  // every role walks the segments in this order

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl.acc_full[b], 1);
      // One lane per local epilogue warp; the even CTA's also counts the odd CTA's forwarder.
      ptx::mbar_init(&ctl.acc_empty[b], kEpiWarps + (rank == 0 ? 1 : 0));
      ptx::mbar_init(&ctl.a_full[b], 1);
      ptx::mbar_init(&ctl.a_empty[b], 1);
    }
    ptx::mbar_init(&ctl.mma_done, 1);
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&mapA);
    ptx::tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&ctl.tmem_base, kLseTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' barriers initialised and Tensor Memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  auto leader = [&](uint64_t* bar) { return ptx::mapa_shared(ptx::smem_u32(bar), 0u); };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------- TMA producer -------------------------------------
      uint32_t stage = 0, ph = 0;
      int64_t issued = 0, segs = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < so.n; ++i) {
        int64_t t, seg_end;
        so.get(i, t, seg_end);
        const int64_t rp = t / NT;
        const int row0 = (int)(rp * 2 * kBM + rank * kBM);  // this CTA's 128 rows
        if constexpr (kARes) {
          if (!ptx::mbar_wait(&ctl.a_empty[0], ((uint32_t)segs & 1u) ^ 1u)) { ok = false; break; }
          if (rank == 0) ptx::mbar_arrive_expect_tx(&ctl.a_full[0], 2u * a_bytes);
          const uint32_t bar = leader(&ctl.a_full[0]);
          for (int kc = 0; kc < kc_count; ++kc)
            ptx::tma_load_2d_pair(&mapA, bar, smem + (size_t)kc * kChunk, kc * kElems, row0);
          ++segs;
        }
        for (int64_t tt = t; ok && tt < seg_end; ++tt) {
          const int col0 = (int)((tt - rp * NT) * kLseBN + rank * kBM);  // this CTA's half
          for (int kc = 0; kc < kc_count; kc += kps) {
            if (!ptx::mbar_wait(&ctl.empty[stage], ph ^ 1u)) { ok = false; break; }
            uint8_t* st = smem + (size_t)a_bytes + (size_t)stage * stage_bytes;
            if (rank == 0) ptx::mbar_arrive_expect_tx(&ctl.full[stage], 2u * stage_bytes);
            const uint32_t bar = leader(&ctl.full[stage]);
            for (int c2 = 0; c2 < kps; ++c2) {
              uint8_t* cst = st + (size_t)c2 * chunk_bytes;
              if constexpr (!kARes)
                ptx::tma_load_2d_pair(&mapA, bar, cst, (kc + c2) * kElems, row0);
              ptx::tma_load_2d_pair(&mapB, bar, cst + b_off, (kc + c2) * kElems, col0);
            }
            ++issued;
            if (++stage == (uint32_t)stages) { stage = 0; ph ^= 1u; }
          }
        }
      }
      if (!ok) flag_error(ctl, status);
      if (rank == 0) {
        // Drain: every copy of both CTAs counted on these barriers has landed.
        for (int s = 0; s < stages; ++s) {
          const int64_t arms = issued / stages + (s < issued % stages ? 1 : 0);
          if (arms > 0) ptx::mbar_wait(&ctl.full[s], (uint32_t)((arms - 1) & 1));
        }
        if (segs > 0) ptx::mbar_wait(&ctl.a_full[0], (uint32_t)((segs - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------- MMA issuer ----------------------------------------
      constexpr uint32_t idesc = ptx::make_idesc<kBF16>(2 * kBM, kLseBN);
      uint32_t stage = 0, ph = 0, ab = 0, acc_ph = 0;
      int64_t segs = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < so.n; ++i) {
        int64_t t, seg_end;
        so.get(i, t, seg_end);
        if constexpr (kARes) {
          if (!ptx::mbar_wait(&ctl.a_full[0], (uint32_t)(segs & 1))) { ok = false; break; }
          ptx::tc_fence_after();
        }
        for (int64_t tt = t; ok && tt < seg_end; ++tt) {
          if (!ptx::mbar_wait_cluster(&ctl.acc_empty[ab], acc_ph ^ 1u)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem + ab * kLseBN;
          for (int kc = 0; kc < kc_count; kc += kps) {
            if (!ptx::mbar_wait(&ctl.full[stage], ph)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t st = sbase + stage * stage_bytes;
            for (int c2 = 0; c2 < kps; ++c2) {
              const uint32_t cst = st + (uint32_t)c2 * chunk_bytes;
              const uint32_t a_addr = kARes ? abase + (uint32_t)(kc + c2) * kChunk : cst;
              const uint64_t a_desc = ptx::sdesc_k128(a_addr);
              const uint64_t b_desc = ptx::sdesc_k128(cst + b_off);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // K advance: 32 bytes = 2 in the address field
                ptx::umma_pair<kBF16>(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                                      (kc | c2 | kk) != 0 ? 1u : 0u);
            }
            ptx::umma_commit_pair(&ctl.empty[stage], 0x3);
            if (++stage == (uint32_t)stages) { stage = 0; ph ^= 1u; }
          }
          if (!ok) break;
          ptx::umma_commit_pair(&ctl.acc_full[ab], 0x3);
          if (++ab == 2) { ab = 0; acc_ph ^= 1u; }
        }
        if constexpr (kARes) ptx::umma_commit_pair(&ctl.a_empty[0], 0x3);
        ++segs;
      }
      if (!ok) flag_error(ctl, status);
      // Every MMA issued must have retired before either CTA releases its Tensor Memory.
      ptx::umma_commit_pair(&ctl.mma_done, 0x1);
      ptx::mbar_wait(&ctl.mma_done, 0);
    } else if (lane == 0) {
      // --------------------- odd CTA: accumulator-drained forwarder ------------------------
      // Once this CTA's eight epilogue warps have read an accumulator (local arrivals), one
      // arrival at cluster scope tells the even CTA's MMA issuer; the epilogue warps never
      // wait on a cluster-scope release themselves.
      uint32_t ab = 0, acc_ph = 0;
      bool ok = true;
      for (int64_t tt = t_begin; tt < t_end; ++tt) {
        if (!ptx::mbar_wait(&ctl.acc_empty[ab], acc_ph)) { ok = false; break; }
        ptx::tc_fence_after();
        ptx::tc_fence_before();
        ptx::mbar_arrive_cluster(leader(&ctl.acc_empty[ab]));
        if (++ab == 2) { ab = 0; acc_ph ^= 1u; }
      }
      if (!ok) flag_error(ctl, status);
    }
  } else {
    // --------------------------------- epilogue ------------------------------------------
    // Warp w reads TMEM lane quarter (w % 4) (this CTA's rows 32q .. 32q+31) and column half
    // h = (w - 2) / 4 of every 256-column tile; each (row, half) keeps its own online
    // (max, sum) and becomes its own partial slot.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t ab = 0, acc_ph = 0;
    bool ok = true;
    if (so.n > 0 && lane < 4) {  // 512 B of bias per half-tile: one line per lane
      int64_t t0, t1;
      so.get(0, t0, t1);
      ptx::prefetch_l1(colBias + (t0 % NT) * kLseBN + h * 128 + lane * 32);
    }
    for (int64_t i = 0; ok && i < so.n; ++i) {
      int64_t t, seg_end;
      so.get(i, t, seg_end);
      const int64_t rp = t / NT;
      float M = kNegBig, S = 0.0f;
      for (int64_t tt = t; tt < seg_end; ++tt) {
        const float4* cb =
            reinterpret_cast<const float4*>(colBias + (tt % NT) * kLseBN + h * 128);
        if (tt + 1 < seg_end && lane < 4)  // the next tile of the segment (a hint only)
          ptx::prefetch_l1(colBias + ((tt + 1) % NT) * kLseBN + h * 128 + lane * 32);
        if (!ptx::mbar_wait(&ctl.acc_full[ab], acc_ph)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t taddr = tmem + lane_base + ab * kLseBN + h * 128;
        float v[64];
        ptx::tmem_ld_x64_sync(taddr, v);
        lse_chunk<64, true>(v, cb, kappa, M, S);
        ptx::tmem_ld_x64_sync(taddr + 64, v);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ctl.acc_empty[ab]);
        if (++ab == 2) { ab = 0; acc_ph ^= 1u; }
        lse_chunk<64, true>(v, cb + 16, kappa, M, S);
      }
      if (!ok) break;
      const int64_t row = rp * 2 * kBM + rank * kBM + q * 32 + lane;
      const int64_t slot = kGroups * (pair - sk_owner(rp * NT, T, G)) + h;
      if (row < n_rows) partial[slot * ld + row] = make_float2(M, S);
    }
    if (!ok) flag_error(ctl, status);
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();  // neither CTA leaves while the pair's MMAs or copies may touch it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kLseTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// Weighted-sum pass: transport application, barycentric gradient, Hadamard-weighted
// transport (FlashSinkhorn, SAI replication review, "Summary" (i)-(ii)). Per CTA = (row
// tile, group of kKV output columns):
//   S   = rows * cols^T                      tcgen05.mma, double-buffered in TMEM
//   w_ij = exp2(kappa S_ij + colBias_j + rowBias_i)         epilogue, fp32 + MUFU ex2
//   O   += W * V^T-tile                      second tcgen05.mma, W written to shared memory
//                                            by the epilogue in the swizzled K-major layout
// The weights are bounded (plan entries, or a_i times softmax weights), so no running max
// is needed. The S MMA of tile j+1 overlaps the epilogue of tile j. kKV == 0: Hadamard
// only (h_i = sum_j w_ij S_ij, no second MMA).
// ---------------------------------------------------------------------------------------
constexpr int kWsMaxStages = 4;

struct __align__(128) WCtrl {
  uint64_t full[kWsMaxStages];
  uint64_t empty[kWsMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t w_full[2];
  uint64_t w_empty[2];
  uint64_t v_full[2];
  uint64_t v_empty[2];
  uint64_t o_full;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float bias[4][2][kBN];     // read as float4
};
static_assert(offsetof(WCtrl, bias) % 16 == 0, "bias is read with 16-byte vector loads");

__device__ __forceinline__ void flag_error_w(WCtrl& ctl, unsigned* status) {
  atomicOr(status, kErrTimeout);
  ctl.abort_flag = 1;
}

template <bool kBF16, int kMode, int kKV>
__global__ void __launch_bounds__(kThreads, 1)
wsum_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
               const __grid_constant__ CUtensorMap mapV, const float* __restrict__ colBias,
               const float* __restrict__ rowBias, int64_t n_rows, int NT, int kc_count, int n_st,
               int n_w, int n_v, float kappa, const float* __restrict__ rowW,
               const float* __restrict__ Xrow, int64_t d, int64_t k, float* __restrict__ out,
               int64_t ldo, unsigned* __restrict__ status, int tps, float* __restrict__ part,
               int64_t rows_pad, int kp) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ WCtrl ctl;
  constexpr bool kHad = (kKV == 0);
  constexpr int es = kBF16 ? 2 : 4;
  constexpr int kElems = 128 / es;                       // elements per 128-byte K-chunk row
  constexpr int kWChunks = kBN * es / 128;               // K-chunks over the 128 columns j
  constexpr uint32_t kWBytes = (uint32_t)kWChunks * kChunk;
  constexpr uint32_t kVChunkBytes = (uint32_t)(kKV > 0 ? kKV : 1) * 128;
  constexpr uint32_t kVBytes = kHad ? 0u : (uint32_t)kWChunks * kVChunkBytes;
  constexpr int kVBoxRows = kKV > 128 ? 128 : (kKV > 0 ? kKV : 1);
  constexpr uint32_t kTmemCols = kHad ? 256u : 512u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = ptx::smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = dyn_smem + (base - raw);
  const uint32_t st_base = 0;
  const uint32_t w_base = (uint32_t)n_st * 2u * kChunk;
  const uint32_t v_base = w_base + (uint32_t)n_w * kWBytes;
  const int64_t rt = blockIdx.x;
  const int64_t o0 = (int64_t)blockIdx.y * kKV;
  // Column split blockIdx.z: global column tiles [j_begin, j_begin + NTl); the loops below
  // count local tiles (buffer parities), the loads and biases use global ones.
  const int j_begin = (int)blockIdx.z * tps;
  const int NTl = min(NT, j_begin + tps) - j_begin;

  if (threadIdx.x == 0) {
    for (int s = 0; s < n_st; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl.acc_full[b], 1);
      ptx::mbar_init(&ctl.acc_empty[b], 128);
      ptx::mbar_init(&ctl.w_full[b], 128);
      ptx::mbar_init(&ctl.w_empty[b], 1);
      ptx::mbar_init(&ctl.v_full[b], 1);
      ptx::mbar_init(&ctl.v_empty[b], 1);
    }
    ptx::mbar_init(&ctl.o_full, 1);
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
      for (int jt = 0; ok && jt < NTl; ++jt) {
        for (int kc = 0; kc < kc_count; ++kc) {
          if (!ptx::mbar_wait(&ctl.empty[stage], ph ^ 1u)) { ok = false; break; }
          uint8_t* st = smem + st_base + (size_t)stage * 2 * kChunk;
          ptx::mbar_arrive_expect_tx(&ctl.full[stage], 2 * kChunk);
          ptx::tma_load_2d(&mapA, &ctl.full[stage], st, kc * kElems, (int)(rt * kBM));
          ptx::tma_load_2d(&mapB, &ctl.full[stage], st + kChunk, kc * kElems,
                           (j_begin + jt) * kBN);
          ++issued;
          if (++stage == (uint32_t)n_st) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        if constexpr (!kHad) {
          const int vs = jt % n_v;
          if (!ptx::mbar_wait(&ctl.v_empty[vs], (uint32_t)((jt / n_v) & 1) ^ 1u)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&ctl.v_full[vs], kVBytes);
          uint8_t* vt = smem + v_base + (size_t)vs * kVBytes;
          for (int vc = 0; vc < kWChunks; ++vc)
            for (int ob = 0; ob < kKV / kVBoxRows; ++ob)
              ptx::tma_load_2d(&mapV, &ctl.v_full[vs], vt + (size_t)vc * kVChunkBytes + ob * kVBoxRows * 128,
                               (j_begin + jt) * kBN + vc * kElems, (int)(o0 + ob * kVBoxRows));
          ++v_issued;
        }
      }
      if (!ok) flag_error_w(ctl, status);
      for (int s = 0; s < n_st; ++s) {
        const int64_t arms = issued / n_st + (s < issued % n_st ? 1 : 0);
        if (arms > 0) ptx::mbar_wait(&ctl.full[s], (uint32_t)((arms - 1) & 1));
      }
      for (int s = 0; s < n_v; ++s) {
        const int64_t arms = v_issued / n_v + (s < v_issued % n_v ? 1 : 0);
        if (arms > 0) ptx::mbar_wait(&ctl.v_full[s], (uint32_t)((arms - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------- MMA issuer ----------------------------------------
      constexpr uint32_t idesc_s = ptx::make_idesc<kBF16>(kBM, kBN);
      constexpr uint32_t idesc_o = ptx::make_idesc<kBF16>(kBM, kKV > 0 ? kKV : 128);
      uint32_t stage = 0, ph = 0;
      bool ok = true;
      for (int t = 0; ok && t <= NTl; ++t) {
        if (t < NTl) {
          const uint32_t ab = (uint32_t)(t & 1);
          if (!ptx::mbar_wait(&ctl.acc_empty[ab], (uint32_t)((t >> 1) & 1) ^ 1u)) { ok = false; break; }
          ptx::tc_fence_after();
          for (int kc = 0; kc < kc_count; ++kc) {
            if (!ptx::mbar_wait(&ctl.full[stage], ph)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t st = base + st_base + stage * 2u * kChunk;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::umma<kBF16>(tmem + ab * kBN, ptx::sdesc_k128(st + kk * 32),
                               ptx::sdesc_k128(st + kChunk + kk * 32), idesc_s,
                               (kc | kk) != 0 ? 1u : 0u);
            ptx::umma_commit(&ctl.empty[stage]);
            if (++stage == (uint32_t)n_st) { stage = 0; ph ^= 1u; }
          }
          if (!ok) break;
          ptx::umma_commit(&ctl.acc_full[ab]);
        }
        if constexpr (!kHad) {
          if (t >= 1) {
            const int u = t - 1;
            const int wb = u % n_w, vs = u % n_v;
            if (!ptx::mbar_wait(&ctl.w_full[wb], (uint32_t)((u / n_w) & 1))) { ok = false; break; }
            if (!ptx::mbar_wait(&ctl.v_full[vs], (uint32_t)((u / n_v) & 1))) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t wa = base + w_base + (uint32_t)wb * kWBytes;
            const uint32_t va = base + v_base + (uint32_t)vs * kVBytes;
#pragma unroll
            for (int vc = 0; vc < kWChunks; ++vc) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::umma<kBF16>(tmem + 256, ptx::sdesc_k128(wa + vc * kChunk + kk * 32),
                                 ptx::sdesc_k128(va + vc * kVChunkBytes + kk * 32), idesc_o,
                                 (u | vc | kk) != 0 ? 1u : 0u);
            }
            ptx::umma_commit(&ctl.w_empty[wb]);
            ptx::umma_commit(&ctl.v_empty[vs]);
          }
        }
      }
      if constexpr (!kHad) ptx::umma_commit(&ctl.o_full);
      if (!ok) flag_error_w(ctl, status);
      ptx::umma_commit(&ctl.mma_done);
      ptx::mbar_wait(&ctl.mma_done, 0);
    }
  } else {
    // --------------------------------- epilogue ------------------------------------------
    const int q = warp & 3;
    const int ew = warp - 2;
    const int rloc = q * 32 + lane;            // row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int64_t row = rt * kBM + rloc;
    const float rb = row < n_rows ? rowBias[row] : neg_inf();
    float sumw = 0.0f, had = 0.0f;
    bool ok = true;
    float4 bnext = __ldg(reinterpret_cast<const float4*>(colBias + (int64_t)j_begin * kBN) + lane);
    for (int jt = 0; jt < NTl; ++jt) {
      const int bb = jt & 1;
      reinterpret_cast<float4*>(ctl.bias[ew][bb])[lane] = bnext;
      if (jt + 1 < NTl)
        bnext = __ldg(reinterpret_cast<const float4*>(colBias + (int64_t)(j_begin + jt + 1) * kBN) +
                      lane);
      __syncwarp();
      const uint32_t ab = (uint32_t)(jt & 1);
      if (!ptx::mbar_wait(&ctl.acc_full[ab], (uint32_t)((jt >> 1) & 1))) { ok = false; break; }
      ptx::tc_fence_after();
      float v[kBN];
      ptx::tmem_ld_x128_sync(tmem + lane_base + ab * kBN, v);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl.acc_empty[ab]);
      const float4* cb = reinterpret_cast<const float4*>(ctl.bias[ew][bb]);
#pragma unroll
      for (int j = 0; j < kBN; j += 4) {
        const float4 b4 = cb[j / 4];
        const float w0 = ex2(fmaf(kappa, v[j + 0], b4.x) + rb);
        const float w1 = ex2(fmaf(kappa, v[j + 1], b4.y) + rb);
        const float w2 = ex2(fmaf(kappa, v[j + 2], b4.z) + rb);
        const float w3 = ex2(fmaf(kappa, v[j + 3], b4.w) + rb);
        if constexpr (kHad) {
          had = fmaf(w0, v[j + 0], had);
          had = fmaf(w1, v[j + 1], had);
          had = fmaf(w2, v[j + 2], had);
          had = fmaf(w3, v[j + 3], had);
        }
        sumw += (w0 + w1) + (w2 + w3);
        v[j + 0] = w0;
        v[j + 1] = w1;
        v[j + 2] = w2;
        v[j + 3] = w3;
      }
      if constexpr (!kHad) {
        const int wb = jt % n_w;
        if (!ptx::mbar_wait(&ctl.w_empty[wb], (uint32_t)((jt / n_w) & 1) ^ 1u)) { ok = false; break; }
        const uint32_t wrow = base + w_base + (uint32_t)wb * kWBytes + (uint32_t)rloc * 128u;
#pragma unroll
        for (int c = 0; c < kWChunks; ++c) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint32_t p0, p1, p2, p3;
            if constexpr (kBF16) {
              const int j = c * 64 + u * 8;
              __nv_bfloat162 h0 = __floats2bfloat162_rn(v[j + 0], v[j + 1]);
              __nv_bfloat162 h1 = __floats2bfloat162_rn(v[j + 2], v[j + 3]);
              __nv_bfloat162 h2 = __floats2bfloat162_rn(v[j + 4], v[j + 5]);
              __nv_bfloat162 h3 = __floats2bfloat162_rn(v[j + 6], v[j + 7]);
              p0 = *reinterpret_cast<uint32_t*>(&h0);
              p1 = *reinterpret_cast<uint32_t*>(&h1);
              p2 = *reinterpret_cast<uint32_t*>(&h2);
              p3 = *reinterpret_cast<uint32_t*>(&h3);
            } else {
              const int j = c * 32 + u * 4;
              asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(p0) : "f"(v[j + 0]));
              asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(p1) : "f"(v[j + 1]));
              asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(p2) : "f"(v[j + 2]));
              asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(p3) : "f"(v[j + 3]));
            }
            ptx::st_shared_v4(wrow + (uint32_t)c * kChunk + (uint32_t)((u ^ (rloc & 7)) << 4),
                              p0, p1, p2, p3);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&ctl.w_full[wb]);
      }
    }
    // With column splits (part != NULL) the raw sums go to part[(split rows_pad + row) kp + o]
    // (sum w or the Hadamard sum in column kp - 1) for wsum_split_reduce_kernel.
    float* pr = part != nullptr ? part + ((int64_t)blockIdx.z * rows_pad + row) * kp : nullptr;
    if constexpr (kHad) {
      if (ok && row < n_rows) {
        if (pr != nullptr) pr[kp - 1] = had;
        else out[row] = had;
      }
    } else {
      if (ok && !ptx::mbar_wait(&ctl.o_full, 0)) ok = false;
      if (ok) {
        ptx::tc_fence_after();
        const float a = (kMode == kWsumGrad && row < n_rows) ? rowW[row] : 0.0f;
        const float inv = sumw > 0.0f ? 1.0f / sumw : 0.0f;
#pragma unroll 1
        for (int c = 0; c < kKV / 32; ++c) {
          float o[32];
          ptx::tmem_ld_x32_sync(tmem + lane_base + 256 + c * 32, o);
          if (row < n_rows && pr != nullptr) {
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              const int64_t oo = o0 + c * 32 + t;
              if (oo < kp - 1) pr[oo] = o[t];
            }
            if (c == 0 && blockIdx.y == 0) pr[kp - 1] = sumw;
          } else if (row < n_rows) {
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              const int64_t oo = o0 + c * 32 + t;
              if constexpr (kMode == kWsumGrad) {
                if (oo < d)
                  out[row * ldo + oo] = a > 0.0f ? 2.0f * a * (Xrow[row * d + oo] - o[t] * inv) : 0.0f;
              } else {
                if (oo < k) out[row * ldo + oo] = o[t];
              }
            }
          }
        }
      }
    }
    if (!ok) flag_error_w(ctl, status);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Waits on a barrier that never completes; the bounded wait gives up and reports.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, unsigned* __restrict__ status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
    if (!ptx::mbar_wait(&bar, 0, limit_ns)) atomicOr(status, kErrTimeout);
  }
}

}  // namespace tc

using namespace tc;

int tc_selftest_bounded_wait(unsigned* status, int64_t limit_ns, cudaStream_t st) {
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
    bounded_wait_selftest_kernel<<<1, 32, 0, st>>>((uint64_t)limit_ns, status);
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

int tc_pack_inputs(int mode, const float* X, const float* Y, int64_t n, int64_t m, int64_t d,
                   int64_t n_pad, int64_t m_pad, int64_t dpt, void* xq, void* yq, int sms,
                   cudaStream_t st) {
  const int T = 256;
  const unsigned g1 = (unsigned)std::min<int64_t>((n_pad * dpt + T - 1) / T, (int64_t)sms * 16);
  const unsigned g2 = (unsigned)std::min<int64_t>((m_pad * dpt + T - 1) / T, (int64_t)sms * 16);
  const bool bf16 = (mode == 1);
  if (mode == 2) {
    { TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      pack_rows_tf32x3_kernel<<<g1, T, 0, st>>>(X, static_cast<uint32_t*>(xq), n, d, n_pad, dpt,
                                                0b100); }
    { TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      pack_rows_tf32x3_kernel<<<g2, T, 0, st>>>(Y, static_cast<uint32_t*>(yq), m, d, m_pad, dpt,
                                                0b010); }
  } else if (bf16) {
    { TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      pack_rows_kernel<PackKind::BF16><<<g1, T, 0, st>>>(X, xq, n, d, n_pad, dpt); }
    { TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      pack_rows_kernel<PackKind::BF16><<<g2, T, 0, st>>>(Y, yq, m, d, m_pad, dpt); }
  } else {
    { TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      pack_rows_kernel<PackKind::TF32><<<g1, T, 0, st>>>(X, xq, n, d, n_pad, dpt); }
    { TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      pack_rows_kernel<PackKind::TF32><<<g2, T, 0, st>>>(Y, yq, m, d, m_pad, dpt); }
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

// Dynamic shared memory of the pair kernel: the row tile when resident, then as many
// stages as fit (at least 4); 0 if fewer fit.
// Shared-memory plan of the pair kernel: the row tile when resident, then a ring of stages
// of kps K-chunks. Two chunks per stage when the chunk count is even and at least three
// such stages fit; else one chunk per stage and at least four stages. Returns the dynamic
// shared memory (0 if no plan fits) and sets *stages and *kps.
template <bool kARes>
static int lse_pair_smem(int kc, int* stages_out = nullptr, int* kps_out = nullptr) {
  const int ctrl = (int)sizeof(Ctrl) + 2 * 4 * (int)sizeof(float);
  const int a_bytes = kARes ? kc * kChunk : 0;
  const int chunk_bytes = kARes ? kChunk : 2 * kChunk;
  const int room = kSmemLimit - ctrl - 1024 - a_bytes;
  int kps = 1, stages = std::min(kMaxStages, room / chunk_bytes);
  if (kc % 2 == 0 && room / (2 * chunk_bytes) >= 3) {
    kps = 2;
    stages = std::min(kMaxStages, room / (2 * chunk_bytes));
  } else if (stages < 4) {
    return 0;
  }
  if (stages_out) *stages_out = stages;
  if (kps_out) *kps_out = kps;
  return a_bytes + stages * kps * chunk_bytes + 1024;
}

template <bool kBF16, bool kARes, bool kStageBias>
static int launch_lse(const CUtensorMap& mA, const CUtensorMap& mB, const float* colBias,
                      int64_t n_rows, int64_t NT, int64_t T, int kc, int64_t G, float kappa,
                      float2* partial, int64_t ld, unsigned* status, cudaStream_t st) {
  // Static shared memory: the control block and the staged column biases.
  const int ctrl = (int)sizeof(Ctrl) +
                   (kStageBias ? kLseEpiThreads / 32 * 2 * kLseBN : 2 * 4) * (int)sizeof(float);
  const int a_bytes = kARes ? kc * kChunk : 0;
  const int stage_bytes = kARes ? 2 * kChunk : 3 * kChunk;
  // A second row-tile buffer when at least four operand stages still fit beside it.
  const int a_bufs =
      (kARes && (kSmemLimit - ctrl - 1024 - 2 * a_bytes) / stage_bytes >= 4) ? 2 : 1;
  const int budget = kSmemLimit - ctrl - 1024 - a_bufs * a_bytes;
  const int stages = std::min(kMaxStages, budget / stage_bytes);
  if (stages < 2) return FLASHOT_ERR_INVALID_ARG;
  const int dyn = a_bufs * a_bytes + stages * stage_bytes + 1024;
  auto kern = lse_tc_kernel<kBF16, kARes, kStageBias>;
  int rc = set_smem(kern, dyn);
  if (rc != FLASHOT_OK) return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_LSE, st);
    if constexpr (kStageBias) {
      // Programmatic dependent of the kernel ahead of it (see the kernel's epilogue).
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)G);
      cfg.blockDim = dim3(kLseThreads);
      cfg.dynamicSmemBytes = (size_t)dyn;
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, kern, mA, mB, colBias, n_rows, NT, T, kc, stages, a_bufs,
                             kappa, partial, ld, status) != cudaSuccess)
        return FLASHOT_ERR_CUDA;
    } else {
      kern<<<(unsigned)G, kLseThreads, dyn, st>>>(mA, mB, colBias, n_rows, NT, T, kc, stages,
                                                  a_bufs, kappa, partial, ld, status);
    }
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

// The CTA-pair pass: cluster launch of 2 CTAs, grid = 2 x pairs.
template <bool kBF16, bool kARes>
static int launch_lse_pair(const CUtensorMap& mA, const CUtensorMap& mB, const float* colBias,
                           int64_t n_rows, int64_t NT, int64_t T, int kc, int64_t pairs,
                           float kappa, float2* partial, int64_t ld, unsigned* status,
                           cudaStream_t st) {
  int stages = 0, kps = 1;
  const int dyn = lse_pair_smem<kARes>(kc, &stages, &kps);
  if (dyn <= 0) return FLASHOT_ERR_INVALID_ARG;
  auto kern = lse_pair_kernel<kBF16, kARes>;
  int rc = set_smem(kern, dyn);
  if (rc != FLASHOT_OK) return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_LSE, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kLseThreads);
    cfg.dynamicSmemBytes = (size_t)dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mA, mB, colBias, n_rows, NT, T, kc, stages, kps, kappa,
                           partial, ld, status) != cudaSuccess)
      return FLASHOT_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

// How many 2-CTA clusters of the pair kernel can be resident at once (0 if none, or if
// the query fails); cached per variant.
template <bool kBF16, bool kARes>
static int lse_pair_max_clusters(int kc) {
  static int cached_kc = -1, cached = 0;
  if (cached_kc == kc) return cached;
  const int dyn = lse_pair_smem<kARes>(kc);
  int n = 0;
  if (dyn > 0) {
    auto kern = lse_pair_kernel<kBF16, kARes>;
    if (set_smem(kern, dyn) == FLASHOT_OK) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(kLseThreads);
      cfg.dynamicSmemBytes = (size_t)dyn;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
    } else {
      cudaGetLastError();
    }
  }
  cached_kc = kc;
  cached = n;
  return n;
}

int tc_lse_pass(bool bf16, const void* rowQ, const void* colQ, const float* colBias,
                int64_t n_rows, int64_t rows_pad, int64_t cols_pad, int64_t dpt, float kappa,
                float2* partial, int max_splits, int sms, unsigned* status, SplitInfo* info,
                cudaStream_t st) {
  const int es = bf16 ? 2 : 4;
  const int kc = (int)(dpt * es / 128);
  if (rows_pad % kBM != 0 || cols_pad % kLseBN != 0) return FLASHOT_ERR_INVALID_ARG;
  const int64_t row_tiles = rows_pad / kBM, NT = cols_pad / kLseBN;
  const int64_t T = row_tiles * NT;
  const bool ares = kc * kChunk <= 128 * 1024;
  // Stage the biases in shared memory when the contraction is short (at most 6 K-chunks,
  // e.g. d <= 192 in bf16 or d <= 64 in split tf32: the epilogue bounds the tile, and at
  // least 3 operand stages still fit).
  const bool stage = kc <= 6;
  CUtensorMap mA, mB;
  int rc = make_map(&mA, rowQ, rows_pad, dpt, bf16);
  if (rc != FLASHOT_OK) return rc;
  info->n_splits = 0;
  info->slots_per_owner = 2;
  info->sk_NT = NT;
  // Long contractions run on CTA pairs (cta_group::2) when 256-row pair tiles divide the rows
  // and enough 2-CTA clusters fit; FLASHOT_LSE_PAIRS=0 in the environment keeps them on
  // single CTAs (for comparisons).
  static const bool pairs_enabled = [] {
    const char* e = std::getenv("FLASHOT_LSE_PAIRS");
    return !(e && e[0] == '0');
  }();
  if (!stage && pairs_enabled && rows_pad % (2 * kBM) == 0) {
    const int max_cl = bf16 ? (ares ? lse_pair_max_clusters<true, true>(kc)
                                    : lse_pair_max_clusters<true, false>(kc))
                            : (ares ? lse_pair_max_clusters<false, true>(kc)
                                    : lse_pair_max_clusters<false, false>(kc));
    const int64_t prt = rows_pad / (2 * kBM);
    if (max_cl >= std::max(1, sms / 4)) {
      const int64_t T2 = prt * NT;
      // Two partial slots (column halves) per pair and pair tile.
      const int64_t G2 = choose_grid(prt, NT, std::min(max_cl, sms / 2), max_splits / 2);
      rc = make_map(&mB, colQ, cols_pad, dpt, bf16);
      if (rc != FLASHOT_OK) return rc;
      info->sk_T = T2;
      info->sk_G = G2;
      info->unit_rows = 2 * kBM;
#define FLASHOT_LAUNCH_PAIR(BF, AR) \
  launch_lse_pair<BF, AR>(mA, mB, colBias, n_rows, NT, T2, kc, G2, kappa, partial, rows_pad, status, st)
      if (bf16) return ares ? FLASHOT_LAUNCH_PAIR(true, true) : FLASHOT_LAUNCH_PAIR(true, false);
      return ares ? FLASHOT_LAUNCH_PAIR(false, true) : FLASHOT_LAUNCH_PAIR(false, false);
#undef FLASHOT_LAUNCH_PAIR
    }
  }
  // Two partial slots (column halves) per CTA and row tile.
  const int64_t G = choose_grid(row_tiles, NT, sms, max_splits / 2);
  rc = make_map_rows(&mB, colQ, cols_pad, dpt, bf16, kLseBN);
  if (rc != FLASHOT_OK) return rc;
  info->sk_T = T;
  info->sk_G = G;
  info->unit_rows = kBM;
#define FLASHOT_LAUNCH_LSE(BF, AR, SB)                                                        \
  launch_lse<BF, AR, SB>(mA, mB, colBias, n_rows, NT, T, kc, G, kappa, partial, rows_pad, \
                         status, st)
  if (stage) return bf16 ? FLASHOT_LAUNCH_LSE(true, true, true) : FLASHOT_LAUNCH_LSE(false, true, true);
  if (bf16) return ares ? FLASHOT_LAUNCH_LSE(true, true, false) : FLASHOT_LAUNCH_LSE(true, false, false);
  return ares ? FLASHOT_LAUNCH_LSE(false, true, false) : FLASHOT_LAUNCH_LSE(false, false, false);
#undef FLASHOT_LAUNCH_LSE
}

template <bool kBF16, int kMode, int kKV>
static int launch_wsum(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mV,
                       const float* colBias, const float* rowBias, int64_t n_rows,
                       int64_t row_tiles, int groups, int NT, int kc, float kappa,
                       const float* rowW, const float* X, int64_t d, int64_t k, float* out,
                       int64_t ldo, unsigned* status, cudaStream_t st, int splits, int tps,
                       float* part, int64_t rows_pad, int kp) {
  constexpr int es = kBF16 ? 2 : 4;
  const int w_bytes = (kKV == 0) ? 0 : kBN * es * 128;             // 128 rows x 128 columns
  const int v_bytes = (kKV == 0) ? 0 : kKV * 128 * (kBN * es / 128);
  const int budget = kSmemLimit - (int)sizeof(WCtrl) - 1024;
  // At least 2 operand stages, one W and one V buffer; then double W, double V, more stages.
  int n_st = 2, n_w = (kKV == 0) ? 0 : 1, n_v = (kKV == 0) ? 0 : 1;
  auto total = [&]() { return n_st * 2 * kChunk + n_w * w_bytes + n_v * v_bytes; };
  if (total() > budget) return FLASHOT_ERR_INVALID_ARG;
  if (kKV != 0 && total() + w_bytes <= budget) ++n_w;
  if (kKV != 0 && total() + v_bytes <= budget) ++n_v;
  while (n_st < kWsMaxStages && total() + 2 * kChunk <= budget) ++n_st;
  const int dyn = total() + 1024;
  auto kern = wsum_tc_kernel<kBF16, kMode, kKV>;
  int rc = set_smem(kern, dyn);
  if (rc != FLASHOT_OK) return rc;
  dim3 grid((unsigned)row_tiles, (unsigned)groups, (unsigned)splits);
  {
    TraceScope ts_(FLASHOT_KERNEL_WSUM, st);
    kern<<<grid, kThreads, dyn, st>>>(mA, mB, mV, colBias, rowBias, n_rows, NT, kc, n_st,
                                      std::max(n_w, 1), std::max(n_v, 1), kappa, rowW, X, d, k,
                                      out, ldo, status, tps, splits > 1 ? part : nullptr,
                                      rows_pad, kp);
  }
  if (cudaGetLastError() != cudaSuccess) return FLASHOT_ERR_CUDA;
  if (splits > 1) {
    // the splits' raw sums, added in a fixed order, and the mode's epilogue
    const int64_t total = n_rows * (kMode == kWsumHadamard ? 1 : (kMode == kWsumGrad ? d : k));
    TraceScope ts2_(FLASHOT_KERNEL_OTHER, st);
    wsum_split_reduce_kernel<kMode><<<(unsigned)std::min<int64_t>((total + 255) / 256, 1 << 20),
                                      256, 0, st>>>(part, splits, rows_pad, kp, n_rows,
                                                    kMode == kWsumGrad ? d : k, rowW, X, d, out,
                                                    ldo);
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

// Column splits for the tf32 weighted sums: the split count s (at most 8, and as many as the
// partial buffer holds) that minimises the makespan ceil(CTAs s / SMs) / s, in units of one
// CTA covering a whole row of column tiles; 1 when one wave already fits.
static int choose_splits(int64_t ctas, int NT, int sms, int64_t cap) {
  int best = 1;
  double best_mk = (double)((ctas + sms - 1) / sms);
  for (int sp = 2; sp <= 8 && sp <= NT && sp <= cap; ++sp) {
    const double mk = (double)((ctas * sp + sms - 1) / sms) / sp;
    if (mk < best_mk - 1e-9) {
      best_mk = mk;
      best = sp;
    }
  }
  return best;
}

size_t tc_wsum_split_bytes(int64_t rows_pad, int64_t k_or_d) {
  // kp = output columns (whole 64- or 128-column groups) + 1, at most 8 splits, capped at
  // 64 MB (wide outputs have enough CTAs in their column groups anyway)
  const int64_t kv = k_or_d <= 64 ? 64 : 128;
  const int64_t kp = (k_or_d + kv - 1) / kv * kv + 1;
  return (size_t)std::min<int64_t>(8 * rows_pad * kp * (int64_t)sizeof(float), 64ll << 20);
}

int tc_wsum_pass(bool bf16, int mode, const void* rowQ, const void* colQ, const float* colBias,
                 const float* rowBias, int64_t n_rows, int64_t n_cols, int64_t rows_pad,
                 int64_t cols_pad, int64_t d, int64_t dpt, float kappa, const float* V,
                 int64_t ldv, int64_t k, void* vtq, const float* rowW, const float* X,
                 float* out, int64_t ldo, int sms, unsigned* status, cudaStream_t st,
                 void* split_buf, size_t split_bytes) {
  const int es = bf16 ? 2 : 4;
  const int kc = (int)(dpt * es / 128);
  const int64_t row_tiles = rows_pad / kBM;
  const int NT = (int)(cols_pad / kBN);
  float* part = static_cast<float*>(split_buf);
  CUtensorMap mA, mB, mV;
  int rc = make_map(&mA, rowQ, rows_pad, dpt, bf16);
  if (rc == FLASHOT_OK) rc = make_map(&mB, colQ, cols_pad, dpt, bf16);
  if (rc != FLASHOT_OK) return rc;
  if (mode == kWsumHadamard) {
    mV = mB;  // unused
    const int kp = 2;
    const int64_t cap = part ? (int64_t)(split_bytes / ((size_t)rows_pad * kp * sizeof(float))) : 1;
    int splits = choose_splits(row_tiles, NT, sms, cap);
    const int tps = (NT + splits - 1) / splits;
    splits = (NT + tps - 1) / tps;
    return bf16 ? launch_wsum<true, kWsumHadamard, 0>(mA, mB, mV, colBias, rowBias, n_rows,
                                                      row_tiles, 1, NT, kc, kappa, rowW, X, d, 1,
                                                      out, ldo, status, st, splits, tps, part,
                                                      rows_pad, kp)
                : launch_wsum<false, kWsumHadamard, 0>(mA, mB, mV, colBias, rowBias, n_rows,
                                                       row_tiles, 1, NT, kc, kappa, rowW, X, d,
                                                       1, out, ldo, status, st, splits, tps, part,
                                                       rows_pad, kp);
  }
  // Output-column group width: 64, 128, or 256 (bf16 only; tf32 W/V tiles are twice as big).
  const int kv = (k <= 64) ? 64 : (k <= 128 || !bf16) ? 128 : 256;
  const int groups = (int)((k + kv - 1) / kv);
  const int64_t out_rows_pad = (int64_t)groups * kv;
  if (ldv != k) return FLASHOT_ERR_INVALID_ARG;
  {
    dim3 blk(32, 8), grd((unsigned)(cols_pad / 32), (unsigned)(out_rows_pad / 32));
    TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
    if (bf16)
      pack_transpose_kernel<PackKind::BF16><<<grd, blk, 0, st>>>(V, vtq, n_cols, k, cols_pad,
                                                                 out_rows_pad);
    else
      pack_transpose_kernel<PackKind::TF32><<<grd, blk, 0, st>>>(V, vtq, n_cols, k, cols_pad,
                                                                 out_rows_pad);
  }
  if (cudaGetLastError() != cudaSuccess) return FLASHOT_ERR_CUDA;
  rc = make_map_rows(&mV, vtq, out_rows_pad, cols_pad, bf16, kv > 128 ? 128 : kv);
  if (rc != FLASHOT_OK) return rc;
  const int kp = (int)out_rows_pad + 1;
  const int64_t cap = part ? (int64_t)(split_bytes / ((size_t)rows_pad * kp * sizeof(float))) : 1;
  int splits = choose_splits(row_tiles * groups, NT, sms, cap);
  const int tps = (NT + splits - 1) / splits;
  splits = (NT + tps - 1) / tps;
#define FLASHOT_WSUM_TC(B, M, KV)                                                             \
  launch_wsum<B, M, KV>(mA, mB, mV, colBias, rowBias, n_rows, row_tiles, groups, NT, kc, kappa, \
                        rowW, X, d, k, out, ldo, status, st, splits, tps, part, rows_pad, kp)
  if (mode == kWsumGrad) {
    if (bf16) {
      if (kv == 64) return FLASHOT_WSUM_TC(true, kWsumGrad, 64);
      if (kv == 128) return FLASHOT_WSUM_TC(true, kWsumGrad, 128);
      return FLASHOT_WSUM_TC(true, kWsumGrad, 256);
    }
    if (kv == 64) return FLASHOT_WSUM_TC(false, kWsumGrad, 64);
    return FLASHOT_WSUM_TC(false, kWsumGrad, 128);
  }
  if (bf16) {
    if (kv == 64) return FLASHOT_WSUM_TC(true, kWsumApply, 64);
    if (kv == 128) return FLASHOT_WSUM_TC(true, kWsumApply, 128);
    return FLASHOT_WSUM_TC(true, kWsumApply, 256);
  }
  if (kv == 64) return FLASHOT_WSUM_TC(false, kWsumApply, 64);
  return FLASHOT_WSUM_TC(false, kWsumApply, 128);
#undef FLASHOT_WSUM_TC
}

}  // namespace flashot
