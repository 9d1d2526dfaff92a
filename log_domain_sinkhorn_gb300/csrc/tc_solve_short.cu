// tc_solve_short.cu -- every half-step of an alternating Sinkhorn solve of a short
// contraction in one persistent, cooperative launch (sm_103a, tcgen05).
//
// The method alternates F- and G-updates, each a row-wise log-sum-exp of biased dot-product
// scores whose biases are the other side's latest potentials (FlashSinkhorn: IO-Aware
// Entropic Optimal Transport on GPU, abstract; SAI replication review, "Summary"). For
// short contractions (at most six 128-byte K-chunks: bf16 d <= 192, tf32 d <= 96, split
// tf32 d <= 64) a half-step is a few microseconds of work per SM, and launching a pass and
// then a merge of its stream-K partials costs several more in ramp-up, tail and dependency
// resolution. Here one CTA per SM runs the whole solve:
//   - the TMA producer (warp 0) and the MMA issuer (warp 1) walk the tiles of all passes
//     without stopping: the scores <x_i, y_j> do not depend on the potentials, so the next
//     pass's row tile and first score tiles are loaded and computed while the epilogue is
//     still finishing the current pass;
//   - the eight epilogue warps run the online (max, sum) of the per-pass kernel on the same
//     tiles, the same stream-K ranges and the same partial slots;
//   - at the end of a pass a grid-wide barrier (one counter, release / acquire at GPU scope,
//     bounded wait) waits for every CTA's partials; then every CTA merges an equal share of
//     the rows (the merge of lse_combine_kernel, slots in fixed order), writing the potential
//     and the bias the next pass reads, and a second barrier publishes the merges.
// The arithmetic, and so every bit of the result, is that of the per-pass path.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cstdlib>

#include "flashot.h"
#include "combine.cuh"
#include "common.cuh"
#include "lse_epilogue.cuh"
#include "ptx.cuh"
#include "tc_host.h"
#include "tc_solve_short.h"
#include "trace.h"

namespace flashot {
namespace tc {
namespace ssolve {

constexpr int kBM = 128;                 // rows per tile (MMA M)
constexpr int kBN = 256;                 // columns per tile (MMA N)
constexpr int kChunk = 128 * 128;        // bytes of one 128-row x 128-byte K-chunk box
constexpr int kThreads = 320;            // TMA warp, MMA warp, 8 epilogue warps
constexpr int kEpiThreads = 256;
constexpr int kMaxKc = 6;                // K-chunks of a short contraction
constexpr int kMaxStages = 8;
constexpr int kMaxEps = 32;              // eps stages carried in the launch parameters
constexpr uint32_t kTmemCols = 512;      // two 256-column fp32 accumulators
constexpr int kSmemLimit = 232448;       // 227 KB per block (opt-in maximum)

// One kind of pass: side 0 is the F-update (rows X, columns Y), side 1 the G-update.
struct Side {
  int64_t n_rows, rows_pad, NT, T, G;
  const float* norms;      // squared norms of the row points
  const float* lw2;        // log2 weights of the row points
  float* pot;              // the potential the pass writes
  const float* col_bias;   // bias of the column points (read)
  float* next_bias;        // bias of the row points, read by the other side's pass
};

// The update schedules (of the method's alternating form, and the averaged symmetric one
// whose two updates both read the previous iterate).
enum Schedule : int {
  kAlternating = 0,  // f = F(g), then g = G(f): a merge and two grid barriers per half-step
  kSymmetric = 1,    // f, g = (old + F(g_old)) / 2, (old + G(f_old)) / 2: both passes, then
                     // one merge of both sides between two grid barriers per iteration
  kSymmetricSelf = 2 // the same with X = Y and a = b started from f = g: one pass per
                     // iteration (g stays equal to f)
};

struct Params {
  Side side[2];
  float2* partial;         // stream-K partials of the current pass, slot * rows_pad + row
  float2* partial_g;       // symmetric: the G-update's partials (the F-update's in partial)
  unsigned* grid_bar;      // arrivals at the grid barriers, over all passes
  unsigned* status;
  // Convergence check (alternating schedule): the merge of pass err_pass (an F-update; -1:
  // none) also writes each row's share of the L1 row-marginal error of the previous
  // iterate into err_rows (weights err_w), as the combine does.
  float* err_rows;
  const float* err_w;
  int64_t err_pass;
  int kc, stages, a_bufs, n_stages, iters_per_stage, schedule;
  float eps[kMaxEps];
};

struct __align__(128) Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t a_full[2];
  uint64_t a_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  // A failed wait in pass p: slot [p % 2][0] for the tiles, [p % 2][1] and [p % 2][2] for
  // the pass's two grid barriers. Each is written in one phase of the pass and read by every
  // epilogue thread after the named barrier that closes that phase; it is next written two
  // passes later, after every thread has read it.
  int epi_abort[2][3];
};

// The 256 epilogue threads (named barrier 1; barrier 0 is __syncthreads).
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Release / acquire at GPU scope in the fence form: fence.acq_rel.gpu before a relaxed
// arrival makes the CTA's earlier writes (ordered before it by the CTA barrier) visible to
// whoever observes the arrival; a relaxed observation followed by fence.acq_rel.gpu makes
// them visible to the observer. (With sc fences around acq_rel atomics the end-of-pass
// counting took about a quarter more cycles.)
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ unsigned atom_add_relaxed_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.relaxed.gpu.global.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Status-word bit set, besides kErrTimeout, when a grid-barrier wait gives up.
constexpr unsigned kErrGridTimeout = 2u;

// The grid barrier's wait: until *bar >= target (relaxed polling, then an acquire fence that
// pairs with the arrivals' release fences); false once limit_ns have passed.
__device__ __forceinline__ bool grid_wait(const unsigned* bar, unsigned target,
                                          uint64_t limit_ns) {
  bool arrived = ld_relaxed_gpu(bar) >= target;
  if (!arrived) {
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 32 && !arrived; ++i) arrived = ld_relaxed_gpu(bar) >= target;
      if (arrived || ptx::globaltimer() - t0 > limit_ns) break;
    }
  }
  fence_acq_rel_gpu();
  return arrived;
}

// This CTA's stream-K range of side s (empty when the side uses fewer CTAs).
__device__ __forceinline__ void cta_range(const Side& S, int64_t cta, int64_t& tb, int64_t& te) {
  if (cta < S.G) {
    tb = sk_begin(cta, S.T, S.G);
    te = sk_begin(cta + 1, S.T, S.G);
  } else {
    tb = te = 0;
  }
}

// Passes of the launch and the side (0: F-update, 1: G-update) of pass p.
__device__ __forceinline__ int64_t pass_count(const Params& P) {
  const int64_t iters = (int64_t)P.n_stages * P.iters_per_stage;
  return P.schedule == kSymmetricSelf ? iters : 2 * iters;
}
__device__ __forceinline__ int pass_side(const Params& P, int64_t p) {
  return P.schedule == kSymmetricSelf ? 0 : (int)(p & 1);
}
__device__ __forceinline__ int64_t pass_iteration(const Params& P, int64_t p) {
  return P.schedule == kSymmetricSelf ? p : p >> 1;
}

// eps of pass p and the ratio eps / eps_next the merge folds into the next bias (the
// alternating G-update at the end of a stage hands over to the next stage's eps).
__device__ __forceinline__ void pass_eps(const Params& P, int64_t p, float& eps,
                                         float& ratio) {
  const int64_t it = pass_iteration(P, p);
  const int st = (int)(it / P.iters_per_stage);
  eps = P.eps[st];
  ratio = 1.0f;
  const bool last_of_stage = (it % P.iters_per_stage) == P.iters_per_stage - 1;
  if (P.schedule == kAlternating && (p & 1) && last_of_stage && st + 1 < P.n_stages)
    ratio = eps / P.eps[st + 1];
}

}  // namespace ssolve

// mapXr / mapYr: the packed clouds as row operands (128-row boxes); mapYc / mapXc: as column
// operands (256-row boxes). Shared memory: the row tile of the current segment (resident, up
// to two buffers), then a ring of 256-row column K-chunks.
template <bool kBF16>
__global__ void __launch_bounds__(ssolve::kThreads, 1)
lse_solve_short_kernel(const __grid_constant__ CUtensorMap mapXr,
                       const __grid_constant__ CUtensorMap mapYc,
                       const __grid_constant__ CUtensorMap mapYr,
                       const __grid_constant__ CUtensorMap mapXc,
                       const __grid_constant__ ssolve::Params P) {
  using namespace ssolve;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctrl ctl;
  // Column biases of each epilogue warp's current and next tile (cp.async, one tile ahead).
  __shared__ __align__(16) float bias_s[kEpiThreads / 32][2][kBN];
  constexpr int kElems = kBF16 ? 64 : 32;  // elements per 128-byte K-chunk row
  constexpr uint32_t kBChunk = 2u * kChunk;  // 256 rows x 128 bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = ptx::smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = dyn_smem + (base - raw);
  const int kc_count = P.kc, stages = P.stages, a_bufs = P.a_bufs;
  const uint32_t a_bytes = (uint32_t)kc_count * kChunk;
  const int64_t cta = blockIdx.x;
  const int64_t n_pass = pass_count(P);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl.acc_full[b], 1);
      ptx::mbar_init(&ctl.acc_empty[b], kEpiThreads / 2);  // the four warps of one parity
      ptx::mbar_init(&ctl.a_full[b], 1);
      ptx::mbar_init(&ctl.a_empty[b], 1);
    }
    ptx::mbar_init(&ctl.mma_done, 1);
    for (int i = 0; i < 6; ++i) (&ctl.epi_abort[0][0])[i] = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&mapXr);
    ptx::tma_prefetch_desc(&mapYc);
    ptx::tma_prefetch_desc(&mapYr);
    ptx::tma_prefetch_desc(&mapXc);
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
      int64_t issued = 0, segs = 0;
      bool ok = true;
      for (int64_t p = 0; ok && p < n_pass; ++p) {
        const int side = pass_side(P, p);
        const Side& S = P.side[side];
        const CUtensorMap* mA = side ? &mapYr : &mapXr;
        const CUtensorMap* mB = side ? &mapXc : &mapYc;
        int64_t tb, te;
        cta_range(S, cta, tb, te);
        for (int64_t t = tb; ok && t < te;) {
          const int64_t rt = t / S.NT;
          const int64_t seg_end = min(te, (rt + 1) * S.NT);
          // segment s uses row-tile buffer s % a_bufs (its (s / a_bufs)-th use)
          const int ab = (int)(segs % a_bufs);
          const uint32_t use = (uint32_t)(segs / a_bufs);
          if (!ptx::mbar_wait(&ctl.a_empty[ab], (use & 1u) ^ 1u)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&ctl.a_full[ab], a_bytes);
          for (int kc = 0; kc < kc_count; ++kc)
            ptx::tma_load_2d(mA, &ctl.a_full[ab], smem + (size_t)ab * a_bytes + (size_t)kc * kChunk,
                             kc * kElems, (int)(rt * kBM));
          ++segs;
          for (int64_t tt = t; ok && tt < seg_end; ++tt) {
            const int jt = (int)(tt - rt * S.NT);
            for (int kc = 0; kc < kc_count; ++kc) {
              if (!ptx::mbar_wait(&ctl.empty[stage], ph ^ 1u)) { ok = false; break; }
              uint8_t* st = smem + (size_t)a_bufs * a_bytes + (size_t)stage * kBChunk;
              ptx::mbar_arrive_expect_tx(&ctl.full[stage], kBChunk);
              ptx::tma_load_2d(mB, &ctl.full[stage], st, kc * kElems, jt * kBN);
              ++issued;
              if (++stage == (uint32_t)stages) { stage = 0; ph ^= 1u; }
            }
          }
          t = seg_end;
        }
      }
      if (!ok) atomicOr(P.status, kErrTimeout);
      // Drain: every copy issued must have landed before the CTA may exit.
      for (int s = 0; s < stages; ++s) {
        const int64_t arms = issued / stages + (s < issued % stages ? 1 : 0);
        if (arms > 0) ptx::mbar_wait(&ctl.full[s], (uint32_t)((arms - 1) & 1));
      }
      for (int b = 0; b < a_bufs; ++b) {
        const int64_t uses = segs / a_bufs + (b < segs % a_bufs ? 1 : 0);
        if (uses > 0) ptx::mbar_wait(&ctl.a_full[b], (uint32_t)((uses - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------- MMA issuer ----------------------------------------
      // Within a pass, tile number l of this CTA's range goes to accumulator l % 2 (the
      // parity of the epilogue warps that read it); each accumulator keeps its own phase.
      constexpr uint32_t idesc = ptx::make_idesc<kBF16>(kBM, kBN);
      uint32_t stage = 0, ph = 0, acc_ph[2] = {0u, 0u};
      int64_t segs = 0;
      bool ok = true;
      for (int64_t p = 0; ok && p < n_pass; ++p) {
        const Side& S = P.side[pass_side(P, p)];
        int64_t tb, te;
        cta_range(S, cta, tb, te);
        for (int64_t t = tb; ok && t < te;) {
          const int64_t rt = t / S.NT;
          const int64_t seg_end = min(te, (rt + 1) * S.NT);
          const int abuf = (int)(segs % a_bufs);
          if (!ptx::mbar_wait(&ctl.a_full[abuf], (uint32_t)((segs / a_bufs) & 1))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          for (int64_t tt = t; ok && tt < seg_end; ++tt) {
            const int ab = (int)((tt - tb) & 1);
            if (!ptx::mbar_wait(&ctl.acc_empty[ab], acc_ph[ab] ^ 1u)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)ab * kBN;
            for (int kc = 0; kc < kc_count; ++kc) {
              if (!ptx::mbar_wait(&ctl.full[stage], ph)) { ok = false; break; }
              ptx::tc_fence_after();
              const uint32_t st = base + (uint32_t)a_bufs * a_bytes + stage * kBChunk;
              const uint64_t a_desc =
                  ptx::sdesc_k128(base + (uint32_t)abuf * a_bytes + (uint32_t)kc * kChunk);
              const uint64_t b_desc = ptx::sdesc_k128(st);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // K advance: 32 bytes = 2 in the address field
                ptx::umma<kBF16>(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                                 (kc | kk) != 0 ? 1u : 0u);
              ptx::umma_commit(&ctl.empty[stage]);
              if (++stage == (uint32_t)stages) { stage = 0; ph ^= 1u; }
            }
            if (!ok) break;
            ptx::umma_commit(&ctl.acc_full[ab]);
            acc_ph[ab] ^= 1u;
          }
          ptx::umma_commit(&ctl.a_empty[abuf]);
          ++segs;
          t = seg_end;
        }
      }
      if (!ok) atomicOr(P.status, kErrTimeout);
      // Every MMA issued must have retired before Tensor Memory is released.
      ptx::umma_commit(&ctl.mma_done);
      ptx::mbar_wait(&ctl.mma_done, 0);
    }
  } else {
    // --------------------------------- epilogue ------------------------------------------
    // Warp w reads TMEM lane quarter (w % 4) (rows 32q .. 32q+31); the warps of parity
    // par = (w - 2) / 4 take tiles l = par, par + 2, ... of each pass's range (all 256
    // columns) from accumulator par, so the two warps of a sub-partition interleave their
    // SFU bursts. Each (row, parity) keeps one online (max, sum) per row-tile segment, written
    // to its partial slot. Every epilogue warp passes the same sequence of named barriers,
    // also on the error path (a failed wait is noted in a per-pass flag that all warps read
    // after a barrier), so no warp is left waiting on one.
    const int q = warp & 3;
    const int par = (warp - 2) >> 2;
    const int etid = (int)threadIdx.x - 64;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float (*bslot)[kBN] = bias_s[warp - 2];
    uint32_t acc_ph = 0;
    int bs = 0;
    bool ok = true;
    // Grid barrier among all CTAs' epilogues (thread 0 of the epilogue arrives and waits;
    // the named barriers around it order the other epilogue threads' writes before the
    // arrival and their later reads after the wait). On time-out the pass's abort flag is
    // set, which every epilogue thread reads after the closing named barrier.
    unsigned barriers = 0;  // grid barriers passed so far
    auto grid_barrier = [&](int& abort_flag) {
      const unsigned target = ++barriers * gridDim.x;
      if (etid == 0) {
        fence_acq_rel_gpu();
        atom_add_relaxed_gpu(P.grid_bar, 1u);
        if (!grid_wait(P.grid_bar, target, ptx::kWaitLimitNs)) {
          atomicOr(P.status, kErrTimeout | kErrGridTimeout);
          abort_flag = 1;
        }
      }
      epi_sync();
    };
    for (int64_t p = 0; p < n_pass; ++p) {
      const int side = pass_side(P, p);
      const Side& S = P.side[side];
      // this pass's partials: the symmetric G-update keeps its own, since the F-update's
      // are merged only after it
      float2* const partial = (P.schedule == kSymmetric && side == 1) ? P.partial_g : P.partial;
      float eps, ratio;
      pass_eps(P, p, eps, ratio);
      const float kappa = 2.0f * kLog2e / eps;
      const int64_t NT = S.NT;
      int64_t tb, te;
      cta_range(S, cta, tb, te);
      // The warp's 256 biases of a tile (1 KB, 32 bytes per lane) are copied global -> shared
      // with cp.async (L2 only: the biases were written by other CTAs) into one of two slots.
      auto stage_bias = [&](int64_t tile, int slot) {
        const float* src = S.col_bias + (tile % NT) * kBN + lane * 4;
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
      if (tb + par < te) stage_bias(tb + par, bs);
      for (int64_t t = tb; ok && t < te;) {
        const int64_t rt = t / NT;
        const int64_t seg_end = min(te, (rt + 1) * NT);
        float M = kNegBig, Ssum = 0.0f;
        // this warp's first tile of the segment: (tt - tb) % 2 == par
        for (int64_t tt = t + (((t - tb) & 1) != par ? 1 : 0); tt < seg_end; tt += 2) {
          if (tt + 2 < te) {
            stage_bias(tt + 2, bs ^ 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
          } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
          }
          __syncwarp();
          const float4* cb = reinterpret_cast<const float4*>(bslot[bs]);
          const bool got = ptx::mbar_wait(&ctl.acc_full[par], acc_ph);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t taddr = tmem + lane_base + (uint32_t)par * kBN;
          float v[64];
#pragma unroll 1
          for (int c = 0; c < 3; ++c) {
            ptx::tmem_ld_x64_sync(taddr + c * 64, v);
            lse_chunk<64, false>(v, cb + c * 16, kappa, M, Ssum);
          }
          ptx::tmem_ld_x64_sync(taddr + 192, v);
          ptx::tc_fence_before();
          ptx::mbar_arrive(&ctl.acc_empty[par]);   // this warp's part of the tile is read
          acc_ph ^= 1u;
          lse_chunk<64, false>(v, cb + 48, kappa, M, Ssum);
          __syncwarp();  // every lane is done with bslot[bs] before it is refilled
          bs ^= 1;
        }
        if (!ok) break;
        const int64_t row = rt * kBM + q * 32 + lane;
        const int64_t slot = 2 * (cta - sk_owner(rt * NT, S.T, S.G)) + par;
        if (row < S.n_rows) partial[slot * S.rows_pad + row] = make_float2(M, Ssum);
        t = seg_end;
      }
      asm volatile("cp.async.wait_group 0;" ::: "memory");

      // ---- end of the pass ----------------------------------------------------------------
      // A failed wait anywhere ends the solve at the next check: every epilogue warp reads
      // the pass's abort flag after the same named barrier.
      int* abort_flags = ctl.epi_abort[p & 1];
      if (!ok) abort_flags[0] = 1;
      epi_sync();
      if (abort_flags[0]) break;
      // the symmetric F-update's partials wait for the G-update's: both read the previous
      // iterate, and both merge after the G-update's pass
      if (P.schedule == kSymmetric && side == 0) continue;
      // (1) barrier: every CTA's partials of this pass (symmetric: of both passes) are written
      grid_barrier(abort_flags[1]);
      if (abort_flags[1]) break;
      // (2) merge: this CTA's equal share of the rows, partials read from L2 in fixed slot
      // order; new potential and next bias of each row
      if (P.schedule == kAlternating) {
        CombineArgs args;
        args.rows = S.n_rows;
        args.rows_pad = S.rows_pad;
        args.norms = S.norms;
        args.eps = eps;
        args.lw2 = S.lw2;
        args.eps_ratio = ratio;
        args.out_pot = S.pot;
        args.next_bias = S.next_bias;
        args.out_lse2 = nullptr;
        args.average = 0;
        args.err_w = p == P.err_pass ? P.err_w : nullptr;
        args.err_rows = p == P.err_pass ? P.err_rows : nullptr;
        const SplitInfo split{0, 2, S.T, S.G, NT, kBM};
        const int64_t share = (S.rows_pad + gridDim.x - 1) / gridDim.x;
        const int64_t r_end = min(S.rows_pad, (cta + 1) * share);
        for (int64_t r = cta * share + etid; r < r_end; r += kEpiThreads)
          combine_row<true>(P.partial, S.rows_pad, split, r, args);
      } else {
        // Symmetric: each side's potential averaged with its previous value, then the bias
        // the next iteration reads, from the averaged potentials at that iteration's eps
        // ((pot - norm) log2e / eps + log2 w; -inf on padding rows). The self-transport
        // problem's single pass also provides the G-side bias (its g equals f).
        const int64_t it = pass_iteration(P, p);
        const int64_t n_iters = (int64_t)P.n_stages * P.iters_per_stage;
        const bool more = it + 1 < n_iters;
        const float inv_eps_log2e =
            more ? kLog2e / P.eps[(int)((it + 1) / P.iters_per_stage)] : 0.0f;
        for (int t = 0; t < (P.schedule == kSymmetric ? 2 : 1); ++t) {
          const Side& U = P.side[t];
          const Side& B = P.schedule == kSymmetric ? U : P.side[1];  // whose bias is written
          CombineArgs args;
          args.rows = U.n_rows;
          args.rows_pad = U.rows_pad;
          args.norms = U.norms;
          args.eps = eps;
          args.lw2 = U.lw2;
          args.eps_ratio = 1.0f;
          args.out_pot = U.pot;
          args.next_bias = nullptr;
          args.out_lse2 = nullptr;
          args.average = 1;
          args.err_w = nullptr;
          args.err_rows = nullptr;
          const SplitInfo split{0, 2, U.T, U.G, U.NT, kBM};
          float2* const part = t == 1 ? P.partial_g : P.partial;
          const int64_t share = (U.rows_pad + gridDim.x - 1) / gridDim.x;
          const int64_t r_end = min(U.rows_pad, (cta + 1) * share);
          for (int64_t r = cta * share + etid; r < r_end; r += kEpiThreads) {
            combine_row<true>(part, U.rows_pad, split, r, args);
            if (more)
              B.next_bias[r] =
                  r < U.n_rows ? (U.pot[r] - B.norms[r]) * inv_eps_log2e + B.lw2[r] : neg_inf();
          }
        }
      }
      epi_sync();
      // (3) barrier: every merge is visible before any CTA reads the new biases
      grid_barrier(abort_flags[2]);
      if (abort_flags[2]) break;
    }
    if (!ok) atomicOr(P.status, kErrTimeout);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Self-test of the grid barrier's bounded wait: one thread waits for a word that nothing
// writes to reach 1, gives up after limit_ns and records it in the status word.
__global__ void grid_wait_selftest_kernel(const unsigned* __restrict__ word, uint64_t limit_ns,
                                          unsigned* __restrict__ status) {
  if (threadIdx.x == 0 && !ssolve::grid_wait(word, 1u, limit_ns))
    atomicOr(status, kErrTimeout | ssolve::kErrGridTimeout);
}

namespace {

// Shared memory of the persistent kernel, planned as for the per-pass short kernel: the
// resident row tile (two buffers when at least four column stages still fit beside them),
// then as many 256-row column K-chunk stages as fit (at least two).
bool smem_plan(int kc, int* dyn, int* stages, int* a_bufs) {
  const int ctrl = (int)sizeof(ssolve::Ctrl) + ssolve::kEpiThreads / 32 * 2 * ssolve::kBN * 4;
  const int a_bytes = kc * ssolve::kChunk;
  const int stage_bytes = 2 * ssolve::kChunk;
  const int ab =
      (ssolve::kSmemLimit - ctrl - 1024 - 2 * a_bytes) / stage_bytes >= 4 ? 2 : 1;
  const int budget = ssolve::kSmemLimit - ctrl - 1024 - ab * a_bytes;
  const int st = std::min(ssolve::kMaxStages, budget / stage_bytes);
  if (st < 2) return false;
  *dyn = ab * a_bytes + st * stage_bytes + 1024;
  *stages = st;
  *a_bufs = ab;
  return true;
}

}  // namespace
}  // namespace tc

int tc_selftest_grid_wait(unsigned* status, unsigned* word, int64_t limit_ns, cudaStream_t st) {
  if (cudaMemsetAsync(word, 0, sizeof(unsigned), st) != cudaSuccess) return FLASHOT_ERR_CUDA;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
    tc::grid_wait_selftest_kernel<<<1, 32, 0, st>>>(word, (uint64_t)limit_ns, status);
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

size_t tc_short_solve_sync_bytes(int64_t n_pad, int64_t m_pad) {
  // the grid barrier's word, on a 128-byte line of its own
  (void)n_pad;
  (void)m_pad;
  return 32 * sizeof(unsigned);
}

int tc_short_solve(bool bf16, const void* xq, const void* yq, int64_t n, int64_t m,
                   int64_t n_pad, int64_t m_pad, int64_t dpt, const float* alpha,
                   const float* beta, const float* la2, const float* lb2, float* biasF,
                   float* biasG, float* f, float* g, const float* eps_sched, int n_stages,
                   int iters_per_stage, int schedule, float* err_rows, const float* err_w,
                   int err_iter, float2* partial, size_t partial_bytes, int max_splits,
                   void* sync_words, size_t sync_bytes, int sms, unsigned* status,
                   cudaStream_t st) {
  using namespace tc;
  using namespace tc::ssolve;
  // FLASHOT_SHORT_SOLVE in the environment: 0 keeps the per-pass path, 1 takes the
  // persistent solve whenever it applies; unset, it is taken when the CTAs average at least
  // 1.5 tiles per pass on both sides (with one each, the two grid barriers and the merge
  // cost more than the launches they replace: measured 21-34 % slower at 512^2 to 2048^2,
  // one tile per CTA, and 11-28 % faster at 3072^2 and 4096^2, 1.9 and 3.4 tiles per CTA,
  // 2-10 % from 6144^2, d = 16..128).
  static const int mode = [] {
    const char* e = std::getenv("FLASHOT_SHORT_SOLVE");
    return e && e[0] == '0' ? 0 : (e && e[0] == '1' ? 1 : 2);
  }();
  const bool enabled = mode != 0;
  const int es = bf16 ? 2 : 4;
  const int kc = (int)(dpt * es / 128);
  if (!enabled || kc < 1 || kc > kMaxKc || n_stages < 1 || n_stages > kMaxEps ||
      iters_per_stage < 1 || n_pad % 256 != 0 || m_pad % 256 != 0 ||
      tc_short_solve_sync_bytes(n_pad, m_pad) > sync_bytes)
    return FLASHOT_ERR_NOT_IMPLEMENTED;
  int dyn = 0, stages = 0, a_bufs = 0;
  if (!smem_plan(kc, &dyn, &stages, &a_bufs)) return FLASHOT_ERR_NOT_IMPLEMENTED;
  const int64_t rtX = n_pad / kBM, rtY = m_pad / kBM, NTX = n_pad / kBN, NTY = m_pad / kBN;
  // The per-pass path's stream-K grids, so that tiles, ranges and partial slots coincide.
  const int64_t GF = choose_grid(rtX, NTY, sms, max_splits / 2);
  const int64_t GG = choose_grid(rtY, NTX, sms, max_splits / 2);
  const int64_t grid = std::max(GF, GG);
  if (mode == 2 && (2 * rtX * NTY < 3 * GF || 2 * rtY * NTX < 3 * GG))
    return FLASHOT_ERR_NOT_IMPLEMENTED;
  if (schedule < kAlternating || schedule > kSymmetricSelf) return FLASHOT_ERR_INVALID_ARG;
  const int64_t iters = (int64_t)n_stages * iters_per_stage;
  const int64_t barriers = 2 * (schedule == kAlternating ? 2 * iters : iters);
  if (barriers * grid >= (1LL << 31)) return FLASHOT_ERR_NOT_IMPLEMENTED;
  // Partial slots: two per owning CTA and row tile. The symmetric G-update keeps its own
  // region after the F-update's.
  auto max_slots = [](int64_t row_tiles, int64_t NT, int64_t G) {
    const int64_t T = row_tiles * NT;
    int64_t worst = 1;
    for (int64_t rt = 0; rt < row_tiles; ++rt)
      worst = std::max(worst, sk_owner((rt + 1) * NT - 1, T, G) - sk_owner(rt * NT, T, G) + 1);
    return 2 * worst;
  };
  const int64_t f_region = max_slots(rtX, NTY, GF) * n_pad;
  float2* const partial_g = partial + f_region;
  if (schedule == kSymmetric &&
      (size_t)(f_region + max_slots(rtY, NTX, GG) * m_pad) * sizeof(float2) > partial_bytes)
    return FLASHOT_ERR_NOT_IMPLEMENTED;
  auto kern = bf16 ? lse_solve_short_kernel<true> : lse_solve_short_kernel<false>;
  if (set_smem(kern, dyn) != FLASHOT_OK) return FLASHOT_ERR_CUDA;
  // Every CTA must be resident at once (the grid barrier); the cooperative launch checks it
  // too, this only avoids asking for a launch that would be refused.
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, (size_t)dyn) !=
      cudaSuccess) {
    cudaGetLastError();
    return FLASHOT_ERR_NOT_IMPLEMENTED;
  }
  if ((int64_t)per_sm * sms < grid) return FLASHOT_ERR_NOT_IMPLEMENTED;
  CUtensorMap mXr, mYc, mYr, mXc;
  int rc = make_map(&mXr, xq, n_pad, dpt, bf16);
  if (rc == FLASHOT_OK) rc = make_map_rows(&mYc, yq, m_pad, dpt, bf16, kBN);
  if (rc == FLASHOT_OK) rc = make_map(&mYr, yq, m_pad, dpt, bf16);
  if (rc == FLASHOT_OK) rc = make_map_rows(&mXc, xq, n_pad, dpt, bf16, kBN);
  if (rc != FLASHOT_OK) return rc;
  unsigned* words = static_cast<unsigned*>(sync_words);
  Params P = {};
  P.side[0] = Side{n, n_pad, NTY, rtX * NTY, GF, alpha, la2, f, biasF, biasG};
  P.side[1] = Side{m, m_pad, NTX, rtY * NTX, GG, beta, lb2, g, biasG, biasF};
  P.partial = partial;
  P.partial_g = partial_g;
  P.schedule = schedule;
  P.err_rows = err_rows;
  P.err_w = err_w;
  P.err_pass = (schedule == kAlternating && err_rows != nullptr && err_iter >= 0) ? 2LL * err_iter
                                                                                 : -1;
  P.grid_bar = words;
  P.status = status;
  P.kc = kc;
  P.stages = stages;
  P.a_bufs = a_bufs;
  P.n_stages = n_stages;
  P.iters_per_stage = iters_per_stage;
  for (int s = 0; s < n_stages; ++s) P.eps[s] = eps_sched[s];
  if (cudaMemsetAsync(sync_words, 0, tc_short_solve_sync_bytes(n_pad, m_pad), st) !=
      cudaSuccess)
    return FLASHOT_ERR_CUDA;
  {
    TraceScope ts_(FLASHOT_KERNEL_LSE, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mXr, mYc, mYr, mXc, P);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
      // fewer SMs free for co-residency than the occupancy query promised: the per-pass
      // path runs instead (the barrier word zeroed above is not read by it)
      cudaGetLastError();
      return FLASHOT_ERR_NOT_IMPLEMENTED;
    }
    if (e != cudaSuccess) return FLASHOT_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

}  // namespace flashot
