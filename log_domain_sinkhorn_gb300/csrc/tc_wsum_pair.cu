// tc_wsum_pair.cu -- tensor-core weighted-sum passes on CTA pairs: transport application
// P V / P^T U, the barycentric gradient and the Hadamard-weighted transport (FlashSinkhorn:
// IO-Aware Entropic Optimal Transport on GPU, SAI replication review, "Summary" (i)-(ii)),
// in bf16, tf32 and split tf32.
//
// Two CTAs of a cluster own a unit of 256 rows (128 each) x 256 columns. Per unit:
//   S   = rows * cols^T                 tcgen05.mma.cta_group::2, M = 256, N = 256, into each
//                                       CTA's Tensor Memory (its 128 rows), K-chunks of both
//                                       operands streamed by TMA (each CTA loads its own 128
//                                       rows and half of the 256 column points)
//   w_ij = exp2(kappa S_ij + colBias_j + rowBias_i)        8 epilogue warps per CTA
//   O  += W * V^T-tile                  second cta_group::2 MMA, A = W from Tensor Memory,
//                                       B = V^T tile (each CTA holds half of its kKV rows)
// W in Tensor Memory:
//   bf16        bf16 pairs in columns [256, 384); S stays in [0, 256), so the S MMA of the
//               next unit runs while the epilogue turns this unit's S into W.
//   tf32        W is rounded to tf32 and written over S in [0, 256) (one element per
//               column), so the next S MMA is issued after this unit's W V MMA.
//   split tf32  the same W_hi = tf32(W) over S, plus W_lo = bf16(W - W_hi) as bf16 pairs in
//               [384, 512); O = W_hi V_hi + W_hi V_lo (tf32, V = V_hi + V_lo) + W_lo bf16(V)
//               (bf16): the weights and V both enter with about fp32 accuracy, the dropped
//               W_lo V_lo term is ~2^-22 relative.
// The weights are plan entries (or a_i times softmax weights), all <= 1: no running max.
//
// Work split: units (output-column group, 256-row pair tile, column tile) are cut into
// contiguous ranges per CTA pair (stream-K); each CTA writes per pair tile it touched a
// partial O (its 128 rows x kKV) and per-row (sum w, sum w S) per column half, and
// wsum_pair_reduce_kernel adds the partials in a fixed order and finishes the output.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cstdlib>

#include "flashot.h"
#include "common.cuh"
#include "pack_kernels.cuh"
#include "ptx.cuh"
#include "ptx_wsum.cuh"
#include "tc_api.h"
#include "tc_host.h"
#include "tc_wsum_pair.h"
#include "trace.h"

namespace flashot {
namespace tcp {

constexpr int kBM = 128;           // rows per CTA (the pair tile has 256)
constexpr int kSBN = 256;          // columns per unit (S MMA N)
constexpr int kChunk = 128 * 128;  // one 128-row x 128-byte K-chunk box
constexpr int kThreads = 320;      // TMA warp, MMA warp, 8 epilogue warps
constexpr int kEpiWarps = 8;
constexpr int kMaxStages = 6;
constexpr int kMaxOwners = 4;      // partial slots per (group, pair tile)
constexpr int kSmemLimit = 232448;

enum : int { kPrecBF16 = 0, kPrecTF32 = 1, kPrecSplit = 2 };

struct __align__(128) PCtrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t s_full, s_empty, w_full, w_empty, v_full, v_empty, o_full, o_empty, mma_done;
  uint64_t w_read;  // tf32 / split: the W V MMA of a unit has completed (W may be overwritten)
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void flag_error(PCtrl& ctl, unsigned* status) {
  atomicOr(status, kErrTimeout);
  ctl.abort_flag = 1;
}

// Parity of the n-th completion (0-based) of a barrier that is waited on by its consumer.
__device__ __forceinline__ uint32_t par(int64_t n) { return (uint32_t)(n & 1); }

// Shape of the V^T operand of one unit, per CTA: kKV / 2 rows (output columns) x 256 K.
// The segments a pair walks, each a run of consecutive units of one row group (one output
// group and pair tile), and the partial slot each writes:
//   run_len == 0: the pair's stream-K range, in SegOrder's order, slot = the pair's rank
//                 among the row group's owners;
//   run_len > 0:  round-robin runs of run_len column tiles: run r = pair + i G covers row
//                 group r / R and column tiles (r % R) run_len .. + run_len (R runs per row
//                 group), slot = r % R. At any moment the pairs then work on a few row
//                 groups, several pairs on each, all at the same column offsets of their
//                 runs, so the row and column tiles in use fit in L2 even when the pairs'
//                 row tiles alone would not (split tf32 at large d).
struct Walk {
  SegOrder so;
  int64_t pair, G, NT, L, R, n;
  __device__ __forceinline__ Walk(int64_t pair_, int64_t G_, int64_t T, int64_t NT_,
                                  int64_t run_len)
      : so(sk_begin(pair_, T, G_), sk_begin(pair_ + 1, T, G_), NT_), pair(pair_), G(G_),
        NT(NT_), L(run_len), R(run_len > 0 ? (NT_ + run_len - 1) / run_len : 1), n(0) {
    if (L == 0) {
      n = so.n;
    } else {
      const int64_t runs = (T / NT) * R;
      n = runs > pair ? (runs - pair + G - 1) / G : 0;
    }
  }
  __device__ __forceinline__ void get(int64_t i, int64_t& a, int64_t& b) const {
    if (L == 0) {
      so.get(i, a, b);
      return;
    }
    const int64_t r = pair + i * G, vr = r / R, k = r - vr * R;
    a = vr * NT + k * L;
    b = vr * NT + min(NT, (k + 1) * L);
  }
  // Partial slot of the segment that starts at unit a (row group vr).
  __device__ __forceinline__ int64_t slot(int64_t a, int64_t vr, int64_t T) const {
    return L == 0 ? pair - sk_owner(vr * NT, T, G) : (a - vr * NT) / L;
  }
};

template <int kPrec, int kKV>
struct VShape {
  static constexpr int rows = kKV / 2;                       // per CTA
  static constexpr uint32_t chunk = (uint32_t)rows * 128u;   // one 128-byte K-chunk box
  // K-chunks per unit: bf16 256 x 2 B / 128 = 4; tf32 8; split: 8 (hi) + 8 (lo) + 4 (bf16)
  static constexpr int chunks_main = kPrec == kPrecBF16 ? 4 : 8;
  static constexpr int chunks_total = kPrec == kPrecSplit ? 20 : chunks_main;
  static constexpr uint32_t bytes = kKV == 0 ? 0u : (uint32_t)chunks_total * chunk;
};

template <int kPrec, int kKV>  // kKV: output columns per group (64 or 128); 0 = Hadamard
__global__ void __launch_bounds__(kThreads, 1)
wsum_pair_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                 const __grid_constant__ CUtensorMap mapV,
                 const __grid_constant__ CUtensorMap mapVlo,
                 const __grid_constant__ CUtensorMap mapVb, const float* __restrict__ colBias,
                 const float* __restrict__ rowBias, int64_t n_rows, int64_t pair_tiles,
                 int64_t NT, int64_t T, int64_t run_len, int kc_count, int kps, int n_st,
                 float kappa,
                 float* __restrict__ pO, float2* __restrict__ pW, int64_t ldp,
                 unsigned* __restrict__ status) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ PCtrl ctl;
  constexpr bool kHad = (kKV == 0);
  constexpr bool kBf = (kPrec == kPrecBF16);
  constexpr bool kSplitW = (kPrec == kPrecSplit);
  // W overwrites S in tensor memory (tf32, split): the next S MMA waits for this unit's W V.
  // bf16 with 256 output columns per group (wide outputs such as the gradient): O needs
  // [256, 512), so W (bf16 pairs) is written over S as well.
  constexpr bool kWide = kBf && kKV == 256;
  constexpr bool kAlias = (!kBf || kWide) && !kHad;
  // Split tf32: each unit's W V lands in a fresh tensor-memory accumulator that the epilogue
  // adds into fp32 registers (round to nearest), so no accumulation chain in the tensor core
  // is longer than one unit's K = 256 (x 3 terms); long in-tensor-memory chains over a whole
  // row (20k terms) measured a ~1e-4 relative error against the fp64 oracle.
  constexpr bool kPromote = kSplitW;
  constexpr int kElems = kBf ? 64 : 32;  // K elements per 128-byte chunk of the S operands
  using VS = VShape<kPrec, kKV>;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kTmemW = (kBf && !kWide) ? 256u : 0u;  // W (bf16 pairs) or W_hi (over S)
  constexpr uint32_t kTmemO = (kBf && !kWide) ? 384u : 256u;
  constexpr uint32_t kTmemWL = 384u;            // W_lo bf16 pairs (split)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: the pair's MMA issuer
  const uint32_t raw = ptx::smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = dyn_smem + (base - raw);
  constexpr uint32_t kChunkBytes = 2u * kChunk;  // A chunk + B half chunk
  const uint32_t stage_bytes = (uint32_t)kps * kChunkBytes;
  const uint32_t v_base = (uint32_t)n_st * stage_bytes;
  const int64_t G = gridDim.x / 2, pair = blockIdx.x / 2;
  const Walk so(pair, G, T, NT, run_len);  // every role walks the segments in this order
  auto leader = [&](uint64_t* bar) { return ptx::mapa_shared(ptx::smem_u32(bar), 0u); };
  // Barriers that the odd CTA's epilogue arrivals reach through a forwarder: local count 8,
  // plus the forwarder's one arrival in the even CTA.
  const uint32_t fwd_count = kEpiWarps + (rank == 0 ? 1u : 0u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < n_st; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    ptx::mbar_init(&ctl.s_full, 1);
    ptx::mbar_init(&ctl.s_empty, fwd_count);
    ptx::mbar_init(&ctl.w_full, fwd_count);
    ptx::mbar_init(&ctl.w_empty, 1);
    ptx::mbar_init(&ctl.v_full, 1);
    ptx::mbar_init(&ctl.v_empty, 1);
    ptx::mbar_init(&ctl.o_full, 1);
    ptx::mbar_init(&ctl.o_empty, fwd_count);
    ptx::mbar_init(&ctl.mma_done, 1);
    ptx::mbar_init(&ctl.w_read, 1);
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&mapA);
    ptx::tma_prefetch_desc(&mapB);
    if constexpr (!kHad) ptx::tma_prefetch_desc(&mapV);
    if constexpr (kSplitW) {
      ptx::tma_prefetch_desc(&mapVlo);
      ptx::tma_prefetch_desc(&mapVb);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&ctl.tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' barriers initialised and Tensor Memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ----------------------------- S operand producer ---------------------------------
      uint32_t stage = 0, ph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < so.n; ++i) {
       int64_t ta, tb;
       so.get(i, ta, tb);
       for (int64_t t = ta; ok && t < tb; ++t) {
        const int64_t vr = t / NT;
        const int64_t jt = t - vr * NT;
        const int64_t rp = vr % pair_tiles;
        const int row0 = (int)(rp * 2 * kBM + rank * kBM);
        const int col0 = (int)(jt * kSBN + rank * kBM);
        for (int kc = 0; kc < kc_count; kc += kps) {
          if (!ptx::mbar_wait(&ctl.empty[stage], ph ^ 1u)) { ok = false; break; }
          uint8_t* st = smem + (size_t)stage * stage_bytes;
          if (rank == 0) ptx::mbar_arrive_expect_tx(&ctl.full[stage], 2u * stage_bytes);
          const uint32_t bar = leader(&ctl.full[stage]);
          for (int c2 = 0; c2 < kps; ++c2) {
            uint8_t* cst = st + (size_t)c2 * kChunkBytes;
            ptx::tma_load_2d_pair(&mapA, bar, cst, (kc + c2) * kElems, row0);
            ptx::tma_load_2d_pair(&mapB, bar, cst + kChunk, (kc + c2) * kElems, col0);
          }
          ++issued;
          if (++stage == (uint32_t)n_st) { stage = 0; ph ^= 1u; }
        }
       }
      }
      if (!ok) flag_error(ctl, status);
      if (rank == 0)  // drain: every copy of both CTAs counted on these barriers has landed
        for (int s = 0; s < n_st; ++s) {
          const int64_t arms = issued / n_st + (s < issued % n_st ? 1 : 0);
          if (arms > 0) ptx::mbar_wait(&ctl.full[s], par(arms - 1));
        }
    } else if (lane == 1 && !kHad) {
      // ------------------------------ V^T tile producer ---------------------------------
      // A separate thread, so that waiting for the V buffer never holds back the S operands.
      int64_t v_issued = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < so.n; ++i) {
       int64_t ta, tb;
       so.get(i, ta, tb);
       for (int64_t t = ta; t < tb; ++t) {
        const int64_t vr = t / NT;
        const int64_t jt = t - vr * NT;
        const int64_t grp = vr / pair_tiles;
        const int vrow = (int)(grp * kKV + rank * VS::rows);
        if (!ptx::mbar_wait(&ctl.v_empty, par(v_issued) ^ 1u)) { ok = false; break; }
        if (rank == 0) ptx::mbar_arrive_expect_tx(&ctl.v_full, 2u * VS::bytes);
        const uint32_t bar = leader(&ctl.v_full);
        for (int vc = 0; vc < VS::chunks_main; ++vc)
          ptx::tma_load_2d_pair(&mapV, bar, smem + v_base + (size_t)vc * VS::chunk,
                                (int)(jt * kSBN) + vc * (kBf ? 64 : 32), vrow);
        if constexpr (kSplitW) {
          for (int vc = 0; vc < 8; ++vc)
            ptx::tma_load_2d_pair(&mapVlo, bar, smem + v_base + (size_t)(8 + vc) * VS::chunk,
                                  (int)(jt * kSBN) + vc * 32, vrow);
          for (int vc = 0; vc < 4; ++vc)
            ptx::tma_load_2d_pair(&mapVb, bar, smem + v_base + (size_t)(16 + vc) * VS::chunk,
                                  (int)(jt * kSBN) + vc * 64, vrow);
        }
        ++v_issued;
       }
      }
      if (!ok) flag_error(ctl, status);
      if (rank == 0 && v_issued > 0) ptx::mbar_wait(&ctl.v_full, par(v_issued - 1));
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------- MMA issuer ----------------------------------------
      constexpr uint32_t idesc_s = ptx::make_idesc<kBf>(2 * kBM, kSBN);
      constexpr uint32_t idesc_o = ptx::make_idesc<kBf>(2 * kBM, kHad ? 64 : kKV);
      constexpr uint32_t idesc_ob = ptx::make_idesc<true>(2 * kBM, kHad ? 64 : kKV);
      uint32_t stage = 0, ph = 0;
      int64_t s_uses = 0, w_uses = 0, segs = 0;
      bool ok = true;
      // S(u): the K loop of one unit into TMEM [0, 256).
      auto issue_s = [&]() -> bool {
        for (int kc = 0; kc < kc_count; kc += kps) {
          if (!ptx::mbar_wait(&ctl.full[stage], ph)) return false;
          ptx::tc_fence_after();
          const uint32_t st = base + stage * stage_bytes;
          for (int c2 = 0; c2 < kps; ++c2) {
            const uint64_t a_desc = ptx::sdesc_k128(st + (uint32_t)c2 * kChunkBytes);
            const uint64_t b_desc = ptx::sdesc_k128(st + (uint32_t)c2 * kChunkBytes + kChunk);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K advance: 32 bytes = 2 in the address field
              ptx::umma_pair<kBf>(tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc_s,
                                  (kc | c2 | kk) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_pair(&ctl.empty[stage], 0x3);
          if (++stage == (uint32_t)n_st) { stage = 0; ph ^= 1u; }
        }
        ptx::umma_commit_pair(&ctl.s_full, 0x3);
        ++s_uses;
        return true;
      };
      // O += W(u) V(u)^T; `first`: the segment's first unit (overwrite O).
      auto issue_o = [&](bool first) -> bool {
        if constexpr (kPromote) {
          // the epilogue has read the previous unit's O (one o_empty completion per unit)
          if (!ptx::mbar_wait_cluster(&ctl.o_empty, par(w_uses) ^ 1u)) return false;
        } else {
          if (first && !ptx::mbar_wait_cluster(&ctl.o_empty, par(segs) ^ 1u)) return false;
        }
        if (!ptx::mbar_wait_cluster(&ctl.w_full, par(w_uses))) return false;
        if (!ptx::mbar_wait(&ctl.v_full, par(w_uses))) return false;
        ptx::tc_fence_after();
        const uint32_t vb = base + v_base;
        // K = 256 in steps of 16 (bf16) or 8 (tf32); each step is 8 W columns in TMEM and
        // 32 bytes inside a 128-byte V chunk.
#pragma unroll
        for (int vc = 0; vc < VS::chunks_main; ++vc) {
          const uint64_t v_desc = ptx::sdesc_k128(vb + (uint32_t)vc * VS::chunk);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // wide bf16: warp half h wrote its 64 pair-columns (K = 128h .. 128h + 127) at
            // column 128h, so K >= 128 starts at column 128
            const uint32_t wcol = kWide ? (uint32_t)((vc >> 1) * 128 + ((vc & 1) * 4 + kk) * 8)
                                        : (uint32_t)(vc * 4 + kk) * 8u;
            ptx::umma_pair_ts<kBf>(tmem + kTmemO, tmem + kTmemW + wcol, v_desc + 2u * kk, idesc_o,
                                   ((!first && !kPromote) || vc > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if constexpr (kSplitW) {
#pragma unroll
          for (int vc = 0; vc < 8; ++vc) {  // W_hi V_lo
            const uint64_t v_desc = ptx::sdesc_k128(vb + (uint32_t)(8 + vc) * VS::chunk);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::umma_pair_ts<false>(tmem + kTmemO, tmem + kTmemW + (uint32_t)(vc * 4 + kk) * 8u,
                                       v_desc + 2u * kk, idesc_o, 1u);
          }
#pragma unroll
          for (int vc = 0; vc < 4; ++vc) {  // W_lo bf16(V)
            const uint64_t v_desc = ptx::sdesc_k128(vb + (uint32_t)(16 + vc) * VS::chunk);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::umma_pair_ts<true>(tmem + kTmemO, tmem + kTmemWL + (uint32_t)(vc * 4 + kk) * 8u,
                                      v_desc + 2u * kk, idesc_ob, 1u);
          }
        }
        ptx::umma_commit_pair(&ctl.v_empty, 0x3);
        if constexpr (kBf) ptx::umma_commit_pair(&ctl.w_empty, 0x3);
        ++w_uses;
        return true;
      };
      for (int64_t i = 0; ok && i < so.n; ++i) {
        int64_t t, seg_end;
        so.get(i, t, seg_end);
        const int64_t L = seg_end - t;
        if constexpr (kAlias) {
          // S(u), then (once the epilogue has written W(u) over it) O(u), then S(u + 1),
          // which overwrites W(u): it is issued only after O(u) has completed.
          for (int64_t u = 0; ok && u < L; ++u) {
            if (!issue_s() || !issue_o(u == 0)) {
              ok = false;
              break;
            }
            ptx::umma_commit_pair(&ctl.w_read, 0x1);
            if (!ptx::mbar_wait(&ctl.w_read, par(w_uses - 1))) ok = false;
          }
        } else {
          // S(u + 1) runs while the epilogue turns S(u) into W(u); O(u) after it.
          for (int64_t u = 0; ok && u <= L; ++u) {
            if (u < L) {
              if (!ptx::mbar_wait_cluster(&ctl.s_empty, par(s_uses) ^ 1u) || !issue_s()) {
                ok = false;
                break;
              }
            }
            if constexpr (!kHad) {
              if (u >= 1 && !issue_o(u == 1)) ok = false;
            }
          }
        }
        if (!ok) break;
        if constexpr (!kHad) ptx::umma_commit_pair(&ctl.o_full, 0x3);
        ++segs;
      }
      if (!ok) flag_error(ctl, status);
      // Every MMA issued must have retired before either CTA releases its Tensor Memory.
      ptx::umma_commit_pair(&ctl.mma_done, 0x1);
      ptx::mbar_wait(&ctl.mma_done, 0);
    } else if (lane == 0) {
      // --------------------- odd CTA: forwarder of the epilogue's arrivals -----------------
      // The odd CTA's eight epilogue warps arrive locally; once all have, one arrival at
      // cluster scope tells the even CTA's MMA issuer. Per unit: S read (s_empty; bf16 and
      // Hadamard), W written (w_full); per segment: O read (o_empty). The epilogue produces
      // them in this order, so one thread forwards them in turn.
      int64_t n_s = 0, n_w = 0, n_o = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < so.n; ++i) {
        int64_t t, seg_end;
        so.get(i, t, seg_end);
        for (int64_t tt = t; tt < seg_end; ++tt) {
          if constexpr (!kAlias) {
            if (!ptx::mbar_wait(&ctl.s_empty, par(n_s++))) { ok = false; break; }
            ptx::tc_fence_after();
            ptx::tc_fence_before();
            ptx::mbar_arrive_cluster(leader(&ctl.s_empty));
          }
          if constexpr (kPromote) {
            if (tt > t) {  // the epilogue read the previous unit's O
              if (!ptx::mbar_wait(&ctl.o_empty, par(n_o++))) { ok = false; break; }
              ptx::tc_fence_after();
              ptx::tc_fence_before();
              ptx::mbar_arrive_cluster(leader(&ctl.o_empty));
            }
          }
          if constexpr (!kHad) {
            if (!ptx::mbar_wait(&ctl.w_full, par(n_w++))) { ok = false; break; }
            ptx::tc_fence_after();
            ptx::tc_fence_before();
            ptx::mbar_arrive_cluster(leader(&ctl.w_full));
          }
        }
        if (!ok) break;
        if constexpr (!kHad) {
          if (!ptx::mbar_wait(&ctl.o_empty, par(n_o++))) { ok = false; break; }
          ptx::tc_fence_after();
          ptx::tc_fence_before();
          ptx::mbar_arrive_cluster(leader(&ctl.o_empty));
        }
      }
      if (!ok) flag_error(ctl, status);
    }
  } else {
    // --------------------------------- epilogue ------------------------------------------
    // Warp w reads TMEM lane quarter (w % 4) (this CTA's rows 32q .. 32q+31) and column half
    // h = (w - 2) / 4 of each S tile.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int rloc = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int64_t s_uses = 0, w_uses = 0, segs = 0;
    bool ok = true;
    const uint64_t k2 = ptx::pack2(kappa, kappa);
    for (int64_t i = 0; ok && i < so.n; ++i) {
      int64_t t, seg_end;
      so.get(i, t, seg_end);
      const int64_t vr = t / NT;
      const int64_t rp = vr % pair_tiles;
      const int64_t row = rp * 2 * kBM + rank * kBM + rloc;
      const float rb = row < n_rows ? rowBias[row] : neg_inf();
      const uint64_t rb2 = ptx::pack2(rb, rb);
      float sumw = 0.0f, had = 0.0f;
      float oacc[kPromote ? kKV / 2 : 1];
#pragma unroll
      for (int c = 0; c < (kPromote ? kKV / 2 : 1); ++c) oacc[c] = 0.0f;
      // Split tf32: add this warp's half row of the unit's O (32 columns) into registers.
      auto promote_o = [&]() {
        if constexpr (kPromote) {
          float o[32];
          ptx::tmem_ld_x32_sync(tmem + lane_base + kTmemO + h * (kKV / 2), o);
#pragma unroll
          for (int c = 0; c < 32; ++c) oacc[c] += o[c];
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&ctl.o_empty);
        }
      };
      // Column biases: 512 B per warp and unit, one 128-byte line per lane 0..3, fetched into
      // L1 one unit ahead (the first unit of a segment while its S MMA runs).
      if (lane < 4) ptx::prefetch_l1(colBias + (t - vr * NT) * kSBN + h * 128 + lane * 32);
      for (int64_t tt = t; tt < seg_end; ++tt) {
        const int64_t jt = tt - vr * NT;
        const float4* cb = reinterpret_cast<const float4*>(colBias + jt * kSBN + h * 128);
        if (tt + 1 < seg_end && lane < 4)
          ptx::prefetch_l1(colBias + (jt + 1) * kSBN + h * 128 + lane * 32);
        if (!ptx::mbar_wait(&ctl.s_full, par(s_uses))) { ok = false; break; }
        ++s_uses;
        ptx::tc_fence_after();
        // S(u) was issued after the previous unit's W V completed: its O can be read now.
        if (tt > t) promote_o();
        const uint32_t s_addr = tmem + lane_base + (uint32_t)h * 128u;
        uint64_t sw2 = 0ull, hd2 = 0ull;
        if constexpr (!kAlias) {
          // bf16 / Hadamard: the 128-column half row in two 64-column loads, both taken
          // before any arithmetic so that S is released (and the next unit's S MMA can
          // start) as early as possible; bf16 writes each half's 64 weights (32 bf16 pairs)
          // to tensor memory as soon as they are formed.
          float va[64], vb[64];
          ptx::tmem_ld_x64_sync(s_addr, va);
          ptx::tmem_ld_x64_sync(s_addr + 64, vb);
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&ctl.s_empty);
          if constexpr (!kHad) {
            // W row rloc, K = 128h .. 128h + 127: 64 columns of bf16 pairs at TMEM column
            // 256 + 64h, once the previous unit's W V has read W.
            if (!ptx::mbar_wait(&ctl.w_empty, par(w_uses) ^ 1u)) { ok = false; break; }
            ptx::tc_fence_after();
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float (&v)[64] = half ? vb : va;
            uint32_t wp[kHad ? 1 : 32];
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
              const float4 b4 = __ldg(cb + 16 * half + j / 4);
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
            if constexpr (!kHad)
              ptx::tmem_st_x32_sync(tmem + lane_base + kTmemW + (uint32_t)h * 64u + 32u * half, wp);
          }
          if constexpr (!kHad) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ctl.w_full);
            ++w_uses;
          }
        } else {
          // tf32 / split: in two 64-column halves, W_hi = tf32(w) written over S (and
          // W_lo = bf16(w - W_hi) beside it). The previous unit's W V has completed: its
          // commit precedes this unit's s_full.
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float v[64];
            ptx::tmem_ld_x64_sync(s_addr + 64 * half, v);
            uint32_t lo[(kSplitW || kWide) ? 32 : 1];
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
              const float4 b4 = __ldg(cb + 16 * half + j / 4);
              const uint64_t e01 = ptx::add2(ptx::fma2(k2, ptx::pack2(v[j + 0], v[j + 1]),
                                                       ptx::pack2(b4.x, b4.y)), rb2);
              const uint64_t e23 = ptx::add2(ptx::fma2(k2, ptx::pack2(v[j + 2], v[j + 3]),
                                                       ptx::pack2(b4.z, b4.w)), rb2);
              float x0, x1, x2, x3;
              ptx::unpack2(e01, x0, x1);
              ptx::unpack2(e23, x2, x3);
              const float w0 = ex2(x0), w1 = ex2(x1), w2 = ex2(x2), w3 = ex2(x3);
              sw2 = ptx::add2(sw2, ptx::add2(ptx::pack2(w0, w1), ptx::pack2(w2, w3)));
              if constexpr (kWide) {
                __nv_bfloat162 p01 = __floats2bfloat162_rn(w0, w1);
                __nv_bfloat162 p23 = __floats2bfloat162_rn(w2, w3);
                lo[j / 2] = *reinterpret_cast<uint32_t*>(&p01);
                lo[j / 2 + 1] = *reinterpret_cast<uint32_t*>(&p23);
                continue;
              }
              const uint32_t h0 = tf32_rna(w0), h1 = tf32_rna(w1), h2 = tf32_rna(w2),
                             h3 = tf32_rna(w3);
              if constexpr (kSplitW) {
                __nv_bfloat162 l01 = __floats2bfloat162_rn(w0 - __uint_as_float(h0),
                                                           w1 - __uint_as_float(h1));
                __nv_bfloat162 l23 = __floats2bfloat162_rn(w2 - __uint_as_float(h2),
                                                           w3 - __uint_as_float(h3));
                lo[j / 2] = *reinterpret_cast<uint32_t*>(&l01);
                lo[j / 2 + 1] = *reinterpret_cast<uint32_t*>(&l23);
              }
              v[j + 0] = __uint_as_float(h0);
              v[j + 1] = __uint_as_float(h1);
              v[j + 2] = __uint_as_float(h2);
              v[j + 3] = __uint_as_float(h3);
            }
            if constexpr (kWide) {
              // bf16 pairs of this half's 64 weights over the first half's (already read)
              // S columns: pair-columns 128h + 32 half .. + 31
              ptx::tmem_st_x32_sync(s_addr + 32 * half, lo);
              continue;
            }
            ptx::tmem_st_x64_sync(s_addr + 64 * half, *reinterpret_cast<uint32_t(*)[64]>(v));
            if constexpr (kSplitW)
              ptx::tmem_st_x32_sync(tmem + lane_base + kTmemWL + (uint32_t)h * 64u + 32u * half,
                                    lo);
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&ctl.w_full);
          ++w_uses;
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
      }
      if (!ok) break;
      const int64_t slot = so.slot(t, vr, T);
      const int64_t prow = vr * 2 * kBM + rank * kBM + rloc;  // row of the partial buffers
      if constexpr (!kHad) {
        if (!ptx::mbar_wait(&ctl.o_full, par(segs))) { ok = false; break; }
        ptx::tc_fence_after();
        float* dst = pO + ((size_t)slot * ldp + (size_t)prow) * kKV + h * (kKV / 2);
        if constexpr (kPromote) {
          promote_o();  // the segment's last unit
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) =
                make_float4(oacc[e], oacc[e + 1], oacc[e + 2], oacc[e + 3]);
        } else {
#pragma unroll 1
          for (int c = 0; c < kKV / 64; ++c) {
            float o[32];
            ptx::tmem_ld_x32_sync(tmem + lane_base + kTmemO + h * (kKV / 2) + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + c * 32 + e) =
                  make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&ctl.o_empty);
        }
      }
      pW[((size_t)(2 * slot + h)) * ldp + (size_t)prow] = make_float2(sumw, had);
      ++segs;
    }
    if (!ok) flag_error(ctl, status);
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();  // neither CTA leaves while the pair's MMAs or copies may touch it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Adds the partial slots of one (group, pair tile) in a fixed order and finishes the output:
// apply: out = O; gradient: out = 2 a (x - O / sum w); Hadamard: out = sum w S.
template <int kMode>
__global__ void wsum_pair_reduce_kernel(const float* __restrict__ pO, const float2* __restrict__ pW,
                                        int64_t ldp, int kKV, int64_t pair_tiles, int64_t NT,
                                        int64_t T, int64_t G, int64_t run_len, int64_t n_rows,
                                        const float* __restrict__ rowW, const float* __restrict__ X,
                                        int64_t d, int64_t k, float* __restrict__ out,
                                        int64_t ldo) {
  const int64_t per_row = (kMode == kWsumHadamard) ? 1 : kKV;
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (idx >= ldp * per_row) return;
  const int64_t prow = idx / per_row;
  const int64_t o = idx - prow * per_row;
  const int64_t vr = prow / (2 * kBM);
  const int64_t grp = vr / pair_tiles;
  const int64_t row = (vr - grp * pair_tiles) * 2 * kBM + (prow - vr * 2 * kBM);
  if (row >= n_rows) return;
  const int slots = run_len > 0 ? (int)((NT + run_len - 1) / run_len)
                                : (int)(sk_owner((vr + 1) * NT - 1, T, G) - sk_owner(vr * NT, T, G) + 1);
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

// V^T planes for the split second contraction: hi = tf32(v), lo = tf32(v - hi), and bf16(v),
// each rows_pad x cols_pad (row c holds column c of V, zero padded).
__global__ void pack_transpose_split_kernel(const float* __restrict__ src, uint32_t* __restrict__ hi,
                                            uint32_t* __restrict__ lo,
                                            __nv_bfloat16* __restrict__ bf, int64_t rows,
                                            int64_t cols, int64_t rows_pad, int64_t cols_pad) {
  __shared__ float tile[32][33];
  const int64_t r0 = (int64_t)blockIdx.x * 32, c0 = (int64_t)blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < rows && c < cols) ? src[r * cols + c] : 0.0f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;  // dst row c, dst column r
    if (c >= cols_pad || r >= rows_pad) continue;
    const float v = tile[threadIdx.x][i];
    const int64_t e = c * rows_pad + r;
    const uint32_t h = tf32_rna(v);
    hi[e] = h;
    lo[e] = tf32_rna(v - __uint_as_float(h));
    bf[e] = __float2bfloat16_rn(v);
  }
}

// Stage plan: two K-chunks per stage when the chunk count is even and at least three such
// stages fit beside the V tile; else one chunk per stage and at least three stages.
static bool stage_plan(int kc, uint32_t v_bytes, int* n_st, int* kps) {
  const int room = kSmemLimit - (int)sizeof(PCtrl) - 1024 - (int)v_bytes;
  const int chunk = 2 * kChunk;
  if (kc % 2 == 0 && room / (2 * chunk) >= 3) {
    *kps = 2;
    *n_st = std::min(kMaxStages, room / (2 * chunk));
    return true;
  }
  *kps = 1;
  *n_st = std::min(kMaxStages, room / chunk);
  return *n_st >= 3;
}

template <int kPrec, int kKV>
static int launch(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mV,
                  const CUtensorMap& mVlo, const CUtensorMap& mVb, const float* colBias,
                  const float* rowBias, int64_t n_rows, int64_t pair_tiles, int64_t NT, int64_t T,
                  int64_t run_len, int64_t pairs, int kc, float kappa, float* pO, float2* pW,
                  int64_t ldp, unsigned* status, cudaStream_t st) {
  int n_st = 0, kps = 1;
  if (!stage_plan(kc, VShape<kPrec, kKV>::bytes, &n_st, &kps)) return FLASHOT_ERR_INVALID_ARG;
  const int dyn = n_st * kps * 2 * kChunk + (int)VShape<kPrec, kKV>::bytes + 1024;
  auto kern = wsum_pair_kernel<kPrec, kKV>;
  int rc = tc::set_smem(kern, dyn);
  if (rc != FLASHOT_OK) return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_WSUM, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mA, mB, mV, mVlo, mVb, colBias, rowBias, n_rows,
                           pair_tiles, NT, T, run_len, kc, kps, n_st, kappa, pO, pW, ldp,
                           status) != cudaSuccess)
      return FLASHOT_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

// Resident 2-CTA clusters of the widest variant (the grid is sized by it for all).
static int max_clusters() {
  static int cached = -1;
  if (cached >= 0) return cached;
  int n = 0;
  int n_st = 0, kps = 1;
  stage_plan(16, VShape<kPrecTF32, 128>::bytes, &n_st, &kps);
  const int dyn = n_st * kps * 2 * kChunk + (int)VShape<kPrecTF32, 128>::bytes + 1024;
  auto kern = wsum_pair_kernel<kPrecTF32, 128>;
  if (tc::set_smem(kern, dyn) == FLASHOT_OK) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)dyn;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cached = n;
  return n;
}

}  // namespace tcp

size_t tc_wsum_pair_scratch_bytes(int64_t rows_pad, int64_t k_or_d) {
  // pO: kMaxOwners slots x rows_pad x (groups x kKV) floats, groups x kKV <= round_up(k, 128)
  // (or 64); pW: 2 kMaxOwners slots x groups x rows_pad float2, groups <= kk / 64.
  const int64_t kk = k_or_d <= 64 ? 64 : (k_or_d <= 128 ? 128 : (k_or_d + 255) / 256 * 256);
  return (size_t)tcp::kMaxOwners * rows_pad * kk * sizeof(float) +
         (size_t)2 * tcp::kMaxOwners * (kk / 64) * rows_pad * sizeof(float2) + 1024;
}

size_t tc_wsum_pair_vt_bytes(int prec, int64_t rows_pad, int64_t k_or_d) {
  // V^T planes: out_rows_pad (whole 64- or 128-column groups) x cols_pad elements each.
  const int64_t kk = k_or_d <= 64 ? 64 : (k_or_d <= 128 ? 128 : (k_or_d + 255) / 256 * 256);
  const int64_t e = kk * rows_pad;
  return (size_t)e * (prec == FLASHOT_PREC_BF16 ? 2 : (prec == FLASHOT_PREC_TF32 ? 4 : 10)) + 1024;
}

bool tc_wsum_pair_available(int sms) { return tcp::max_clusters() >= std::max(1, sms / 4); }

int tc_wsum_pair_pass(int prec, int mode, const void* rowQ, const void* colQ,
                      const float* colBias, const float* rowBias, int64_t n_rows, int64_t n_cols,
                      int64_t rows_pad, int64_t cols_pad, int64_t d, int64_t dpt, float kappa,
                      const float* V, int64_t ldv, int64_t k, void* vtq, void* scratch,
                      const float* rowW, const float* X, float* out, int64_t ldo, int sms,
                      unsigned* status, cudaStream_t st) {
  using namespace tcp;
  const bool bf = (prec == FLASHOT_PREC_BF16);
  const bool split = (prec == FLASHOT_PREC_TF32X3);
  const int es = bf ? 2 : 4;
  const int kc = (int)(dpt * es / 128);
  if (rows_pad % (2 * kBM) != 0 || cols_pad % kSBN != 0) return FLASHOT_ERR_INVALID_ARG;
  const int64_t pair_tiles = rows_pad / (2 * kBM), NT = cols_pad / kSBN;
  const bool had = (mode == kWsumHadamard);
  if (!had && ldv != k) return FLASHOT_ERR_INVALID_ARG;
  // Output columns per group: 128 (64 for split tf32, whose V planes need the room; 64 when
  // k <= 64).
  // bf16 outputs wider than 128 columns (the gradient at d = 512) take 256-column groups, so
  // S is formed half as often.
  const int kv = had ? 0 : ((k <= 64 || split) ? 64 : ((bf && k > 128) ? 256 : 128));
  const int64_t groups = had ? 1 : (k + kv - 1) / kv;
  const int64_t vrows = groups * pair_tiles;
  const int64_t T = vrows * NT;
  // Split tf32 rows are three tf32 segments long: when the pairs' row tiles alone would fill
  // most of L2 (d = 512 and up), the pairs take round-robin runs of a quarter of a row
  // group's column tiles instead of stream-K ranges. FLASHOT_WSUM_RUNS=0 in the environment
  // keeps stream-K (for comparisons; read once per process).
  static const bool runs_enabled = [] {
    const char* e = std::getenv("FLASHOT_WSUM_RUNS");
    return !(e && e[0] == '0');
  }();
  const int64_t max_pairs = std::min(max_clusters(), sms / 2);
  const bool runs = runs_enabled && split && NT >= 2 &&
                    max_pairs * 2 * kBM * dpt * (int64_t)sizeof(float) > (96ll << 20);
  const int64_t run_len = runs ? (NT + kMaxOwners - 1) / kMaxOwners : 0;
  const int64_t G = runs ? max_pairs : tc::choose_grid(vrows, NT, max_pairs, kMaxOwners);
  const int64_t ldp = vrows * 2 * kBM;
  float* pO = static_cast<float*>(scratch);
  const size_t po_bytes = (size_t)kMaxOwners * ldp * (had ? 0 : kv) * sizeof(float);
  float2* pW = reinterpret_cast<float2*>(static_cast<char*>(scratch) + (po_bytes + 255) / 256 * 256);
  CUtensorMap mA, mB, mV, mVlo, mVb;
  int rc = tc::make_map(&mA, rowQ, rows_pad, dpt, bf);
  if (rc == FLASHOT_OK) rc = tc::make_map(&mB, colQ, cols_pad, dpt, bf);
  if (rc != FLASHOT_OK) return rc;
  mV = mVlo = mVb = mB;  // unused unless set below
  if (!had) {
    const int64_t out_rows_pad = groups * kv;
    dim3 blk(32, 8), grd((unsigned)(cols_pad / 32), (unsigned)(out_rows_pad / 32));
    const int64_t plane = out_rows_pad * cols_pad;
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
      if (bf)
        pack_transpose_kernel<PackKind::BF16><<<grd, blk, 0, st>>>(V, vtq, n_cols, k, cols_pad,
                                                                   out_rows_pad);
      else if (!split)
        pack_transpose_kernel<PackKind::TF32><<<grd, blk, 0, st>>>(V, vtq, n_cols, k, cols_pad,
                                                                   out_rows_pad);
      else
        pack_transpose_split_kernel<<<grd, blk, 0, st>>>(
            V, static_cast<uint32_t*>(vtq), static_cast<uint32_t*>(vtq) + plane,
            reinterpret_cast<__nv_bfloat16*>(static_cast<uint32_t*>(vtq) + 2 * plane), n_cols,
            k, cols_pad, out_rows_pad);
    }
    if (cudaGetLastError() != cudaSuccess) return FLASHOT_ERR_CUDA;
    rc = tc::make_map_rows(&mV, vtq, out_rows_pad, cols_pad, bf, kv / 2);
    if (rc == FLASHOT_OK && split) {
      rc = tc::make_map_rows(&mVlo, static_cast<uint32_t*>(vtq) + plane, out_rows_pad, cols_pad,
                             false, kv / 2);
      if (rc == FLASHOT_OK)
        rc = tc::make_map_rows(&mVb, static_cast<uint32_t*>(vtq) + 2 * plane, out_rows_pad,
                               cols_pad, true, kv / 2);
    }
    if (rc != FLASHOT_OK) return rc;
  }
#define FLASHOT_PAIR_WSUM(P, KV)                                                            \
  launch<P, KV>(mA, mB, mV, mVlo, mVb, colBias, rowBias, n_rows, pair_tiles, NT, T, run_len, G, \
                kc, kappa, pO, pW, ldp, status, st)
  if (had)
    rc = bf ? FLASHOT_PAIR_WSUM(kPrecBF16, 0) : FLASHOT_PAIR_WSUM(kPrecTF32, 0);
  else if (bf)
    rc = kv == 64 ? FLASHOT_PAIR_WSUM(kPrecBF16, 64)
                  : (kv == 128 ? FLASHOT_PAIR_WSUM(kPrecBF16, 128) : FLASHOT_PAIR_WSUM(kPrecBF16, 256));
  else if (!split)
    rc = kv == 64 ? FLASHOT_PAIR_WSUM(kPrecTF32, 64) : FLASHOT_PAIR_WSUM(kPrecTF32, 128);
  else
    rc = FLASHOT_PAIR_WSUM(kPrecSplit, 64);
#undef FLASHOT_PAIR_WSUM
  if (rc != FLASHOT_OK) return rc;
  const int64_t total = ldp * (had ? 1 : kv);
  const unsigned blocks = (unsigned)((total + 255) / 256);
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, st);
    if (mode == kWsumGrad)
      wsum_pair_reduce_kernel<kWsumGrad><<<blocks, 256, 0, st>>>(
          pO, pW, ldp, kv, pair_tiles, NT, T, G, run_len, n_rows, rowW, X, d, k, out, ldo);
    else if (mode == kWsumApply)
      wsum_pair_reduce_kernel<kWsumApply><<<blocks, 256, 0, st>>>(
          pO, pW, ldp, kv, pair_tiles, NT, T, G, run_len, n_rows, rowW, X, d, k, out, ldo);
    else
      wsum_pair_reduce_kernel<kWsumHadamard><<<blocks, 256, 0, st>>>(
          pO, pW, ldp, 1, pair_tiles, NT, T, G, run_len, n_rows, rowW, X, d, k, out, ldo);
  }
  return cudaGetLastError() == cudaSuccess ? FLASHOT_OK : FLASHOT_ERR_CUDA;
}

}  // namespace flashot
