// tc_solve_short.h -- the persistent solve of short tensor-core contractions
// (tc_solve_short.cu), used by flashot.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace flashot {

// Self-test of the grid barrier's bounded wait: zeroes *word, then one thread waits for it to
// reach 1 (nothing writes it), gives up after limit_ns and sets bits 1 and 2 of *status.
int tc_selftest_grid_wait(unsigned* status, unsigned* word, int64_t limit_ns, cudaStream_t st);

// Bytes of device memory the persistent solve needs for its arrival counters and grid
// barrier word (zeroed by tc_short_solve itself on `st`).
size_t tc_short_solve_sync_bytes(int64_t n_pad, int64_t m_pad);

// Every half-step of a solve (n_stages x iters_per_stage iterations) in one cooperative
// launch, for contractions of at most six 128-byte K-chunks. schedule: 0 alternating (f =
// F(g), then g = G(f)); 1 symmetric (f and g both averaged with the update from the previous
// iterate); 2 symmetric for a self-transport problem (X = Y, a = b, started from f = g: one
// pass per iteration, g left to the caller as a copy of f). With err_rows != NULL and
// err_iter >= 0 (alternating only) the f-update of iteration err_iter (counted from 0 in
// this launch) also writes each row's share of the L1 row-marginal error of the iterate
// before it, w_i |expm1((f_old - f_new) / eps)| with w = err_w (0 on padding rows), as
// the per-pass combine does. Inputs and outputs are those of
// the per-pass path: xq / yq the packed clouds (n_pad / m_pad rows of dpt elements), alpha /
// beta the squared norms, la2 / lb2 the log2 weights, biasF (and for the symmetric schedule
// biasG) the first pass's column biases on entry, f and g the potentials (read too by the
// symmetric schedule) and written. partial holds partial_bytes of scratch for the stream-K
// partials (max_splits x max(n_pad, m_pad) float2 serve every schedule but a symmetric one
// with many owners per row tile). Returns FLASHOT_ERR_NOT_IMPLEMENTED, having enqueued
// nothing the per-pass path reads (at most the zeroing of sync_words), when the solve does
// not qualify: a longer contraction, more than 32 eps stages, a grid that cannot be
// co-resident (or a cooperative launch refused for that), fewer than 1.5 tiles per CTA and
// pass on either side, partials that do not fit, or FLASHOT_SHORT_SOLVE=0 in the
// environment (FLASHOT_SHORT_SOLVE=1 drops the tile-count condition). The caller then runs
// the per-pass path.
int tc_short_solve(bool bf16, const void* xq, const void* yq, int64_t n, int64_t m,
                   int64_t n_pad, int64_t m_pad, int64_t dpt, const float* alpha,
                   const float* beta, const float* la2, const float* lb2, float* biasF,
                   float* biasG, float* f, float* g, const float* eps_sched, int n_stages,
                   int iters_per_stage, int schedule, float* err_rows, const float* err_w,
                   int err_iter, float2* partial, size_t partial_bytes, int max_splits,
                   void* sync_words, size_t sync_bytes, int sms, unsigned* status,
                   cudaStream_t st);

}  // namespace flashot
