// trace.h -- launch accounting for diagnostics: a process-wide launch counter and an
// optional per-launch CUDA-event timer (see flashot_launch_count / flashot_timer_* in
// include/flashot.h). A TraceScope brackets exactly one kernel launch.
#pragma once

#include <cuda_runtime.h>

namespace flashot {

void trace_before(int kernel_class, cudaStream_t st);
void trace_after(int kernel_class, cudaStream_t st);

struct TraceScope {
  int cls;
  cudaStream_t st;
  TraceScope(int c, cudaStream_t s) : cls(c), st(s) { trace_before(c, s); }
  ~TraceScope() { trace_after(cls, st); }
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;
};

}  // namespace flashot
