// noalloc.cu -- an f-update for callers that must not allocate device memory.
//
// Some programs that embed this library cannot hand it a workspace from cudaMalloc: a
// host framework that owns every device byte through its own fixed arena and does not let
// plugins allocate, or a latency-critical loop where a cudaMalloc / cudaFree (which can
// synchronise the device) is not acceptable. flashot_sinkhorn_step_f_noalloc serves them:
// it runs the same f-update as flashot_sinkhorn_step_f, with its scratch taken from a
// fixed array compiled into the library instead of from the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "flashot.h"

namespace {

// The scratch: FLASHOT_NOALLOC_SCRATCH_BYTES of device memory, reserved on every GPU that
// loads this library for as long as the process lives. In host code `g_noalloc_scratch`
// only names a host-side shadow of the symbol; its device address comes from
// cudaGetSymbolAddress (see scratch_for_current_device).
constexpr size_t kScratchBytes = FLASHOT_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
  bool ready = false;
  void* ptr = nullptr;
};
DeviceScratch g_scratch[64];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device, looked up once per device
// (the first call on a device does this set-up, with that device current).
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return FLASHOT_ERR_CUDA;
  if (dev < 0 || dev >= 64) return FLASHOT_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  DeviceScratch& s = g_scratch[dev];
  if (!s.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FLASHOT_ERR_CUDA;
    }
    s.ptr = p;
    s.ready = true;
  }
  *out = s.ptr;
  return FLASHOT_OK;
}

}  // namespace

extern "C" int flashot_sinkhorn_step_f_noalloc(const float* X, const float* Y, const float* b,
                                               const float* g, int64_t n, int64_t m, int64_t d,
                                               float eps, int flags, float* f,
                                               flashot_stream_t stream) {
  // Only the precision bits are honoured: the shared array may hold another call's data,
  // so the inputs are always packed afresh.
  const int prec = flags & FLASHOT_PREC_MASK;
  const size_t need = flashot_workspace_bytes(n, m, d, 0, prec);
  if (need == 0) return FLASHOT_ERR_INVALID_ARG;
  if (need > kScratchBytes) return FLASHOT_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != FLASHOT_OK) return rc;
  return flashot_sinkhorn_step_f(X, Y, b, g, n, m, d, eps, prec, f, scratch, kScratchBytes,
                                 stream);
}
