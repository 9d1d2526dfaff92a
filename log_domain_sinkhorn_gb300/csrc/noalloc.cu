// noalloc.cu -- an f-update for callers that must not allocate device memory.
//
// Some programs that embed this library cannot hand it a workspace from cudaMalloc: a
// host framework that owns every device byte through its own fixed arena and does not let
// plugins allocate, or a latency-critical loop where a cudaMalloc / cudaFree (which can
// synchronise the device) is not acceptable. flashot_sinkhorn_step_f_noalloc serves them:
// it runs the same f-update as flashot_sinkhorn_step_f, with its scratch taken from a
// fixed array compiled into the library instead of from the caller.
#include <cuda_runtime.h>

#include "flashot.h"
#include "host_internal.h"

namespace {

// The scratch: FLASHOT_NOALLOC_SCRATCH_BYTES of device memory in every context that loads
// this file's module, held until the context goes away. Its first 4 bytes are the status
// word of the workspace layout (sticky bounded-wait timeouts); static storage starts it at
// zero. In host code `g_noalloc_scratch` only names a host-side shadow of the symbol; the
// device address comes from cudaGetSymbolAddress (scratch_in_current_context).
constexpr size_t kScratchBytes = FLASHOT_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array in the current context. The device check comes
// first: on a GPU other than sm_103 the module has no image to resolve the symbol in.
// The address is looked up on every call rather than cached, because it belongs to a
// context, not to a device ordinal: after cudaDeviceReset, or with another context
// current on the same device, a cached address would point into memory this context does
// not own. Once the module is loaded the lookup allocates nothing; the first lookup in a
// context is what loads it (under CUDA's default lazy module loading).
int scratch_in_current_context(void** out) {
  const int rc = flashot::checked_current_device();
  if (rc != FLASHOT_OK) return rc;
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return flashot::record_cuda_error(e);
  if (p == nullptr) return FLASHOT_ERR_CUDA;
  *out = p;
  return FLASHOT_OK;
}

}  // namespace

extern "C" int flashot_sinkhorn_step_f_noalloc(const float* X, const float* Y, const float* b,
                                               const float* g, int64_t n, int64_t m, int64_t d,
                                               float eps, int flags, float* f,
                                               flashot_stream_t stream) {
  // FLASHOT_REUSE_PACK is dropped: the shared array may hold another call's packed
  // inputs, so they are always packed afresh. Every other flag means what it means for
  // flashot_sinkhorn_step_f (precision bits, FLASHOT_VALIDATE).
  const int fl = flags & ~FLASHOT_REUSE_PACK;
  const size_t need = flashot_workspace_bytes(n, m, d, 0, fl);
  if (need == 0) return FLASHOT_ERR_INVALID_ARG;
  if (need > kScratchBytes) return FLASHOT_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = scratch_in_current_context(&scratch);
  if (rc != FLASHOT_OK) return rc;
  return flashot_sinkhorn_step_f(X, Y, b, g, n, m, d, eps, fl, f, scratch, kScratchBytes,
                                 stream);
}

extern "C" int flashot_noalloc_status(flashot_stream_t stream) {
  void* scratch = nullptr;
  const int rc = scratch_in_current_context(&scratch);
  if (rc != FLASHOT_OK) return rc;
  return flashot_workspace_status(scratch, stream);
}
