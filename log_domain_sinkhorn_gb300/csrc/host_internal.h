// host_internal.h -- host helpers of flashot.cu that other translation units of the
// library use. Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

namespace flashot {

// FLASHOT_OK if the current device is an sm_103 GPU, else FLASHOT_ERR_UNSUPPORTED_DEVICE
// (or FLASHOT_ERR_CUDA when the runtime cannot say, with the error recorded).
int checked_current_device();

// Records e for flashot_last_cuda_error() and returns FLASHOT_ERR_CUDA.
int record_cuda_error(cudaError_t e);

}  // namespace flashot
