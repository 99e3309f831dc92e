// Host-side helpers shared by the C-ABI entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bsfroute.h"

namespace bsf {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Status of the launch just enqueued (configuration errors only; the kernel
// itself runs asynchronously).
inline bsf_status launch_status() {
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? BSF_OK : BSF_ERR_CUDA;
}

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the library's sticky error word on the current device
// (nullptr if it cannot be resolved).
int* device_error_ptr();

}  // namespace bsf
