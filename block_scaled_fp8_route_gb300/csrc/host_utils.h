// Host-side helpers shared by the C-ABI entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bsfroute.h"

namespace bsf {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sizes beyond any real problem are refused (BSF_ERR_UNSUPPORTED) before a product of them is
// formed, so no grid or offset computation can wrap: at most 2^31 - 1 rows (tokens, or experts x
// rows) of at most 2^24 elements or bytes each.
constexpr int64_t kMaxRows = INT32_MAX;
constexpr int64_t kMaxRowWidth = int64_t(1) << 24;
inline bool fits_rows(int64_t rows, int64_t width) { return rows <= kMaxRows && width <= kMaxRowWidth; }
// E x N weight rows of width K
inline bool fits_weights(int64_t E, int64_t N, int64_t K) {
  return E <= kMaxRows && N <= kMaxRowWidth && fits_rows(E * N, K);
}

// Status of the launch just enqueued (configuration errors only; the kernel
// itself runs asynchronously).
inline bsf_status launch_status() {
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? BSF_OK : BSF_ERR_CUDA;
}

// Launch `kernel` as a programmatic dependent of the preceding kernel on `stream`
// (cudaLaunchAttributeProgrammaticStreamSerialization): its CTAs may be scheduled while
// that kernel drains, and it must call pdl_wait() before its first global memory access.
// Returns the launch's configuration status.
template <class... Params, class... Args>
inline bsf_status launch_dependent(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
#ifdef BSF_DISABLE_PDL
  cfg.numAttrs = 0;
#else
  cfg.numAttrs = 1;
#endif
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return BSF_ERR_CUDA;
  }
  return launch_status();
}

// Per-device values the library resolves on first use are cached in atomics, so
// first calls from several host threads at once are well defined (each stores
// the same value).  The caches are not invalidated: after cudaDeviceReset() the
// process must not call the library again on that device.

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the library's sticky error word on the current device
// (nullptr if it cannot be resolved).
int* device_error_ptr();

}  // namespace bsf
