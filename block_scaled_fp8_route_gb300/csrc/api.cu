// Library-wide entry points: status strings, version, the device error word.
#include "common.cuh"
#include "host_utils.h"

namespace bsf {

__device__ int g_device_error = 0;

int* device_error_ptr() {
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (cached[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace bsf

extern "C" const char* bsf_status_string(bsf_status status) {
  switch (status) {
    case BSF_OK: return "ok";
    case BSF_ERR_INVALID_ARGUMENT: return "invalid argument";
    case BSF_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case BSF_ERR_UNSUPPORTED: return "unsupported shape";
    case BSF_ERR_CUDA: return "CUDA error";
    case BSF_ERR_DEVICE: return "device is not sm_100-class";
  }
  return "unknown status";
}

extern "C" int bsf_version(void) { return 1; }

extern "C" bsf_status bsf_get_device_error(int32_t* code, int clear, bsf_stream_t stream) {
  if (!code) return BSF_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int value = 0;
  if (cudaMemcpyFromSymbolAsync(&value, bsf::g_device_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return BSF_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSF_ERR_CUDA;
  *code = value;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(bsf::g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return BSF_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BSF_ERR_CUDA;
  }
  return BSF_OK;
}
