// Library-wide entry points: status strings, version, the device error word.
#include "common.cuh"
#include "host_utils.h"

namespace bsf {

__device__ int g_device_error = 0;

int* device_error_ptr() {
  static std::atomic<int*> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int* ptr = cached[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptr = static_cast<int*>(p);
    cached[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
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

// ---------------------------------------------------------------------------
// Streaming read of a buffer: XOR of all 64-bit words.  Used to measure the
// bandwidth at which the SMs read a memory (HBM, or pinned host memory over the
// host link through its device-mapped address) and to checksum buffers.
namespace bsf {
namespace {
__global__ void __launch_bounds__(256) checksum_kernel(const uint4* __restrict__ p, int64_t n16,
                                                        unsigned long long* out) {
  uint64_t acc = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {   // four independent 16-byte loads in flight per thread
    const uint4 v0 = __ldcs(p + i), v1 = __ldcs(p + i + stride), v2 = __ldcs(p + i + 2 * stride),
                v3 = __ldcs(p + i + 3 * stride);
    acc ^= (static_cast<uint64_t>(v0.y) << 32 | v0.x) ^ (static_cast<uint64_t>(v0.w) << 32 | v0.z);
    acc ^= (static_cast<uint64_t>(v1.y) << 32 | v1.x) ^ (static_cast<uint64_t>(v1.w) << 32 | v1.z);
    acc ^= (static_cast<uint64_t>(v2.y) << 32 | v2.x) ^ (static_cast<uint64_t>(v2.w) << 32 | v2.z);
    acc ^= (static_cast<uint64_t>(v3.y) << 32 | v3.x) ^ (static_cast<uint64_t>(v3.w) << 32 | v3.z);
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(p + i);
    acc ^= (static_cast<uint64_t>(v.y) << 32 | v.x) ^ (static_cast<uint64_t>(v.w) << 32 | v.z);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) atomicXor(out, static_cast<unsigned long long>(acc));
}
}  // namespace
}  // namespace bsf

extern "C" bsf_status bsf_checksum_u64(const void* p, size_t bytes, int flags, unsigned long long* out,
                                       bsf_stream_t stream) {
  if (!p || !out || bytes % 16 || (flags & ~BSF_B_HOST_MAPPED)) return BSF_ERR_INVALID_ARGUMENT;
  if (!bsf::aligned16(p)) return BSF_ERR_MISALIGNED;
  const void* src = p;
  if (flags & BSF_B_HOST_MAPPED) {
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, const_cast<void*>(p), 0) != cudaSuccess) {
      cudaGetLastError();
      return BSF_ERR_INVALID_ARGUMENT;
    }
    src = dp;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(out, 0, sizeof(unsigned long long), s) != cudaSuccess) return BSF_ERR_CUDA;
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  if (n16 == 0) return BSF_OK;
  int64_t blocks = static_cast<int64_t>(bsf::sm_count()) * 8;
  const int64_t need = (n16 + 255) / 256;
  if (need < blocks) blocks = need;
  bsf::checksum_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint4*>(src), n16, out);
  return bsf::launch_status();
}
