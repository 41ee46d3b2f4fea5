// idx_copy_async: a byte copy run by the GPU's SMs, for the few hundred KB a
// decode step moves between page-locked host memory and the device (its
// inputs in, its indices out).  On GB300 the SMs reach page-locked host memory
// over NVLink-C2C with ordinary loads and stores, so a transfer this small
// costs about a kernel launch and one memory round trip, where a copy-engine
// transfer (cudaMemcpyAsync) costs several microseconds of setup of its own.
// The pages have no counterpart for this entry; it only serves the step's
// host<->device traffic.
//
// Each pointer is resolved with cudaPointerGetAttributes: device memory of the
// current device, managed memory, or page-locked host memory mapped into the
// device's address space (its device pointer); anything else is refused before
// a launch, so the kernel only ever touches addresses the device can reach.
#include <cuda_runtime.h>

#include "common.cuh"
#include "idx.h"
#include "launch.h"

namespace {

constexpr int kCopyBlock = 256;

// 16-byte moves when both ends and the size allow it, else bytes; every
// thread's loads are issued before its stores.
__global__ void __launch_bounds__(kCopyBlock) copy_kernel(uint8_t* __restrict__ dst,
                                                          const uint8_t* __restrict__ src,
                                                          size_t n, int vec) {
  idx::pdl_launch_dependents();
  idx::pdl_wait();  // the source may come from the previous kernel
  const size_t tid = (size_t)blockIdx.x * kCopyBlock + threadIdx.x;
  const size_t nt = (size_t)gridDim.x * kCopyBlock;
  size_t done = 0;
  if (vec) {
    const size_t n16 = n / 16;
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    constexpr int kU = 4;
    size_t i = tid;
    for (; i + (kU - 1) * nt < n16; i += kU * nt) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) v[u] = s[i + u * nt];
#pragma unroll
      for (int u = 0; u < kU; ++u) d[i + u * nt] = v[u];
    }
    for (; i < n16; i += nt) d[i] = s[i];
    done = n16 * 16;
  }
  for (size_t i = done + tid; i < n; i += nt) dst[i] = src[i];
}

// The device's view of p (nullptr if the device cannot reach it).
void* device_view(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
      return a.device == dev ? a.devicePointer : nullptr;
    case cudaMemoryTypeManaged:
    case cudaMemoryTypeHost:
      return a.devicePointer;
    default:
      return nullptr;
  }
}

}  // namespace

extern "C" IDX_API idx_status idx_copy_async(void* dst, const void* src, size_t bytes,
                                             idx_stream_t stream) {
  if (bytes == 0) return idx::ok();
  if (dst == nullptr || src == nullptr) return idx::fail(IDX_ERR_INVALID_ARG, "null pointer");
  int sms = 0;
  idx_status s = idx::current_device_ok(&sms);
  if (s != IDX_OK) return s;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return idx::fail(IDX_ERR_CUDA, "cudaGetDevice failed");
  }
  // both whole ranges must lie in one allocation the device can reach: the
  // attributes of their first and last bytes must give matching views
  uint8_t* d0 = static_cast<uint8_t*>(device_view(dst, dev));
  const uint8_t* s0 = static_cast<const uint8_t*>(device_view(src, dev));
  uint8_t* d1 = static_cast<uint8_t*>(device_view(static_cast<uint8_t*>(dst) + bytes - 1, dev));
  const uint8_t* s1 =
      static_cast<const uint8_t*>(device_view(static_cast<const uint8_t*>(src) + bytes - 1, dev));
  if (d0 == nullptr || s0 == nullptr || d1 != d0 + (bytes - 1) || s1 != s0 + (bytes - 1))
    return idx::fail(IDX_ERR_INVALID_ARG,
                     "dst and src must be device memory of the current device, managed memory, "
                     "or page-locked host memory mapped for the device");
  const int vec = ((reinterpret_cast<uintptr_t>(d0) | reinterpret_cast<uintptr_t>(s0)) & 15u) == 0;
  const size_t units = vec ? bytes / 16 : bytes;
  size_t blocks = (units + kCopyBlock - 1) / kCopyBlock;
  const size_t cap = (size_t)(sms > 0 ? sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  const cudaError_t e = idx::launch_dependent(copy_kernel, dim3((unsigned)blocks), dim3(kCopyBlock), 0,
                                              (cudaStream_t)stream, d0, s0, bytes, vec);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return idx::fail(IDX_ERR_CUDA, "copy launch: %s", cudaGetErrorString(e));
  }
  return idx::ok();
}
