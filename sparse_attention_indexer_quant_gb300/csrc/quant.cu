// MXFP4 quantisation kernels: key insert into the paged cache, and query
// quantisation (vLLM PR #48558 "[Kernel] MXFP4 indexer cache for GLM-5.2 / DSA",
// sections "Changes" and "Notes").
//
// Sixteen threads own one 128-element vector: each loads 8 bf16 values (16 B),
// four threads make one 32-element block, whose max |x| is reduced with two
// butterfly shuffles on the integer bit patterns (for non-negative floats the
// bit order is the value order).  Each thread then encodes its 8 values into
// 4 packed bytes and stores one 32-bit word; the block leader gathers the 4
// scale bytes into one 32-bit word.  Both kernels are dependent launches: they
// are scheduled while the previous kernel finishes and wait for it before
// reading their inputs.
#include "common.cuh"
#include "launch.h"

namespace idx {

namespace {

constexpr int kThreadsPerVec = 16;
constexpr int kBlockThreads = 256;
constexpr int kVecsPerBlock = kBlockThreads / kThreadsPerVec;

// Quantise the 8 values held by this thread (as 4 x bf16x2 words) of a vector
// whose 16 owner threads are lanes [16*g, 16*g + 16) of the warp.  Returns the
// 4 packed value bytes; *scales_word gets the vector's 4 scale bytes (valid in
// every lane).
__device__ __forceinline__ uint32_t encode8(uint4 raw, uint32_t* scales_word) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    amax = max(amax, w[i] & 0x7FFFu);
    amax = max(amax, (w[i] >> 16) & 0x7FFFu);
  }
  // four consecutive lanes hold one block of 32
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  const uint32_t s = ue8m0_of_amax(amax << 16);
  const float inv = inv_scale_of(s);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = e2m1_code(w[i] & 0xFFFFu, inv);
    const uint32_t hi = e2m1_code(w[i] >> 16, inv);
    packed |= (lo | (hi << 4)) << (8 * i);
  }
  // gather the 4 block scales of this vector: blocks live in lanes 0,4,8,12 of
  // the 16-lane group
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t base = lane & 16u;
  const uint32_t s0 = __shfl_sync(0xFFFFFFFFu, s, base + 0);
  const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, s, base + 4);
  const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, s, base + 8);
  const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, s, base + 12);
  *scales_word = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
  return packed;
}

__global__ void __launch_bounds__(kBlockThreads) quant_insert_kernel(
    const uint16_t* __restrict__ k, int64_t n_tokens, int64_t row_stride,
    const int64_t* __restrict__ slots, uint8_t* __restrict__ cache, int64_t num_slots,
    idx_device_errors* errors) {
  const int64_t vec = (int64_t)blockIdx.x * kVecsPerBlock + threadIdx.x / kThreadsPerVec;
  const int part = threadIdx.x % kThreadsPerVec;
  // whole warps stay converged through the shuffles: a vector index past the
  // end still runs the arithmetic on zeros and skips the stores
  const bool live = vec < n_tokens;
  int64_t slot = -1;
  uint4 raw = make_uint4(0, 0, 0, 0);
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
  if (live) {
    slot = __ldg(slots + vec);
    raw = __ldg(reinterpret_cast<const uint4*>(k + vec * row_stride) + part);
  }
  uint32_t scales;
  const uint32_t packed = encode8(raw, &scales);
  if (!live || slot == -1) return;
  if (slot < 0 || slot >= num_slots) {
    if (part == 0) count_bad_input(errors);
    return;
  }
  const int64_t page = slot / kPage, off = slot % kPage;
  uint8_t* pg = cache + page * kPageBytes;
  reinterpret_cast<uint32_t*>(pg + off * kValBytes)[part] = packed;
  if (part == 0) *reinterpret_cast<uint32_t*>(pg + kPageValBytes + off * kScaleBytes) = scales;
}

__global__ void __launch_bounds__(kBlockThreads) quant_q_kernel(const uint16_t* __restrict__ q,
                                                                int64_t rows,
                                                                uint8_t* __restrict__ vals,
                                                                uint8_t* __restrict__ scales) {
  const int64_t vec = (int64_t)blockIdx.x * kVecsPerBlock + threadIdx.x / kThreadsPerVec;
  const int part = threadIdx.x % kThreadsPerVec;
  const bool live = vec < rows;
  uint4 raw = make_uint4(0, 0, 0, 0);
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
  if (live) raw = __ldg(reinterpret_cast<const uint4*>(q + vec * kHeadDim) + part);
  uint32_t sw;
  const uint32_t packed = encode8(raw, &sw);
  if (!live) return;
  reinterpret_cast<uint32_t*>(vals + vec * kValBytes)[part] = packed;
  if (part == 0) reinterpret_cast<uint32_t*>(scales)[vec] = sw;
}

}  // namespace

cudaError_t launch_quant_insert(const void* k, int64_t n_tokens, int64_t row_stride,
                                const int64_t* slots, uint8_t* cache, int64_t num_blocks,
                                idx_device_errors* errors, cudaStream_t stream) {
  if (n_tokens == 0) return cudaSuccess;
  const int64_t blocks = (n_tokens + kVecsPerBlock - 1) / kVecsPerBlock;
  return launch_dependent(quant_insert_kernel, dim3((unsigned)blocks), dim3(kBlockThreads), 0,
                          stream, static_cast<const uint16_t*>(k), n_tokens, row_stride, slots,
                          cache, num_blocks * kPage, errors);
}

cudaError_t launch_quant_q(const void* q, int64_t rows, uint8_t* vals, uint8_t* scales,
                           cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + kVecsPerBlock - 1) / kVecsPerBlock;
  return launch_dependent(quant_q_kernel, dim3((unsigned)blocks), dim3(kBlockThreads), 0, stream,
                          static_cast<const uint16_t*>(q), rows, vals, scales);
}

}  // namespace idx
