// MXFP4 quantisation kernels: key insert into the paged cache, and query
// quantisation (vLLM PR #48558 "[Kernel] MXFP4 indexer cache for GLM-5.2 / DSA",
// sections "Changes" and "Notes").
//
// Sixteen threads own one 128-element vector at a time (on large inputs four
// vectors per group, loaded together): each loads 8 bf16 values (16 B),
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
  // x * 2^-e is exact for every magnitude that can round to a nonzero code;
  // the hardware convert rounds to nearest with ties to the even code,
  // saturates at 6 and keeps the sign of a value that rounds to zero (the
  // rule of the exhaustive bf16 test); element 2i goes to the low nibble of
  // byte i
  float y[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    y[2 * i] = __uint_as_float(w[i] << 16) * inv;
    y[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u) * inv;
  }
  uint32_t packed;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(packed)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
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

// Each 16-thread group quantises VPG vectors (rows u * gstride + vec for
// u < VPG): all of a thread's loads are issued before any encode, so each
// thread keeps VPG 16-byte loads in flight.  Large inputs take VPG = 4
// (streaming rate); small ones VPG = 1 (the most CTAs, the shortest chain).
constexpr int kBigVpg = 4;
constexpr int64_t kBigRows = 65536;

template <int VPG>
__global__ void __launch_bounds__(kBlockThreads) quant_insert_kernel(
    const uint16_t* __restrict__ k, int64_t n_tokens, int64_t row_stride,
    const int64_t* __restrict__ slots, uint8_t* __restrict__ cache, int64_t num_slots,
    idx_device_errors* errors) {
  const int64_t vec0 = (int64_t)blockIdx.x * kVecsPerBlock + threadIdx.x / kThreadsPerVec;
  const int64_t gstride = (int64_t)gridDim.x * kVecsPerBlock;
  const int part = threadIdx.x % kThreadsPerVec;
  // whole warps stay converged through the shuffles: a vector index past the
  // end still runs the arithmetic on zeros and skips the stores
  int64_t slot[VPG];
  uint4 raw[VPG];
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
#pragma unroll
  for (int u = 0; u < VPG; ++u) {
    const int64_t vec = vec0 + u * gstride;
    slot[u] = -1;
    raw[u] = make_uint4(0, 0, 0, 0);
    if (vec < n_tokens) {
      slot[u] = __ldg(slots + vec);
      raw[u] = __ldg(reinterpret_cast<const uint4*>(k + vec * row_stride) + part);
    }
  }
#pragma unroll
  for (int u = 0; u < VPG; ++u) {
    uint32_t scales;
    const uint32_t packed = encode8(raw[u], &scales);
    const int64_t vec = vec0 + u * gstride;
    if (vec >= n_tokens || slot[u] == -1) continue;
    if (slot[u] < 0 || slot[u] >= num_slots) {
      if (part == 0) count_bad_input(errors);
      continue;
    }
    const int64_t page = slot[u] / kPage, off = slot[u] % kPage;
    uint8_t* pg = cache + page * kPageBytes;
    reinterpret_cast<uint32_t*>(pg + off * kValBytes)[part] = packed;
    if (part == 0) *reinterpret_cast<uint32_t*>(pg + kPageValBytes + off * kScaleBytes) = scales;
  }
}

template <int VPG>
__global__ void __launch_bounds__(kBlockThreads) quant_q_kernel(const uint16_t* __restrict__ q,
                                                                int64_t rows,
                                                                uint8_t* __restrict__ vals,
                                                                uint8_t* __restrict__ scales) {
  const int64_t vec0 = (int64_t)blockIdx.x * kVecsPerBlock + threadIdx.x / kThreadsPerVec;
  const int64_t gstride = (int64_t)gridDim.x * kVecsPerBlock;
  const int part = threadIdx.x % kThreadsPerVec;
  uint4 raw[VPG];
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
#pragma unroll
  for (int u = 0; u < VPG; ++u) {
    const int64_t vec = vec0 + u * gstride;
    raw[u] = vec < rows ? __ldg(reinterpret_cast<const uint4*>(q + vec * kHeadDim) + part)
                        : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < VPG; ++u) {
    uint32_t sw;
    const uint32_t packed = encode8(raw[u], &sw);
    const int64_t vec = vec0 + u * gstride;
    if (vec >= rows) continue;
    reinterpret_cast<uint32_t*>(vals + vec * kValBytes)[part] = packed;
    if (part == 0) reinterpret_cast<uint32_t*>(scales)[vec] = sw;
  }
}

}  // namespace

cudaError_t launch_quant_insert(const void* k, int64_t n_tokens, int64_t row_stride,
                                const int64_t* slots, uint8_t* cache, int64_t num_blocks,
                                idx_device_errors* errors, cudaStream_t stream) {
  if (n_tokens == 0) return cudaSuccess;
  if (n_tokens >= kBigRows) {
    const int64_t per_block = (int64_t)kVecsPerBlock * kBigVpg;
    return launch_dependent(quant_insert_kernel<kBigVpg>,
                            dim3((unsigned)((n_tokens + per_block - 1) / per_block)),
                            dim3(kBlockThreads), 0, stream, static_cast<const uint16_t*>(k),
                            n_tokens, row_stride, slots, cache, num_blocks * kPage, errors);
  }
  const int64_t blocks = (n_tokens + kVecsPerBlock - 1) / kVecsPerBlock;
  return launch_dependent(quant_insert_kernel<1>, dim3((unsigned)blocks), dim3(kBlockThreads), 0,
                          stream, static_cast<const uint16_t*>(k), n_tokens, row_stride, slots,
                          cache, num_blocks * kPage, errors);
}

cudaError_t launch_quant_q(const void* q, int64_t rows, uint8_t* vals, uint8_t* scales,
                           cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (rows >= kBigRows) {
    const int64_t per_block = (int64_t)kVecsPerBlock * kBigVpg;
    return launch_dependent(quant_q_kernel<kBigVpg>,
                            dim3((unsigned)((rows + per_block - 1) / per_block)),
                            dim3(kBlockThreads), 0, stream, static_cast<const uint16_t*>(q), rows,
                            vals, scales);
  }
  const int64_t blocks = (rows + kVecsPerBlock - 1) / kVecsPerBlock;
  return launch_dependent(quant_q_kernel<1>, dim3((unsigned)blocks), dim3(kBlockThreads), 0, stream,
                          static_cast<const uint16_t*>(q), rows, vals, scales);
}

}  // namespace idx
