// K-pool compressed insert (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": _kpool_compress_insert).
//
// The slot mapping is pool-granular: row p of the batch completes a pool, and
// is written, iff slot[p] >= 0 and p >= P - 1 (a valid slot earlier belongs
// to a pool that began before the batch); nothing is written when the batch
// is shorter than one pool.  The masking happens in the kernel, so the host
// neither compacts the rows nor synchronises.  The pool of row p is rows
// p - P + 1 .. p; per dimension d its keys are weighted by a softmax over the
// pool of gate[row, d] + ape[j, d] (j: position in the pool) and summed:
//     kc[d] = sum_j softmax_j(gate + ape) * k[p - P + 1 + j, d]      (fp32)
// and kc is quantised to MXFP4 like a key and stored at slot[p].
//
// One CTA of 128 threads per batch row: thread d forms kc[d] in two passes
// over the pool (the maximum, then the exponentials, so no term overflows);
// the vector goes through shared memory to the encoder's 16-thread layout.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mxfp4_encode.cuh"

namespace idx {
namespace {

constexpr int kPoolThreads = kHeadDim;  // one thread per dimension

__global__ void __launch_bounds__(kPoolThreads) kpool_insert_kernel(
    const uint16_t* __restrict__ k, const float* __restrict__ gate, const float* __restrict__ ape,
    const int64_t* __restrict__ slots, int64_t n, int32_t P, uint8_t* __restrict__ cache,
    int64_t num_slots, float* __restrict__ pooled, idx_device_errors* errors) {
  __shared__ __align__(16) float kc_s[kHeadDim];
  const int64_t p = blockIdx.x;
  const int d = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
  const int64_t slot = __ldg(slots + p);
  if (slot < 0 || p < P - 1) return;  // not a pool completion in this batch
  if (slot >= num_slots) {
    if (d == 0) count_bad_input(errors);
    return;
  }
  const int64_t r0 = p - P + 1;  // the pool's first row
  float m = -INFINITY;
  for (int j = 0; j < P; ++j)
    m = fmaxf(m, __ldg(gate + (r0 + j) * kHeadDim + d) + __ldg(ape + (int64_t)j * kHeadDim + d));
  float den = 0.f, num = 0.f;
  for (int j = 0; j < P; ++j) {
    const float e =
        expf(__ldg(gate + (r0 + j) * kHeadDim + d) + __ldg(ape + (int64_t)j * kHeadDim + d) - m);
    const float kv = __uint_as_float((uint32_t)__ldg(k + (r0 + j) * kHeadDim + d) << 16);
    den += e;
    num = fmaf(e, kv, num);
  }
  const float kc = num / den;
  if (pooled != nullptr) pooled[p * kHeadDim + d] = kc;
  kc_s[d] = kc;
  __syncthreads();
  if (threadIdx.x >= 32) return;
  // the first 16 lanes encode the vector (the encoder's shuffles need the
  // whole warp; lanes 16-31 work on a copy and store nothing)
  const int part = threadIdx.x & 15;
  float x[8];
  const float4 lo = *reinterpret_cast<const float4*>(kc_s + 8 * part);
  const float4 hi = *reinterpret_cast<const float4*>(kc_s + 8 * part + 4);
  x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
  x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
  uint32_t sw;
  const uint32_t packed = encode8_f32(x, &sw);
  if (threadIdx.x >= 16) return;
  const int64_t page = slot / kPage, off = slot % kPage;
  uint8_t* pg = cache + page * kPageBytes;
  reinterpret_cast<uint32_t*>(pg + off * kValBytes)[part] = packed;
  if (part == 0) *reinterpret_cast<uint32_t*>(pg + kPageValBytes + off * kScaleBytes) = sw;
}

}  // namespace

cudaError_t launch_kpool_insert(const void* k, const float* gate, const float* ape,
                                const int64_t* slots, int64_t n, int32_t kpool, uint8_t* cache,
                                int64_t num_blocks, float* pooled, idx_device_errors* errors,
                                cudaStream_t stream) {
  if (n < kpool || n == 0) return cudaSuccess;  // no pool completes in this batch
  return launch_dependent(kpool_insert_kernel, dim3((unsigned)n), dim3(kPoolThreads), 0, stream,
                          static_cast<const uint16_t*>(k), gate, ape, slots, n, kpool, cache,
                          num_blocks * kPage, pooled, errors);
}

}  // namespace idx
