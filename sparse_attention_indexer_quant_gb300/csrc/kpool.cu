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
// One warp per kPoolWarpRows consecutive batch rows (eight warps per CTA): the
// warp reads their slots at once and forms the pools they complete, one after
// the other (with pools of 4, two per warp: the grid, a sixteenth of the rows
// in warps, is resident in one wave at the kernel's register use, where four
// rows a warp took two waves and 14.3 against 12.5 us on 32768 keys).  Lane l forms kc
// for dimensions 4l .. 4l+3 in two passes over the pool (the maximum, then
// the exponentials, so no term overflows), with 16-byte gate / position-term
// loads when those arrays allow it; shuffles then give each of the encoder's
// 16 lanes its eight dimensions.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mxfp4_encode.cuh"

namespace idx {
namespace {

constexpr int kPoolWarps = 8;     // warps per CTA
constexpr int kPoolWarpRows = 8;  // batch rows per warp

template <bool VEC>
__device__ __forceinline__ float4 load4(const float* __restrict__ a, int64_t i) {
  if (VEC) return __ldg(reinterpret_cast<const float4*>(a + i));
  return make_float4(__ldg(a + i), __ldg(a + i + 1), __ldg(a + i + 2), __ldg(a + i + 3));
}

// The pool completed by row p, quantised and stored at `slot`.  All 32 lanes call it.
template <bool VEC>
__device__ __forceinline__ void kpool_row(const uint16_t* __restrict__ k,
                                          const float* __restrict__ gate,
                                          const float* __restrict__ ape, int64_t p, int32_t P,
                                          int64_t slot, uint8_t* __restrict__ cache,
                                          float* __restrict__ pooled, int lane) {
  const int64_t r0 = p - P + 1;  // the pool's first row
  const int d0 = 4 * lane;
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  for (int j = 0; j < P; ++j) {
    // the second pass's keys start on their way to L1 with the first pass's loads
    asm volatile("prefetch.global.L1 [%0];" ::"l"(k + (r0 + j) * kHeadDim + d0));
    const float4 g = load4<VEC>(gate, (r0 + j) * kHeadDim + d0);
    const float4 a = load4<VEC>(ape, (int64_t)j * kHeadDim + d0);
    m[0] = fmaxf(m[0], g.x + a.x);
    m[1] = fmaxf(m[1], g.y + a.y);
    m[2] = fmaxf(m[2], g.z + a.z);
    m[3] = fmaxf(m[3], g.w + a.w);
  }
  float den[4] = {0.f, 0.f, 0.f, 0.f}, num[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < P; ++j) {
    const float4 g = load4<VEC>(gate, (r0 + j) * kHeadDim + d0);
    const float4 a = load4<VEC>(ape, (int64_t)j * kHeadDim + d0);
    const uint2 kb = __ldg(reinterpret_cast<const uint2*>(k + (r0 + j) * kHeadDim + d0));
    const float s[4] = {g.x + a.x, g.y + a.y, g.z + a.z, g.w + a.w};
    const float kv[4] = {__uint_as_float(kb.x << 16), __uint_as_float(kb.x & 0xFFFF0000u),
                         __uint_as_float(kb.y << 16), __uint_as_float(kb.y & 0xFFFF0000u)};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float e = expf(s[q] - m[q]);
      den[q] += e;
      num[q] = fmaf(e, kv[q], num[q]);
    }
  }
  float kc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) kc[q] = num[q] / den[q];
  if (pooled != nullptr) {
    float* o = pooled + p * kHeadDim + d0;
    if (VEC) {
      *reinterpret_cast<float4*>(o) = make_float4(kc[0], kc[1], kc[2], kc[3]);
    } else {
      o[0] = kc[0]; o[1] = kc[1]; o[2] = kc[2]; o[3] = kc[3];
    }
  }
  // encoder lane `part` (lanes 16-31 repeat 0-15: the encoder's shuffles
  // need the whole warp) takes dimensions 8 part .. 8 part + 7 from lanes
  // 2 part and 2 part + 1
  const int part = lane & 15;
  float x[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[q] = __shfl_sync(0xFFFFFFFFu, kc[q], 2 * part);
    x[4 + q] = __shfl_sync(0xFFFFFFFFu, kc[q], 2 * part + 1);
  }
  uint32_t sw;
  const uint32_t packed = encode8_f32(x, &sw);
  if (lane >= 16) return;
  const int64_t page = slot / kPage, off = slot % kPage;
  uint8_t* pg = cache + page * kPageBytes;
  reinterpret_cast<uint32_t*>(pg + off * kValBytes)[part] = packed;
  if (part == 0) *reinterpret_cast<uint32_t*>(pg + kPageValBytes + off * kScaleBytes) = sw;
}

template <bool VEC>
__global__ void __launch_bounds__(32 * kPoolWarps) kpool_insert_kernel(
    const uint16_t* __restrict__ k, const float* __restrict__ gate, const float* __restrict__ ape,
    const int64_t* __restrict__ slots, int64_t n, int32_t P, uint8_t* __restrict__ cache,
    int64_t num_slots, float* __restrict__ pooled, idx_device_errors* errors) {
  const int64_t p0 = ((int64_t)blockIdx.x * kPoolWarps + threadIdx.x / 32) * kPoolWarpRows;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
  // lane r < kPoolWarpRows reads row p0 + r's slot; a row completes a pool
  // in this batch iff its slot is valid and p >= P - 1
  int64_t slot = -1;
  const int64_t pr = p0 + lane;
  if (lane < kPoolWarpRows && pr < n && pr >= P - 1) slot = __ldg(slots + pr);
  const bool bad = slot >= num_slots;
  if (bad) count_bad_input(errors);
  uint32_t todo = __ballot_sync(0xFFFFFFFFu, slot >= 0 && !bad);
  for (; todo != 0u; todo &= todo - 1u) {
    const int r = __ffs(todo) - 1;
    kpool_row<VEC>(k, gate, ape, p0 + r, P, __shfl_sync(0xFFFFFFFFu, slot, r), cache, pooled,
                   lane);
  }
}

}  // namespace

cudaError_t launch_kpool_insert(const void* k, const float* gate, const float* ape,
                                const int64_t* slots, int64_t n, int32_t kpool, uint8_t* cache,
                                int64_t num_blocks, float* pooled, idx_device_errors* errors,
                                cudaStream_t stream) {
  if (n < kpool || n == 0) return cudaSuccess;  // no pool completes in this batch
  const bool vec = (reinterpret_cast<uintptr_t>(gate) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(ape) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(pooled) & 15u) == 0;
  constexpr int64_t per_cta = (int64_t)kPoolWarps * kPoolWarpRows;
  const dim3 grid((unsigned)((n + per_cta - 1) / per_cta));
  const uint16_t* kb = static_cast<const uint16_t*>(k);
  if (vec)
    return launch_dependent(kpool_insert_kernel<true>, grid, dim3(32 * kPoolWarps), 0, stream, kb,
                            gate, ape, slots, n, kpool, cache, num_blocks * kPage, pooled, errors);
  return launch_dependent(kpool_insert_kernel<false>, grid, dim3(32 * kPoolWarps), 0, stream, kb,
                          gate, ape, slots, n, kpool, cache, num_blocks * kPage, pooled, errors);
}

}  // namespace idx
