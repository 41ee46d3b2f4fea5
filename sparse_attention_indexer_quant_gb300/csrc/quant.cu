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
#include "mxfp4_encode.cuh"

namespace idx {

namespace {

constexpr int kThreadsPerVec = 16;
constexpr int kBlockThreads = 256;
constexpr int kVecsPerBlock = kBlockThreads / kThreadsPerVec;

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

// Rotary embedding of the query heads fused with their quantisation (vLLM PR
// #48558 "Notes": a fused q-rope + MXFP4 q-quant): the thread owning elements
// [8*part, 8*part + 8) turns its pairs (2i, 2i+1) with i < rot_dim / 2 by the
// angle of table column i at the token's position, in fp32 with the products
// y*sin and y*cos rounded first and then one fused multiply-add each, and the
// 16 threads of the vector encode the result.  A token whose position is
// outside the table is skipped (its rows are not written) and counted.
// A group takes VPG consecutive vectors (usually heads of one token): all of
// their query loads and positions are issued first, then all of their table
// loads (one 16-byte load per table and vector for a thread whose four pairs
// are rotated), so that a thread waits for two round trips per VPG vectors.
template <int VPG>
__global__ void __launch_bounds__(kBlockThreads) rope_quant_q_kernel(
    const uint16_t* __restrict__ q, int64_t T, int32_t H, const int32_t* __restrict__ positions,
    const float* __restrict__ cs, const float* __restrict__ sn, int32_t num_pos, int32_t rot_dim,
    uint8_t* __restrict__ vals, uint8_t* __restrict__ scales, idx_device_errors* errors) {
  const int64_t vec0 = ((int64_t)blockIdx.x * kVecsPerBlock + threadIdx.x / kThreadsPerVec) * VPG;
  const int part = threadIdx.x % kThreadsPerVec;
  const int64_t rows = T * H;
  const int half = rot_dim / 2;
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
  // whole warps stay converged through the shuffles: rows past the end and
  // tokens off the table run the arithmetic on zeros and skip the stores
  const int64_t t0 = vec0 / H;
  const int32_t h0 = (int32_t)(vec0 - t0 * H);
  uint4 raw[VPG];
  int32_t pos[VPG];
  bool live[VPG];
#pragma unroll
  for (int u = 0; u < VPG; ++u) {
    const int64_t vec = vec0 + u;
    live[u] = vec < rows;
    raw[u] = make_uint4(0, 0, 0, 0);
    pos[u] = 0;
    if (live[u]) {
      raw[u] = __ldg(reinterpret_cast<const uint4*>(q + vec * kHeadDim) + part);
      // no table without rotated pairs
      if (half > 0) pos[u] = __ldg(positions + t0 + (h0 + u) / H);
    }
  }
  const int col0 = 4 * part;
  float c[VPG][4], s[VPG][4];
#pragma unroll
  for (int u = 0; u < VPG; ++u) {
    if (live[u] && half > 0 && (pos[u] < 0 || pos[u] >= num_pos)) {
      if (part == 0 && (h0 + u) % H == 0) count_bad_input(errors);
      live[u] = false;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      c[u][i] = 1.f;
      s[u][i] = 0.f;
    }
    // the thread's four pairs use table columns 4 * part .. 4 * part + 3
    if (live[u] && col0 < half) {
      const float* c_row = cs + (int64_t)pos[u] * half + col0;
      const float* s_row = sn + (int64_t)pos[u] * half + col0;
      if (col0 + 3 < half &&
          ((reinterpret_cast<uintptr_t>(c_row) | reinterpret_cast<uintptr_t>(s_row)) & 15u) == 0) {
        const float4 cv = __ldg(reinterpret_cast<const float4*>(c_row));
        const float4 sv = __ldg(reinterpret_cast<const float4*>(s_row));
        c[u][0] = cv.x; c[u][1] = cv.y; c[u][2] = cv.z; c[u][3] = cv.w;
        s[u][0] = sv.x; s[u][1] = sv.y; s[u][2] = sv.z; s[u][3] = sv.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (col0 + i < half) {
            c[u][i] = __ldg(c_row + i);
            s[u][i] = __ldg(s_row + i);
          }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < VPG; ++u) {
    float x[8];
    bf16x8_to_f32(raw[u], x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (col0 + i < half) {  // pair (8 * part + 2i, 8 * part + 2i + 1)
        const float a = x[2 * i], b = x[2 * i + 1];
        x[2 * i] = __fmaf_rn(a, c[u][i], -__fmul_rn(b, s[u][i]));
        x[2 * i + 1] = __fmaf_rn(a, s[u][i], __fmul_rn(b, c[u][i]));
      }
    }
    uint32_t sw;
    const uint32_t packed = encode8_f32(x, &sw);
    if (!live[u]) continue;
    const int64_t vec = vec0 + u;
    reinterpret_cast<uint32_t*>(vals + vec * kValBytes)[part] = packed;
    if (part == 0) reinterpret_cast<uint32_t*>(scales)[vec] = sw;
  }
}

}  // namespace

cudaError_t launch_rope_quant_q(const void* q, int64_t T, int32_t H, const int32_t* positions,
                                const float* cs, const float* sn, int32_t num_pos,
                                int32_t rot_dim, uint8_t* vals, uint8_t* scales,
                                idx_device_errors* errors, cudaStream_t stream) {
  const int64_t rows = T * H;
  if (rows == 0) return cudaSuccess;
  const uint16_t* qb = static_cast<const uint16_t*>(q);
  if (rows >= kBigRows) {
    const int64_t per_block = (int64_t)kVecsPerBlock * kBigVpg;
    return launch_dependent(rope_quant_q_kernel<kBigVpg>,
                            dim3((unsigned)((rows + per_block - 1) / per_block)),
                            dim3(kBlockThreads), 0, stream, qb, T, H, positions, cs, sn, num_pos,
                            rot_dim, vals, scales, errors);
  }
  const int64_t blocks = (rows + kVecsPerBlock - 1) / kVecsPerBlock;
  return launch_dependent(rope_quant_q_kernel<1>, dim3((unsigned)blocks), dim3(kBlockThreads), 0,
                          stream, qb, T, H, positions, cs, sn, num_pos, rot_dim, vals, scales,
                          errors);
}

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
