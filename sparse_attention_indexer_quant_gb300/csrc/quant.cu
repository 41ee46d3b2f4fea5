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
// A group takes VPG consecutive vectors: all of their query loads are issued
// first, then the table loads, so that a thread waits for two round trips per
// VPG vectors.  When VPG divides H (every group holds heads of one token),
// the group reads the token's position and table row once.
__device__ __forceinline__ void rope_table(const float* __restrict__ cs,
                                           const float* __restrict__ sn, int32_t pos, int half,
                                           int col0, float (&c)[4], float (&s)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    c[i] = 1.f;
    s[i] = 0.f;
  }
  if (col0 >= half) return;  // the thread's four pairs use table columns col0 .. col0 + 3
  const float* c_row = cs + (int64_t)pos * half + col0;
  const float* s_row = sn + (int64_t)pos * half + col0;
  if (col0 + 3 < half &&
      ((reinterpret_cast<uintptr_t>(c_row) | reinterpret_cast<uintptr_t>(s_row)) & 15u) == 0) {
    const float4 cv = __ldg(reinterpret_cast<const float4*>(c_row));
    const float4 sv = __ldg(reinterpret_cast<const float4*>(s_row));
    c[0] = cv.x; c[1] = cv.y; c[2] = cv.z; c[3] = cv.w;
    s[0] = sv.x; s[1] = sv.y; s[2] = sv.z; s[3] = sv.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (col0 + i < half) {
        c[i] = __ldg(c_row + i);
        s[i] = __ldg(s_row + i);
      }
  }
}

// Turns the thread's pairs and encodes; stores when live.  All 32 lanes call it.
__device__ __forceinline__ void rope_encode_store(uint4 raw, const float (&c)[4],
                                                  const float (&s)[4], int half, int part,
                                                  bool live, int64_t vec, uint8_t* __restrict__ vals,
                                                  uint8_t* __restrict__ scales) {
  float x[8];
  bf16x8_to_f32(raw, x);
  const int col0 = 4 * part;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (col0 + i < half) {  // pair (8 * part + 2i, 8 * part + 2i + 1)
      const float a = x[2 * i], b = x[2 * i + 1];
      x[2 * i] = __fmaf_rn(a, c[i], -__fmul_rn(b, s[i]));
      x[2 * i + 1] = __fmaf_rn(a, s[i], __fmul_rn(b, c[i]));
    }
  }
  uint32_t sw;
  const uint32_t packed = encode8_f32(x, &sw);
  if (!live) return;
  reinterpret_cast<uint32_t*>(vals + vec * kValBytes)[part] = packed;
  if (part == 0) reinterpret_cast<uint32_t*>(scales)[vec] = sw;
}

template <int VPG>
__global__ void __launch_bounds__(kBlockThreads) rope_quant_q_kernel(
    const uint16_t* __restrict__ q, int64_t T, int32_t H, const int32_t* __restrict__ positions,
    const float* __restrict__ cs, const float* __restrict__ sn, int32_t num_pos, int32_t rot_dim,
    uint8_t* __restrict__ vals, uint8_t* __restrict__ scales, idx_device_errors* errors) {
  const int64_t vec0 = ((int64_t)blockIdx.x * kVecsPerBlock + threadIdx.x / kThreadsPerVec) * VPG;
  const int part = threadIdx.x % kThreadsPerVec;
  const int64_t rows = T * H;
  const int half = rot_dim / 2;
  const int col0 = 4 * part;
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
  // whole warps stay converged through the shuffles: rows past the end and
  // tokens off the table run the arithmetic on zeros and skip the stores
  const int64_t t0 = vec0 / H;
  const int32_t h0 = (int32_t)(vec0 - t0 * H);
  uint4 raw[VPG];
#pragma unroll
  for (int u = 0; u < VPG; ++u)
    raw[u] = vec0 + u < rows ? __ldg(reinterpret_cast<const uint4*>(q + (vec0 + u) * kHeadDim) + part)
                             : make_uint4(0, 0, 0, 0);
  // a position outside the table: the token's rows are skipped, counted once
  // (by the group holding its head 0); no table without rotated pairs
  auto position = [&](int64_t t, int32_t h, bool& live) {
    if (!live || half == 0) return 0;
    const int32_t pos = __ldg(positions + t);
    if (pos < 0 || pos >= num_pos) {
      if (part == 0 && h == 0) count_bad_input(errors);
      live = false;
      return 0;
    }
    return pos;
  };
  if (H % VPG == 0) {  // warp-uniform: every group holds heads h0 .. h0 + VPG - 1 of token t0
    bool ok = vec0 < rows;
    const int32_t pos = position(t0, h0, ok);
    float c[4], s[4];
    rope_table(cs, sn, pos, ok ? half : 0, col0, c, s);
#pragma unroll
    for (int u = 0; u < VPG; ++u)
      rope_encode_store(raw[u], c, s, half, part, ok && vec0 + u < rows, vec0 + u, vals, scales);
  } else {
#pragma unroll
    for (int u = 0; u < VPG; ++u) {
      const int64_t t = t0 + (h0 + u) / H;
      const int32_t h = (h0 + u) % H;
      bool live = vec0 + u < rows;
      const int32_t pos = position(t, h, live);
      float c[4], s[4];
      rope_table(cs, sn, pos, live ? half : 0, col0, c, s);
      rope_encode_store(raw[u], c, s, half, part, live, vec0 + u, vals, scales);
    }
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
