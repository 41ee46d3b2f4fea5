// Gather of cached MXFP4 keys into contiguous value/scale arrays (vLLM PR
// #48558 "[Kernel] MXFP4 indexer cache for GLM-5.2 / DSA", "Live validation"
// comment: the shared cp_gather reader of the block-split layout).
//
// A CTA copies one page (64 tokens) of one sequence: 4 threads per token move
// its 64 value bytes as 16-byte words and one of them its 4 scale bytes.
#include "common.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) gather_k_kernel(
    const uint8_t* __restrict__ cache, int64_t num_blocks, const int32_t* __restrict__ bt,
    int32_t max_blocks, const int32_t* __restrict__ seq_lens,
    const int64_t* __restrict__ out_offsets, uint8_t* __restrict__ k_vals,
    uint8_t* __restrict__ k_scales, int64_t out_rows, idx_device_errors* errors) {
  const int b = blockIdx.y;
  const int page_idx = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from the previous kernel
  // the length, the page id and the output offset are read together (the
  // page id of a page past the sequence is read but not used)
  int64_t len = __ldg(seq_lens + b);
  const int32_t id = __ldg(bt + (int64_t)b * max_blocks + page_idx);
  const int64_t base = __ldg(out_offsets + b);
  const int64_t cap = (int64_t)max_blocks * kPage;
  if (len < 0 || len > cap) {
    if (page_idx == 0 && threadIdx.x == 0) count_bad_input(errors);
    len = len < 0 ? 0 : cap;
  }
  const int64_t s0 = (int64_t)page_idx * kPage;
  if (s0 >= len) return;
  if (id < 0 || id >= num_blocks) {
    if (threadIdx.x == 0) count_bad_input(errors);
    return;
  }
  const int tok = threadIdx.x >> 2, part = threadIdx.x & 3;
  const int64_t s = s0 + tok;
  if (s >= len) return;
  const int64_t dst = base + s;
  if (dst < 0 || dst >= out_rows) {
    if (part == 0) count_bad_input(errors);
    return;
  }
  const uint8_t* pg = cache + (int64_t)id * kPageBytes;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(pg + tok * kValBytes) + part);
  reinterpret_cast<uint4*>(k_vals + dst * kValBytes)[part] = v;
  if (part == 0)
    reinterpret_cast<uint32_t*>(k_scales)[dst] =
        __ldg(reinterpret_cast<const uint32_t*>(pg + kPageValBytes) + tok);
}

}  // namespace

cudaError_t launch_gather_k(const uint8_t* cache, int64_t num_blocks, const int32_t* block_table,
                            int32_t max_blocks, const int32_t* seq_lens,
                            const int64_t* out_offsets, int32_t B, uint8_t* k_vals,
                            uint8_t* k_scales, int64_t out_rows, idx_device_errors* errors,
                            cudaStream_t stream) {
  if (B == 0 || max_blocks == 0) return cudaSuccess;
  return launch_dependent(gather_k_kernel, dim3((unsigned)max_blocks, (unsigned)B),
                          dim3(kGatherThreads), 0, stream, cache, num_blocks, block_table,
                          max_blocks, seq_lens, out_offsets, k_vals, k_scales, out_rows, errors);
}

}  // namespace idx
