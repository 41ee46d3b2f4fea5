// Top-k per logits row (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// top_k_per_row into topk_indices_buffer; the rows shorter than k are padded
// with -1).
//
// One CTA per row.  Pass 1 builds the coarse histogram of the row straight
// from global memory; pass 2 emits the elements above the boundary bin and
// compacts the boundary bin's elements into shared memory (when they fit),
// where the exact threshold is found; otherwise the exact passes read the row
// again, restricted to the boundary bin.
#include "common.cuh"
#include "launch.h"
#include "topk_select.cuh"

namespace idx {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kCandCap = 3584;

struct TopkSmem {
  SelectScratch sel;
  uint32_t cand_keys[kCandCap];
  int32_t cand_idx[kCandCap];
  uint32_t n_cand;
};

__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(const float* __restrict__ logits,
                                                                  int64_t ld,
                                                                  const int32_t* row_start,
                                                                  const int32_t* row_end,
                                                                  int32_t k, int32_t* out) {
  __shared__ TopkSmem sm;
  const int64_t row = blockIdx.x;
  const int64_t st = row_start != nullptr ? __ldg(row_start + row) : 0;
  const int64_t en = __ldg(row_end + row);
  const int64_t len = en > st ? en - st : 0;
  int32_t* orow = out + row * k;
  if (len <= k) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) orow[i] = i < len ? i : -1;
    return;
  }
  // positions are reported relative to the window start
  const GlobalLogits<false> src{logits + row * ld + st, 0, len};
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) sm.sel.hist[i] = 0;
  if (threadIdx.x == 0) {
    sm.sel.s.count = 0;
    sm.n_cand = 0;
  }
  __syncthreads();
  src.for_each([&](uint32_t key, int32_t) { hist_add(sm.sel.hist, coarse_bin(key), true); });
  __syncthreads();
  find_threshold_bin(sm.sel.hist, kCoarseBins, (uint32_t)k, sm.sel.s);
  const uint32_t b1 = sm.sel.s.bin;
  const uint32_t above = sm.sel.s.above;
  const bool fits = sm.sel.hist[b1] <= (uint32_t)kCandCap;
  __syncthreads();
  src.for_each([&](uint32_t key, int32_t i) {
    const uint32_t bin = coarse_bin(key);
    const uint32_t slot = warp_claim(&sm.sel.s.count, bin > b1);
    if (bin > b1) orow[slot] = i;
    if (bin == b1 && fits) {
      const uint32_t c = atomicAdd(&sm.n_cand, 1u);
      sm.cand_keys[c] = key;
      sm.cand_idx[c] = i;
    }
  });
  __syncthreads();
  auto emit = [&](uint32_t, int32_t i) { orow[warp_claim(&sm.sel.s.count, true)] = i; };
  const uint32_t need = (uint32_t)k - above;
  if (fits) {
    const SmemPairs cand{sm.cand_keys, sm.cand_idx, (int)sm.n_cand};
    radix_select(sm.sel.hist, sm.sel.s, cand, need, b1 << kCoarseShift, 32 - kCoarseShift,
                 emit);
  } else {
    radix_select(sm.sel.hist, sm.sel.s, src, need, b1 << kCoarseShift, 32 - kCoarseShift, emit);
  }
}

}  // namespace

cudaError_t launch_topk_rows(const float* logits, int64_t rows, int64_t ld,
                             const int32_t* row_start, const int32_t* row_end, int32_t k,
                             int32_t* out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  topk_rows_kernel<<<(unsigned)rows, kTopkThreads, 0, stream>>>(logits, ld, row_start, row_end,
                                                                 k, out);
  return cudaGetLastError();
}

}  // namespace idx
