// Top-k per logits row (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// top_k_per_row into topk_indices_buffer; the rows shorter than k are padded
// with -1).
//
// One CTA per row.  The first digit's histogram is taken straight from the row
// in global memory; the elements in the threshold bin are then compacted into
// shared memory (when they fit) while the elements above it are emitted, and
// the remaining digits run on the compacted set.
#include "common.cuh"
#include "launch.h"
#include "topk_select.cuh"

namespace idx {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kCandCap = 4096;

struct GlobalRow {
  const float* x;
  int64_t n;
  template <class F>
  __device__ __forceinline__ void for_each(F f) const {
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) f(float_key(__ldg(x + i)), (int32_t)i);
  }
};

struct TopkSmem {
  SelectScratch sc;
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
  const GlobalRow src{logits + row * ld + st, len};
  if (threadIdx.x == 0) {
    sm.sc.out_count = 0;
    sm.n_cand = 0;
  }
  auto emit = [&](uint32_t, int32_t idx) { orow[atomicAdd(&sm.sc.out_count, 1u)] = idx; };

  digit_histogram(sm.sc, src, 0, 0u, 0u);
  find_threshold_bin(sm.sc, kRadixBins, (uint32_t)k);
  const uint32_t b1 = sm.sc.bin;
  const uint32_t need = (uint32_t)k - sm.sc.above;
  const bool fits = sm.sc.hist[b1] <= (uint32_t)kCandCap;
  __syncthreads();
  src.for_each([&](uint32_t key, int32_t idx) {
    const uint32_t dg = key >> 21;
    if (dg > b1) {
      emit(key, idx);
    } else if (dg == b1 && fits) {
      const uint32_t slot = atomicAdd(&sm.n_cand, 1u);
      sm.cand_keys[slot] = key;
      sm.cand_idx[slot] = idx;
    }
  });
  __syncthreads();
  const uint32_t prefix = b1 << 21, mask = 0x7FFu << 21;
  if (fits) {
    const SmemPairs cand{sm.cand_keys, sm.cand_idx, (int)sm.n_cand};
    radix_select(sm.sc, cand, need, 1, prefix, mask, emit);
  } else {
    radix_select(sm.sc, src, need, 1, prefix, mask, emit);
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
