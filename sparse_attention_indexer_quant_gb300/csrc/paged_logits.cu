// Paged decode logits over the MXFP4 K-cache (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": paged_mqa_logits; vLLM PR #48558
// "[Kernel] MXFP4 indexer cache for GLM-5.2 / DSA", section "Notes": the paged
// MQA-logits reader), computing for query row r = (b, j)
//     logit[r, s] = sum_h w[r, h] * max(0, q^[r, h] . k^[s]).
//
// The persistent main loop of paged_core.cuh streams each sequence's pages
// (cp.async) through tcgen05 block-scaled MXF4 MMAs; this file's epilogue forms
// sum_h w * max(0, D) for each of the next_n query rows of a key and writes it
// to the logits row (-inf past the window when the rows are clean).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"

namespace idx {
namespace {

template <int H, int NEXT_N>
struct UnfusedEpilogue {
  static constexpr int NH = H * NEXT_N;
  static constexpr size_t kExtraSmem = 0;
  __device__ __forceinline__ static void init(uint8_t*) {}

  // Called once per tile by every epilogue thread with its key's dot products
  // for queries j0 .. j0 + NJ - 1 (column n = (j - j0)*H + h; w_smem points at
  // query j0's weights).
  template <int NJ>
  __device__ __forceinline__ static void tile(const PagedArgs& p, const ItemDesc& it,
                                              const float* w_smem, uint8_t* /*extra*/,
                                              int64_t key, const float (&d)[NJ * H], int j0) {
    float logit[NJ];
    weighted_relu_sum<H, NJ>(w_smem, d, logit);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const int j = j0 + jj;
      const int64_t len = it.L - NEXT_N + j + 1;
      float* row = p.logits + ((int64_t)it.b * NEXT_N + j) * p.ld;
      if (key < len)
        row[key] = logit[jj];
      else if (p.clean && key < p.ld)
        row[key] = -INFINITY;
    }
  }

  // -inf into the item's columns that no tile covered (clean rows only), by
  // the epilogue threads [0, epi_threads).
  __device__ __forceinline__ static void item_done(const PagedArgs& p, const ItemDesc& it,
                                                   uint8_t*, int epi_threads) {
    if (!p.clean) return;
    const int64_t lo = it.k0 + (int64_t)it.n_tiles * kTileKeys;
    const int64_t hi = it.k_end < p.ld ? it.k_end : p.ld;
    const int e = threadIdx.x;
    for (int j = 0; j < NEXT_N; ++j) {
      float* row = p.logits + ((int64_t)it.b * NEXT_N + j) * p.ld;
      for (int64_t s = lo + e; s < hi; s += epi_threads) row[s] = -INFINITY;
    }
  }
};

// STEP: the decode step's scoring pass, which prepares each sequence (its
// query heads quantised, its new keys inserted) before scoring its items
// (step_prepare_sequence).
template <int H, int NEXT_N, bool STEP>
__global__ void __launch_bounds__(paged_threads(H * NEXT_N), paged_ctas_per_sm(H * NEXT_N))
    paged_logits_kernel(const PagedArgs p) {
  paged_persistent_run<H, NEXT_N, UnfusedEpilogue<H, NEXT_N>, STEP>(
      p, p.kcache, p.item_counter != nullptr, p.clean != 0, p.item_counter);
}

template <int H, int NEXT_N, bool STEP>
cudaError_t launch_one(const PagedArgs& a, cudaStream_t stream) {
  using Ep = UnfusedEpilogue<H, NEXT_N>;
  const size_t smem = paged_smem_bytes<H * NEXT_N>() + Ep::kExtraSmem;
  auto kern = paged_logits_kernel<H, NEXT_N, STEP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3((unsigned)a.grid), dim3(paged_threads(H * NEXT_N)), smem,
                          stream, a);
}

template <bool STEP>
cudaError_t launch_shape(int H, int next_n, const PagedArgs& a, cudaStream_t stream) {
  if (H == 32 && next_n == 1) return launch_one<32, 1, STEP>(a, stream);
  if (H == 32 && next_n == 2) return launch_one<32, 2, STEP>(a, stream);
  if (H == 64 && next_n == 1) return launch_one<64, 1, STEP>(a, stream);
  if (H == 64 && next_n == 2) return launch_one<64, 2, STEP>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_paged_logits(int H, int next_n, const PagedArgs& a, cudaStream_t stream) {
  return a.seq_state != nullptr ? launch_shape<true>(H, next_n, a, stream)
                               : launch_shape<false>(H, next_n, a, stream);
}

}  // namespace idx
