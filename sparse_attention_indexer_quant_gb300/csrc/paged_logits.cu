// Paged decode logits over the MXFP4 K-cache (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": paged_mqa_logits; vLLM PR #48558
// "[Kernel] MXFP4 indexer cache for GLM-5.2 / DSA", section "Notes": the paged
// MQA-logits reader), computing for query row r = (b, j)
//     logit[r, s] = sum_h w[r, h] * max(0, q^[r, h] . k^[s]).
//
// One CTA scores a chunk of one sequence's context, 128 keys (two pages) per
// tile, with three warp roles:
//   warp 0      TMA producer: reads the block table and issues, per tile, two
//               64x64-byte value boxes (64-byte swizzle) and two 256-byte scale
//               boxes, gathered by page id, into a ring of shared-memory stages;
//   warp 1      MMA issuer: rearranges the tile's 128 scale words into the
//               32x16-byte scale-factor layout, copies it to tensor memory with
//               tcgen05.cp, and issues two tcgen05.mma kind::mxf4 block-scaled
//               MMAs (K = 64 each): D[key, j*H + h] in TMEM, fp32;
//   warps 2-5   epilogue: one thread per key (TMEM lane) loads its row of D and
//               forms sum_h w * max(0, D) for each of the next_n query rows.
// The query heads of the sequence (the MMA's B operand, N = next_n * H rows)
// and their scale factors are staged once per CTA.
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

  // Called once per tile by every epilogue thread with its key's NH dot
  // products (column n = j*H + h).
  __device__ __forceinline__ static void tile(const PagedArgs& p, const PagedCta& c,
                                              const float* w_smem, uint8_t* /*extra*/,
                                              int64_t key, const float (&d)[NH]) {
    float logit[NEXT_N];
    weighted_relu_sum<H, NEXT_N>(w_smem, d, logit);
#pragma unroll
    for (int j = 0; j < NEXT_N; ++j) {
      const int64_t len = c.L - NEXT_N + j + 1;
      float* row = p.logits + ((int64_t)c.b * NEXT_N + j) * p.ld;
      if (key < len)
        row[key] = logit[j];
      else if (p.clean && key < p.ld)
        row[key] = -INFINITY;
    }
  }
  __device__ __forceinline__ static void chunk_done(const PagedArgs&, const PagedCta&, uint8_t*,
                                                    bool) {}
};

template <int H, int NEXT_N>
__global__ void __launch_bounds__(kPagedThreads, 1)
    paged_logits_kernel(const __grid_constant__ CUtensorMap tm_vals,
                        const __grid_constant__ CUtensorMap tm_scales, const PagedArgs p) {
  PagedCta c;
  if (!paged_cta_setup(p, c)) {
    if (p.clean) clean_tail<NEXT_N>(p, c);
    return;
  }
  if (p.clean) clean_tail<NEXT_N>(p, c);
  paged_cta_run<H, NEXT_N, UnfusedEpilogue<H, NEXT_N>>(&tm_vals, &tm_scales, p, c);
}

template <int H, int NEXT_N>
cudaError_t launch_one(const CUtensorMap& tv, const CUtensorMap& ts, const PagedArgs& a,
                       cudaStream_t stream) {
  using Ep = UnfusedEpilogue<H, NEXT_N>;
  const size_t smem = paged_smem_bytes<H * NEXT_N>() + Ep::kExtraSmem;
  auto kern = paged_logits_kernel<H, NEXT_N>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.chunks, (unsigned)a.B);
  kern<<<grid, kPagedThreads, smem, stream>>>(tv, ts, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_logits(const CUtensorMap& tv, const CUtensorMap& ts, int H, int next_n,
                                const PagedArgs& a, cudaStream_t stream) {
  if (H == 32 && next_n == 1) return launch_one<32, 1>(tv, ts, a, stream);
  if (H == 32 && next_n == 2) return launch_one<32, 2>(tv, ts, a, stream);
  if (H == 64 && next_n == 1) return launch_one<64, 1>(tv, ts, a, stream);
  if (H == 64 && next_n == 2) return launch_one<64, 2>(tv, ts, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace idx
