// Paged decode logits + top-k (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// paged_mqa_logits followed by top_k_per_row into topk_indices_buffer), in two
// launches that hand the logits over through the caller's workspace instead of
// a logits tensor:
//
//   1. score    the persistent cp.async + tcgen05 logits kernel, taking work items
//               from a counter in the workspace and writing each row's valid
//               logits to a row-major scratch that stays in L2 for these sizes;
//   2. select   one CTA per row runs row_topk (topk_row.cuh) over the row's
//               window of the scratch logits.
//
// Workspace (device, caller-owned): a u32 work-item counter (zeroed by a
// memset per call), then f32 logits[rows][ldw], ldw = max_blocks * 64.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"
#include "topk_row.cuh"

namespace idx {
namespace {

constexpr int kFusedTilesPerItem = 8;
constexpr int kSelChunk = 32768;
using SelSmem = RowTopkSmem<kSelChunk>;

struct TopkWs {
  uint32_t* items;    // work-item counter of the scoring pass
  float* logits;      // [rows][ldw]
  int64_t ldw;
  size_t zero_bytes;  // the counter
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) / 256 * 256; }

__host__ __device__ inline TopkWs ws_layout(void* base, int64_t rows, int32_t max_blocks,
                                            size_t* total) {
  const int64_t ldw = (int64_t)max_blocks * kPage;
  const size_t c = 256;
  const size_t e = ws_align((size_t)rows * ldw * 4);
  uint8_t* p = static_cast<uint8_t*>(base);
  TopkWs w;
  w.items = reinterpret_cast<uint32_t*>(p);
  w.logits = reinterpret_cast<float*>(p + c);
  w.ldw = ldw;
  w.zero_bytes = 4;
  if (total) *total = c + e;
  return w;
}

__global__ void __launch_bounds__(kRowThreads, 1) paged_select_kernel(const PagedArgs p,
                                                                       int next_n) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  const int64_t rows = (int64_t)p.B * next_n;
  const TopkWs ws = ws_layout(p.workspace, rows, p.max_blocks, nullptr);
  const int64_t r = blockIdx.x;
  const int b = (int)(r / next_n), j = (int)(r % next_n);
  int64_t L = __ldg(p.context_lens + b);
  const int64_t cap = (int64_t)p.max_blocks * kPage;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int64_t len = L - next_n + j + 1;
  row_topk(sm, ws.logits + r * ws.ldw, len < 0 ? 0 : len, p.topk, p.out_idx + r * p.topk);
}

}  // namespace

size_t paged_topk_workspace_bytes(int32_t B, int32_t next_n, int32_t max_blocks, int32_t k,
                                  int32_t* tiles_per_cta_out, int32_t* chunks_out) {
  (void)k;
  if (B <= 0 || (next_n != 1 && next_n != 2) || max_blocks <= 0) return 0;
  if (tiles_per_cta_out) *tiles_per_cta_out = kFusedTilesPerItem;
  if (chunks_out)
    *chunks_out = (int32_t)(((int64_t)max_blocks * kPage + kFusedTilesPerItem * kTileKeys - 1) /
                            (kFusedTilesPerItem * kTileKeys));
  size_t total = 0;
  ws_layout(nullptr, (int64_t)B * next_n, max_blocks, &total);
  return total;
}

cudaError_t launch_paged_logits_topk(int H, int next_n, const PagedArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.B * next_n;
  const TopkWs ws = ws_layout(a.workspace, rows, a.max_blocks, nullptr);
  cudaError_t e = cudaMemsetAsync(a.workspace, 0, ws.zero_bytes, stream);
  if (e != cudaSuccess) return e;
  // scoring pass: the logits kernel writing into the workspace, work items
  // handed out by the counter
  PagedArgs s = a;
  s.logits = ws.logits;
  s.ld = ws.ldw;
  s.clean = 0;
  s.item_counter = ws.items;
  e = launch_paged_logits(H, next_n, s, stream);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(SelSmem);
  e = cudaFuncSetAttribute(paged_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  paged_select_kernel<<<(unsigned)rows, kRowThreads, smem, stream>>>(a, next_n);
  return cudaGetLastError();
}

}  // namespace idx
