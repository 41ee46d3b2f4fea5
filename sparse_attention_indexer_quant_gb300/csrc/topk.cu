// Top-k per logits row (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// top_k_per_row into topk_indices_buffer; rows shorter than k are padded with
// -1): one CTA per row running row_topk over the row's window.
#include "common.cuh"
#include "launch.h"
#include "topk_row.cuh"

namespace idx {
namespace {

constexpr int kRowsChunk = 8192;
using RowsSmem = RowTopkSmem<kRowsChunk>;

__global__ void __launch_bounds__(kRowThreads) topk_rows_kernel(const float* __restrict__ logits,
                                                                    int64_t ld,
                                                                    const int32_t* row_start,
                                                                    const int32_t* row_end,
                                                                    int32_t k, int32_t* out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RowsSmem& sm = *reinterpret_cast<RowsSmem*>(smem_raw);
  const int64_t row = blockIdx.x;
  const int64_t st = row_start != nullptr ? __ldg(row_start + row) : 0;
  const int64_t en = __ldg(row_end + row);
  // positions are reported relative to the window start
  row_topk(sm, logits + row * ld + st, en > st ? en - st : 0, k, out + row * k);
}

}  // namespace

cudaError_t launch_topk_rows(const float* logits, int64_t rows, int64_t ld,
                             const int32_t* row_start, const int32_t* row_end, int32_t k,
                             int32_t* out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const size_t smem = sizeof(RowsSmem);
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<(unsigned)rows, kRowThreads, smem, stream>>>(logits, ld, row_start, row_end,
                                                                   k, out);
  return cudaGetLastError();
}

}  // namespace idx
