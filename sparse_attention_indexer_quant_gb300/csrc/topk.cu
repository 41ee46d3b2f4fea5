// Top-k per logits row (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// top_k_per_row into topk_indices_buffer; rows shorter than k are padded with
// -1).  Two kernels, chosen by the number of rows:
//   - up to one row per SM: one thread-block cluster of P CTAs per row running
//     cluster_select_row (select_row.cuh), so that a few long rows use the
//     whole GPU;
//   - more rows: one 256-thread CTA per row running row_topk (topk_row.cuh),
//     four CTAs per SM, for throughput over many rows.
#include "common.cuh"
#include "launch.h"
#include "select_row.cuh"
#include "topk_row.cuh"

namespace idx {
namespace {

__global__ void __launch_bounds__(kSelThreads, 1)
    topk_rows_cluster_kernel(const float* __restrict__ logits, int64_t ld,
                             const int32_t* row_start, const int32_t* row_end, int32_t k,
                             int32_t* out, int parts) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  pdl_wait();  // the logits may come from the previous kernel
  const int64_t row = blockIdx.x / parts;
  const int64_t st = row_start != nullptr ? __ldg(row_start + row) : 0;
  const int64_t en = __ldg(row_end + row);
  // positions are reported relative to the window start
  cluster_select_row(sm, logits + row * ld + st, en > st ? en - st : 0, (uint32_t)k,
                     out + row * k, parts);
}

constexpr int kRowsChunk = 4096;
using RowsSmem = RowTopkSmem<kRowsChunk>;

__global__ void __launch_bounds__(kRowThreads, 4) topk_rows_kernel(const float* __restrict__ logits,
                                                                int64_t ld,
                                                                const int32_t* row_start,
                                                                const int32_t* row_end,
                                                                int32_t k, int32_t* out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RowsSmem& sm = *reinterpret_cast<RowsSmem*>(smem_raw);
  pdl_wait();  // the logits may come from the previous kernel
  const int64_t row = blockIdx.x;
  const int64_t st = row_start != nullptr ? __ldg(row_start + row) : 0;
  const int64_t en = __ldg(row_end + row);
  // positions are reported relative to the window start
  row_topk(sm, logits + row * ld + st, en > st ? en - st : 0, k, out + row * k);
}

// Top-k of a candidate list (prefill logits + top-k): row_topk over the list's
// values gives list positions, which are then replaced by the positions in
// the row's window that the list stores beside each value.
__global__ void __launch_bounds__(kRowThreads, 4) cand_topk_kernel(
    const float* __restrict__ cand_vals, const int32_t* __restrict__ cand_idx,
    const uint32_t* __restrict__ cand_cnt, int64_t cand_ld, int32_t k, int32_t* out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RowsSmem& sm = *reinterpret_cast<RowsSmem*>(smem_raw);
  pdl_wait();  // the lists come from the previous kernel
  const int64_t row = blockIdx.x;
  const int64_t n = __ldg(cand_cnt + row);
  int32_t* o = out + row * k;
  row_topk(sm, cand_vals + row * cand_ld, n, k, o);
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += kRowThreads) {
    const int32_t pos = o[i];
    if (pos >= 0) o[i] = __ldg(cand_idx + row * cand_ld + pos);
  }
}

}  // namespace

cudaError_t launch_cand_topk(const float* cand_vals, const int32_t* cand_idx,
                             const uint32_t* cand_cnt, int64_t cand_ld, int64_t rows, int32_t k,
                             int32_t* out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const size_t smem = sizeof(RowsSmem);
  cudaError_t e =
      cudaFuncSetAttribute(cand_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(cand_topk_kernel, dim3((unsigned)rows), dim3(kRowThreads), smem, stream,
                          cand_vals, cand_idx, cand_cnt, cand_ld, k, out);
}

cudaError_t launch_topk_rows(const float* logits, int64_t rows, int64_t ld,
                             const int32_t* row_start, const int32_t* row_end, int32_t k,
                             int32_t* out, int sms, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (sms <= 0) sms = 1;
  if (rows > sms) {
    const size_t smem = sizeof(RowsSmem);
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(topk_rows_kernel, dim3((unsigned)rows), dim3(kRowThreads), smem,
                            stream, logits, ld, row_start, row_end, k, out);
  }
  const size_t smem = sizeof(SelSmem);
  cudaError_t e = cudaFuncSetAttribute(topk_rows_cluster_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_rows_cluster_kernel,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const int parts = select_parts(topk_rows_cluster_kernel, 1, rows, ld, sms, smem);
  return launch_dependent_cluster(topk_rows_cluster_kernel, dim3((unsigned)(rows * parts)),
                                  dim3(kSelThreads), smem, stream, (unsigned)parts, logits, ld,
                                  row_start, row_end, k, out, parts);
}

}  // namespace idx
