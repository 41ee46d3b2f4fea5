// idx_paged_logits_topk_noalloc: the fused decode logits + top-k entry for
// callers that cannot allocate device memory.  The scratch the fused path
// needs lives in a fixed-size array in this library's device memory, so the
// caller passes only inputs and outputs.
//
// Who needs it: code that runs where a device allocation is not allowed or not
// available -- for example an engine loop whose allocator is frozen after
// start-up, a plugin host that hands kernels raw buffers but no allocator, or
// a latency-critical step that must not pay for cudaMalloc (which can block on
// the device).
//
// Costs and rules:
//   - the array below is reserved on every GPU that loads this part of the
//     library and stays reserved until the process exits;
//   - its device address is looked up on the first call on each device (with
//     that device current); make that first call before any stream capture;
//   - all calls share the one array, so calls that overlap on the GPU (on
//     different streams without ordering) race and give wrong results;
//   - the parts of the scratch that must start at zero are cleared by every
//     call; the rest keeps the previous call's contents.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "idx.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

thread_local char g_msg[256] = "";

}  // namespace

extern "C" IDX_API idx_status idx_paged_logits_topk_noalloc(
    const uint8_t* q_vals, const uint8_t* q_scales, int32_t B, int32_t next_n, int32_t H,
    const uint8_t* kcache, int64_t num_blocks, int32_t page_size, const int32_t* block_table,
    int32_t max_blocks, const int32_t* context_lens, const float* weights, int32_t k,
    int32_t* out_idx, idx_device_errors* errors, idx_stream_t stream) {
  const size_t need =
      idx_paged_logits_topk_workspace_bytes(B, next_n, max_blocks, page_size, k);
  if (need > kNoAllocScratchBytes) {
    snprintf(g_msg, sizeof g_msg,
             "this batch needs %zu bytes of scratch; the built-in scratch holds %zu "
             "(use idx_paged_logits_topk with a caller workspace)",
             need, kNoAllocScratchBytes);
    fprintf(stderr, "idx_paged_logits_topk_noalloc: %s\n", g_msg);
    return IDX_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return IDX_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        fprintf(stderr, "idx_paged_logits_topk_noalloc: cudaGetSymbolAddress: %s\n",
                cudaGetErrorString(e));
        return IDX_ERR_CUDA;
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return idx_paged_logits_topk(q_vals, q_scales, B, next_n, H, kcache, num_blocks, page_size,
                               block_table, max_blocks, context_lens, weights, k, out_idx,
                               scratch, kNoAllocScratchBytes, errors, stream);
}
