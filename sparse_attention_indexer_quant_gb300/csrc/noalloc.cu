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
//   - its device address is looked up on the first call in each CUDA context
//     (the current one of the calling thread) and kept for later calls in
//     that context;
//   - all calls share the one array, so calls that overlap on the GPU (on
//     different streams without ordering) race and give wrong results;
//   - nothing has to be cleared between calls: the work-item counter at the
//     start of the scratch carries each call's generation and the select pass
//     resets it at the end of every call; the logits rows behind it are
//     rewritten by every call before they are read.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "idx.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The scratch address per CUDA context: a module global has one address per
// context, so a context made after a device reset (or a second context on the
// same device) gets its own lookup.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

constexpr int kMaxContexts = 64;
std::mutex g_mu;
CUcontext g_ctx[kMaxContexts] = {};
void* g_scratch_addr[kMaxContexts] = {};
int g_n_ctx = 0;

}  // namespace

extern "C" IDX_API idx_status idx_paged_logits_topk_noalloc(
    const uint8_t* q_vals, const uint8_t* q_scales, int32_t B, int32_t next_n, int32_t H,
    const uint8_t* kcache, int64_t num_blocks, int32_t page_size, const int32_t* block_table,
    int32_t max_blocks, const int32_t* context_lens, const float* weights, int32_t k,
    int32_t* out_idx, idx_device_errors* errors, idx_stream_t stream) {
  const size_t need =
      idx_paged_logits_topk_workspace_bytes(B, next_n, max_blocks, page_size, k);
  if (need > kNoAllocScratchBytes)
    return idx::fail(IDX_ERR_INVALID_ARG,
                     "this batch needs %zu bytes of scratch; the built-in scratch holds %zu "
                     "(use idx_paged_logits_topk with a caller workspace)",
                     need, kNoAllocScratchBytes);
  // the device gate first: on any other device the library has no image, so
  // the symbol lookup below could not succeed
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
    return idx::fail(IDX_ERR_CUDA, "no current CUDA context");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_n_ctx; ++i)
      if (g_ctx[i] == ctx) scratch = g_scratch_addr[i];
    if (scratch == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();  // leave no pending error behind
        return idx::fail(IDX_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch: %s",
                         cudaGetErrorString(e));
      }
      if (g_n_ctx == kMaxContexts)
        return idx::fail(IDX_ERR_CUDA, "more than %d CUDA contexts", kMaxContexts);
      g_ctx[g_n_ctx] = ctx;
      g_scratch_addr[g_n_ctx] = p;
      ++g_n_ctx;
      scratch = p;
    }
  }
  return idx_paged_logits_topk(q_vals, q_scales, B, next_n, H, kcache, num_blocks, page_size,
                               block_table, max_blocks, context_lens, weights, k, out_idx,
                               scratch, kNoAllocScratchBytes, errors, stream);
}
