// Paged decode logits + top-k (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// paged_mqa_logits followed by top_k_per_row into topk_indices_buffer), in
// launches that hand the logits over through the caller's workspace instead of
// a logits tensor:
//
//   1. score    the persistent cp.async + tcgen05 logits kernel, taking work items
//               from a generation-tagged counter and writing each row's valid
//               logits to a row-major scratch that stays in L2 for these sizes;
//   2. select   one thread-block cluster of P CTAs per row running
//               cluster_select_row (select_row.cuh) over the row's logits;
//               where one CTA per row is all that fits in one wave (more
//               rows than half the SMs), two-CTA clusters in two waves
//               instead, each cluster taking the sequences in order of
//               decreasing length, so that the longest rows (the slowest
//               selects) are in the first wave.
// Both are dependent launches.  The scoring pass lets the select launch start
// only once every earlier kernel is done, so the select reads the call's
// inputs before waiting for the logits.
//
// Workspace (device, caller-owned), 256-byte aligned pieces: the u64 work-item
// counter (tagged with the call's generation, see claim_item; the select
// clears it at the end of every call, which keeps replays of a captured call
// correct), then f32 logits [rows][ldw], ldw = max_blocks * 64.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"
#include "select_row.cuh"

namespace idx {
namespace {

struct TopkWs {
  unsigned long long* items;  // work-item counter of the scoring pass, then the
                              // decode step's preparation-chunk counter
  float* logits;              // [rows][ldw]
  int64_t ldw;
  uint8_t* q_vals;            // decode step: quantised query heads [rows * H][64]
  uint8_t* q_scales;          //              and their scales [rows * H][4]
  unsigned long long* seq_state;  // decode step: per-sequence preparation state [B]
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) / 256 * 256; }

// H = 0: the fused call's workspace; H > 0: the decode step's, which also
// holds the step's quantised query heads and one state word per sequence
// after the logits (rows = B * next_n).
__host__ __device__ inline TopkWs ws_layout(void* base, int64_t rows, int32_t max_blocks,
                                            size_t* total, int32_t H = 0, int32_t B = 0) {
  const int64_t ldw = (int64_t)max_blocks * kPage;
  const size_t o_lg = 256;
  const size_t o_qv = o_lg + ws_align((size_t)rows * ldw * 4);
  const size_t o_qs = o_qv + ws_align((size_t)rows * H * kValBytes);
  const size_t o_st = o_qs + ws_align((size_t)rows * H * kScaleBytes);
  uint8_t* p = static_cast<uint8_t*>(base);
  TopkWs w;
  w.items = reinterpret_cast<unsigned long long*>(p);
  w.logits = reinterpret_cast<float*>(p + o_lg);
  w.ldw = ldw;
  w.q_vals = H > 0 ? p + o_qv : nullptr;
  w.q_scales = H > 0 ? p + o_qs : nullptr;
  w.seq_state = H > 0 ? reinterpret_cast<unsigned long long*>(p + o_st) : nullptr;
  if (total) *total = H > 0 ? o_st + ws_align((size_t)B * 8) : o_qv;
  return w;
}

// One cluster of `parts` CTAs per query row (b, j) of the decode batch; with
// `by_length` cluster c takes query j = c % next_n of the (c / next_n)-th
// longest sequence (equal lengths: lower index first; needs B <= kCoarseBins).
__global__ void __launch_bounds__(kSelThreads, 1) paged_select_kernel(const PagedArgs p, int next_n,
                                                                      int parts, int by_length) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  const int64_t rows = (int64_t)p.B * next_n;
  const TopkWs ws = ws_layout(p.workspace, rows, p.max_blocks, nullptr);
  int64_t r = blockIdx.x / parts;
  int b = (int)(r / next_n);
  const int j = (int)(r % next_n);
  if (by_length) {
    // the context lengths (clamped to the block table) in the histogram's
    // space, which the select clears only after this; each thread ranks its
    // sequences against all others, and the one of rank b is the cluster's
    const int64_t cap = (int64_t)p.max_blocks * kPage;
    int32_t* lens = reinterpret_cast<int32_t*>(sm.bins);
    __shared__ int picked;
    for (int i = threadIdx.x; i < p.B; i += kSelThreads) {
      const int64_t v = __ldg(p.context_lens + i);
      lens[i] = (int32_t)(v < 0 ? 0 : (v > cap ? cap : v));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < p.B; i += kSelThreads) {
      const int32_t li = lens[i];
      int rank = 0;
      for (int q = 0; q < p.B; ++q) rank += (lens[q] > li || (lens[q] == li && q < i)) ? 1 : 0;
      if (rank == b) picked = i;  // ranks are distinct: exactly one thread writes
    }
    __syncthreads();
    b = picked;
    r = (int64_t)b * next_n + j;
  }
  // an input of the call, read before the wait: this launch can only have
  // started after the scoring pass's wait, i.e. after every kernel issued
  // before the call completed
  int64_t L = __ldg(p.context_lens + b);
  const int64_t cap = (int64_t)p.max_blocks * kPage;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  int64_t len = L - next_n + j + 1;
  len = len < 0 ? 0 : len;
  pdl_wait();  // the scoring pass's logits
  // the work-item counter (and the decode step's chunk counter and counts)
  // are done with: reset them to this call's generation with no claims, so
  // that a replay of this call (a CUDA graph, same generation) starts from
  // zero without installing its generation first (a call with another
  // generation still finds them stale and installs its own)
  if (blockIdx.x == 0) {
    const unsigned long long fresh = p.item_gen << kItemBits;
    if (threadIdx.x < 2) ws.items[threadIdx.x] = fresh;  // scoring items, step chunks
    if (p.seq_state != nullptr)
      for (int i = threadIdx.x; i < p.B; i += kSelThreads) p.seq_state[i] = fresh;
  }
  // the workspace rows are 256-byte aligned
  cluster_select_row(sm, ws.logits + r * ws.ldw, len, (uint32_t)p.topk, p.out_idx + r * p.topk,
                     parts);
}

}  // namespace

size_t paged_topk_workspace_bytes(int32_t B, int32_t next_n, int32_t max_blocks, int32_t k) {
  (void)k;
  if (B <= 0 || (next_n != 1 && next_n != 2) || max_blocks <= 0) return 0;
  size_t total = 0;
  ws_layout(nullptr, (int64_t)B * next_n, max_blocks, &total);
  return total;
}

int32_t paged_topk_item_tiles(int32_t B, int32_t max_blocks, int64_t ctas) {
  // about eight work items per CTA when every sequence fills its block table
  // (small items even out the CTAs' finishing times; each item costs the
  // loader a round of dependent loads, so large batches take larger ones)
  const int64_t tiles = (int64_t)B * (((int64_t)max_blocks * kPage + kTileKeys - 1) / kTileKeys);
  const int64_t per = tiles / ((ctas > 0 ? ctas : 1) * 8);
  return per < 6 ? 4 : (per < 12 ? 8 : 16);
}

size_t paged_step_workspace_bytes(int32_t B, int32_t next_n, int32_t H, int32_t max_blocks,
                                  int32_t k) {
  (void)k;
  if (B <= 0 || (next_n != 1 && next_n != 2) || max_blocks <= 0 || H <= 0) return 0;
  size_t total = 0;
  ws_layout(nullptr, (int64_t)B * next_n, max_blocks, &total, H, B);
  return total;
}

cudaError_t launch_paged_decode_step(int H, int next_n, const PagedArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.B * next_n;
  const TopkWs ws = ws_layout(a.workspace, rows, a.max_blocks, nullptr, H, a.B);
  PagedArgs s = a;
  s.q_vals = ws.q_vals;
  s.q_scales = ws.q_scales;
  s.q_vals_w = ws.q_vals;
  s.q_scales_w = ws.q_scales;
  s.seq_state = ws.seq_state;
  s.prep_counter = ws.items + 1;
  return launch_paged_logits_topk(H, next_n, s, stream);
}

cudaError_t launch_paged_logits_topk(int H, int next_n, const PagedArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.B * next_n;
  const TopkWs ws = ws_layout(a.workspace, rows, a.max_blocks, nullptr);
  const size_t smem = sizeof(SelSmem);
  // the two kernels share one shared-memory carveout, so no SM has to be
  // reconfigured between them
  cudaError_t e = cudaFuncSetAttribute(paged_select_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(paged_select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // scoring pass: the logits kernel writing into the workspace, work items
  // handed out by the counter
  PagedArgs s = a;
  s.logits = ws.logits;
  s.ld = ws.ldw;
  s.clean = 0;
  s.item_counter = ws.items;
  s.wait_first = 1;
  e = launch_paged_logits(H, next_n, s, stream);
  if (e != cudaSuccess) return e;
  const int sms = a.sms > 0 ? a.sms : 1;
  int parts = select_parts(paged_select_kernel, 0, rows, ws.ldw, sms, smem);
  // one CTA per row fits one wave but two do not: two-CTA clusters in two
  // waves, longest rows first (128 rows of 1K - 128K keys: 123 us for the
  // call against 130 with one CTA per row, whose longest selects took ~30 us)
  int by_length = 0;
  if (parts == 1 && rows <= (int64_t)sms && ws.ldw / 2 >= kMinSlice && a.B <= kCoarseBins) {
    parts = 2;
    by_length = 1;
  }
  return launch_dependent_cluster(paged_select_kernel, dim3((unsigned)(rows * parts)),
                                  dim3(kSelThreads), smem, stream, (unsigned)parts, a, next_n,
                                  parts, by_length);
}

}  // namespace idx
