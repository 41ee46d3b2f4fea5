// Paged decode logits + top-k (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// paged_mqa_logits followed by top_k_per_row into topk_indices_buffer), in two
// launches that hand the logits over through the caller's workspace instead of
// a logits tensor:
//
//   1. score    the persistent TMA + tcgen05 main loop (work items taken from
//               a counter in the workspace); the epilogue stores each valid
//               logit to the workspace (a row-major scratch that stays in L2 for
//               these sizes) and adds it to a shared-memory coarse histogram
//               (top 12 key bits) of its row, folded into the row's global
//               histogram at the end of each item.
//   2. select   grid (segment of 8192 keys, row).  Every CTA finds from the
//               row histogram the bin that holds the row's k-th largest logit,
//               writes the positions of its segment's logits above that bin
//               straight to out_idx, and appends the boundary bin's logits to a
//               per-row list.  The last CTA of the row (ticket) picks the exact
//               remainder from that list.
//
// Workspace (device, caller-owned, 256-byte aligned pieces):
//   u32 hist[rows][4096], u32 ctr[rows][4], u32 item counter (zeroed by a
//   memset per call)
//   f32 logits[rows][ldw], u32 bkeys[rows][ldw], i32 bpos[rows][ldw]
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"
#include "topk_select.cuh"

namespace idx {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSegKeys = 8192;
constexpr int kSelCap = 4096;
constexpr int kPerThread = kSegKeys / kSelThreads;  // 32

struct TopkWs {
  uint32_t* hist;     // [rows][kCoarseBins]
  uint32_t* ctr;      // [rows][4]: slot, boundary count, ticket, unused
  uint32_t* items;    // work-item counter of the scoring pass
  float* logits;      // [rows][ldw]
  uint32_t* bkeys;    // [rows][ldw]
  int32_t* bpos;      // [rows][ldw]
  int64_t ldw;
  size_t zero_bytes;  // hist + ctr
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) / 256 * 256; }

__host__ __device__ inline TopkWs ws_layout(void* base, int64_t rows, int32_t max_blocks,
                                            size_t* total) {
  const int64_t ldw = (int64_t)max_blocks * kPage;
  const size_t h = ws_align((size_t)rows * kCoarseBins * 4);
  const size_t c = ws_align((size_t)rows * 16 + 4);
  const size_t e = ws_align((size_t)rows * ldw * 4);
  uint8_t* p = static_cast<uint8_t*>(base);
  TopkWs w;
  w.hist = reinterpret_cast<uint32_t*>(p);
  w.ctr = reinterpret_cast<uint32_t*>(p + h);
  w.items = reinterpret_cast<uint32_t*>(p + h) + rows * 4;
  w.logits = reinterpret_cast<float*>(p + h + c);
  w.bkeys = reinterpret_cast<uint32_t*>(p + h + c + e);
  w.bpos = reinterpret_cast<int32_t*>(p + h + c + 2 * e);
  w.ldw = ldw;
  w.zero_bytes = h + c;
  if (total) *total = h + c + 3 * e;
  return w;
}

template <int H, int NEXT_N>
struct ScoreEpilogue {
  static constexpr int NH = H * NEXT_N;
  static constexpr size_t kExtraSmem = (size_t)NEXT_N * kCoarseBins * 4;

  __device__ __forceinline__ static void init(uint8_t* extra) {
    uint32_t* h = reinterpret_cast<uint32_t*>(extra);
    for (int i = threadIdx.x; i < NEXT_N * kCoarseBins; i += blockDim.x) h[i] = 0;
  }

  __device__ __forceinline__ static void tile(const PagedArgs& p, const ItemDesc& it,
                                              const float* w_smem, uint8_t* extra, int64_t key,
                                              const float (&d)[NH]) {
    uint32_t* hist = reinterpret_cast<uint32_t*>(extra);
    const TopkWs ws = ws_layout(p.workspace, (int64_t)p.B * NEXT_N, p.max_blocks, nullptr);
    float logit[NEXT_N];
    weighted_relu_sum<H, NEXT_N>(w_smem, d, logit);
#pragma unroll
    for (int j = 0; j < NEXT_N; ++j) {
      const int64_t len = it.L - NEXT_N + j + 1;
      const bool valid = key < len;
      const int64_t r = (int64_t)it.b * NEXT_N + j;
      if (valid) ws.logits[r * ws.ldw + key] = logit[j];
      hist_add(hist + j * kCoarseBins, coarse_bin(float_key(logit[j])), valid);
    }
  }

  // Folds the item's histograms into its rows' global histograms and clears
  // them for the next item (the four epilogue warps, after their last tile).
  __device__ __forceinline__ static void item_done(const PagedArgs& p, const ItemDesc& it,
                                                   uint8_t* extra) {
    uint32_t* hist = reinterpret_cast<uint32_t*>(extra);
    const TopkWs ws = ws_layout(p.workspace, (int64_t)p.B * NEXT_N, p.max_blocks, nullptr);
    const int e = threadIdx.x - 2 * 32;  // epilogue threads are warps 2-5
    for (int j = 0; j < NEXT_N; ++j) {
      uint32_t* g = ws.hist + ((int64_t)it.b * NEXT_N + j) * kCoarseBins;
      for (int i = e; i < kCoarseBins; i += kEpiThreads) {
        const uint32_t v = hist[j * kCoarseBins + i];
        if (v) {
          atomicAdd(g + i, v);
          hist[j * kCoarseBins + i] = 0;
        }
      }
    }
    epilogue_sync();
  }
};

template <int H, int NEXT_N>
__global__ void __launch_bounds__(kPagedThreads, paged_ctas_per_sm(H * NEXT_N))
    paged_score_kernel(const __grid_constant__ CUtensorMap tm_vals,
                       const __grid_constant__ CUtensorMap tm_scales, const PagedArgs p) {
  const TopkWs ws = ws_layout(p.workspace, (int64_t)p.B * NEXT_N, p.max_blocks, nullptr);
  paged_persistent_run<H, NEXT_N, ScoreEpilogue<H, NEXT_N>>(&tm_vals, &tm_scales, p, true, false,
                                                            ws.items);
}

struct SelectSmem {
  SelectScratch sel;
  uint32_t cand_keys[kSelCap];
  int32_t cand_idx[kSelCap];
  uint32_t ticket;
  uint32_t slot;
  uint32_t slot_fill;
  uint32_t base_above;
  uint32_t base_bnd;
};

__global__ void __launch_bounds__(kSelThreads) paged_select_kernel(const PagedArgs p,
                                                                    int next_n) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectSmem& sm = *reinterpret_cast<SelectSmem*>(smem_raw);
  const int64_t rows = (int64_t)p.B * next_n;
  const TopkWs ws = ws_layout(p.workspace, rows, p.max_blocks, nullptr);
  const int64_t r = blockIdx.y;
  const int b = (int)(r / next_n), j = (int)(r % next_n);
  int64_t L = __ldg(p.context_lens + b);
  const int64_t cap = (int64_t)p.max_blocks * kPage;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  int64_t len = L - next_n + j + 1;
  len = len < 0 ? 0 : len;
  const uint32_t k = (uint32_t)p.topk;
  int32_t* orow = p.out_idx + r * p.topk;
  const int64_t lo = (int64_t)blockIdx.x * kSegKeys;
  const int64_t hi = lo + kSegKeys < len ? lo + kSegKeys : len;

  if (len <= (int64_t)k) {
    // every valid position is selected; the first segment also pads
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) orow[i] = (int32_t)i;
    if (blockIdx.x == 0)
      for (int64_t i = len + threadIdx.x; i < (int64_t)k; i += blockDim.x) orow[i] = -1;
    return;
  }
  uint32_t* ghist = ws.hist + r * kCoarseBins;
  uint32_t* ctr = ws.ctr + r * 4;
  copy_words_cg(sm.sel.hist, ghist, kCoarseBins);
  __syncthreads();
  find_threshold_bin(sm.sel.hist, kCoarseBins, k, sm.sel.s);
  const uint32_t b1 = sm.sel.s.bin;
  const uint32_t above = sm.sel.s.above;
  const uint32_t nb1 = sm.sel.hist[b1];
  const float* x = ws.logits + r * ws.ldw;
  uint32_t* bkeys = ws.bkeys + r * ws.ldw;
  int32_t* bpos = ws.bpos + r * ws.ldw;
  // this thread's logits of the segment, all loads in flight together
  float v[kPerThread];
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int64_t i = lo + (int64_t)u * kSelThreads + threadIdx.x;
    v[u] = i < hi ? __ldcg(x + i) : 0.f;
  }
  uint32_t n_above = 0, n_bnd = 0;
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int64_t i = lo + (int64_t)u * kSelThreads + threadIdx.x;
    const uint32_t bin = coarse_bin(float_key(v[u]));
    n_above += (i < hi && bin > b1) ? 1u : 0u;
    n_bnd += (i < hi && bin == b1) ? 1u : 0u;
  }
  // one block scan and one global claim per counter for the whole CTA
  const uint32_t packed = (n_above << 16) | n_bnd;
  const uint32_t excl = block_exclusive_scan(packed, sm.sel.s);
  if (threadIdx.x == blockDim.x - 1) {
    const uint32_t tot = excl + packed;
    sm.base_above = (tot >> 16) ? atomicAdd(ctr + 0, tot >> 16) : 0u;
    sm.base_bnd = (tot & 0xFFFFu) ? atomicAdd(ctr + 1, tot & 0xFFFFu) : 0u;
  }
  __syncthreads();
  uint32_t a_slot = sm.base_above + (excl >> 16);
  uint32_t b_slot = sm.base_bnd + (excl & 0xFFFFu);
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int64_t i = lo + (int64_t)u * kSelThreads + threadIdx.x;
    const uint32_t key = float_key(v[u]);
    const uint32_t bin = coarse_bin(key);
    if (i < hi && bin > b1) orow[a_slot++] = (int32_t)i;
    if (i < hi && bin == b1) {
      bkeys[b_slot] = key;
      bpos[b_slot] = (int32_t)i;
      ++b_slot;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sm.ticket = atomicAdd(ctr + 2, 1u);
  __syncthreads();
  if (sm.ticket != gridDim.x - 1) return;
  __threadfence();
  // last CTA of the row: the exact remainder from the boundary bin
  if (threadIdx.x == 0) {
    sm.slot = above;
    sm.slot_fill = 0;
  }
  __syncthreads();
  const uint32_t need = k - above;
  auto emit = [&](uint32_t, int32_t i) { orow[warp_claim(&sm.slot, true)] = i; };
  const GlobalPairs bset{bkeys, bpos, (int64_t)nb1};
  if (nb1 <= (uint32_t)kSelCap) {
    bset.for_each([&](uint32_t key, int32_t i) {
      const uint32_t c = atomicAdd(&sm.slot_fill, 1u);
      sm.cand_keys[c] = key;
      sm.cand_idx[c] = i;
    });
    __syncthreads();
    const SmemPairs cand{sm.cand_keys, sm.cand_idx, (int)nb1};
    radix_select(sm.sel.hist, sm.sel.s, cand, need, b1 << kCoarseShift, 32 - kCoarseShift,
                 emit);
  } else {
    __syncthreads();
    radix_select(sm.sel.hist, sm.sel.s, bset, need, b1 << kCoarseShift, 32 - kCoarseShift,
                 emit);
  }
}

template <int H, int NEXT_N>
cudaError_t launch_score(const CUtensorMap& tv, const CUtensorMap& ts, const PagedArgs& a,
                         cudaStream_t stream) {
  using Ep = ScoreEpilogue<H, NEXT_N>;
  const size_t smem = paged_smem_bytes<H * NEXT_N>() + Ep::kExtraSmem;
  auto kern = paged_score_kernel<H, NEXT_N>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)a.grid, kPagedThreads, smem, stream>>>(tv, ts, a);
  return cudaGetLastError();
}

}  // namespace

size_t paged_topk_workspace_bytes(int32_t B, int32_t next_n, int32_t max_blocks, int32_t k,
                                  int32_t* tiles_per_cta_out, int32_t* chunks_out) {
  (void)k;
  (void)tiles_per_cta_out;
  (void)chunks_out;
  if (B <= 0 || (next_n != 1 && next_n != 2) || max_blocks <= 0) return 0;
  size_t total = 0;
  ws_layout(nullptr, (int64_t)B * next_n, max_blocks, &total);
  return total;
}

cudaError_t launch_paged_logits_topk(const CUtensorMap& tv, const CUtensorMap& ts, int H,
                                     int next_n, const PagedArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.B * next_n;
  const TopkWs ws = ws_layout(a.workspace, rows, a.max_blocks, nullptr);
  cudaError_t e = cudaMemsetAsync(a.workspace, 0, ws.zero_bytes, stream);
  if (e != cudaSuccess) return e;
  if (H == 32 && next_n == 1) e = launch_score<32, 1>(tv, ts, a, stream);
  else if (H == 32 && next_n == 2) e = launch_score<32, 2>(tv, ts, a, stream);
  else if (H == 64 && next_n == 1) e = launch_score<64, 1>(tv, ts, a, stream);
  else if (H == 64 && next_n == 2) e = launch_score<64, 2>(tv, ts, a, stream);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(SelectSmem);
  e = cudaFuncSetAttribute(paged_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t segs = (ws.ldw + kSegKeys - 1) / kSegKeys;
  dim3 grid((unsigned)segs, (unsigned)rows);
  paged_select_kernel<<<grid, kSelThreads, smem, stream>>>(a, next_n);
  return cudaGetLastError();
}

}  // namespace idx
