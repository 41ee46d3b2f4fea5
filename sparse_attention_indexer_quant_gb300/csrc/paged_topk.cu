// Paged decode logits + top-k (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// paged_mqa_logits followed by top_k_per_row into topk_indices_buffer), in two
// launches that hand the logits over through the caller's workspace instead of
// a logits tensor:
//
//   1. score    the persistent cp.async + tcgen05 logits kernel, taking work items
//               from a counter in the workspace, writing each row's valid
//               logits to a row-major scratch that stays in L2 for these sizes
//               and counting each logit into its row's coarse histogram (the
//               top 12 bits of its order-preserving key);
//   2. select   one 1024-thread CTA per row: the row's histogram gives the bin
//               holding the k-th largest logit and the count above it; one pass
//               over the row's logits sends everything above that bin to the
//               output and the bin's own elements to a shared-memory candidate
//               list; two 10-bit radix digits over the candidates finish the
//               exact selection.
// All three launches (zeroing, score, select) are dependent launches, so each
// one's start overlaps the previous one's tail.
//
// Workspace (device, caller-owned): a u32 work-item counter and the u32
// histograms [rows][4096] (both zeroed by a small kernel per call), then f32
// logits[rows][ldw], ldw = max_blocks * 64.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"
#include "topk_select.cuh"

namespace idx {
namespace {

constexpr int kFusedTilesPerItem = 8;
constexpr int kSelThreads = 1024;
constexpr int kSelCandCap = 8192;  // boundary-bin elements kept in shared memory
constexpr int kSelVec = 4;         // float4 loads in flight per thread in the row pass
static_assert(kCoarseBins == 4 * kSelThreads, "each select thread owns four histogram bins");

struct TopkWs {
  uint32_t* items;    // work-item counter of the scoring pass
  uint32_t* hist;     // [rows][kCoarseBins]
  float* logits;      // [rows][ldw]
  int64_t ldw;
  size_t zero_bytes;  // counter + histograms
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) / 256 * 256; }

__host__ __device__ inline TopkWs ws_layout(void* base, int64_t rows, int32_t max_blocks,
                                            size_t* total) {
  const int64_t ldw = (int64_t)max_blocks * kPage;
  const size_t c = 256;
  const size_t h = (size_t)rows * kCoarseBins * 4;
  const size_t e = ws_align((size_t)rows * ldw * 4);
  uint8_t* p = static_cast<uint8_t*>(base);
  TopkWs w;
  w.items = reinterpret_cast<uint32_t*>(p);
  w.hist = reinterpret_cast<uint32_t*>(p + c);
  w.logits = reinterpret_cast<float*>(p + c + h);
  w.ldw = ldw;
  w.zero_bytes = c + h;
  if (total) *total = c + h + e;
  return w;
}

struct SelSmem {
  uint32_t hist[kRadixBins];  // radix-digit scratch
  ScanScratch s;
  uint32_t n_out;             // elements above the boundary bin placed so far
  uint32_t n_cand;            // boundary-bin elements seen so far
  uint32_t slot;              // next output slot of the exact pass
  uint32_t cand_keys[kSelCandCap];
  int32_t cand_idx[kSelCandCap];
};

__global__ void __launch_bounds__(kSelThreads, 1) paged_select_kernel(const PagedArgs p,
                                                                       int next_n) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  pdl_wait();  // the scoring pass's logits and histograms
  const int64_t rows = (int64_t)p.B * next_n;
  const TopkWs ws = ws_layout(p.workspace, rows, p.max_blocks, nullptr);
  const int64_t r = blockIdx.x;
  const int b = (int)(r / next_n), j = (int)(r % next_n);
  int64_t L = __ldg(p.context_lens + b);
  const int64_t cap = (int64_t)p.max_blocks * kPage;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  int64_t len = L - next_n + j + 1;
  len = len < 0 ? 0 : len;
  const uint32_t k = (uint32_t)p.topk;
  int32_t* out = p.out_idx + r * p.topk;
  const int t = threadIdx.x;
  if (len <= (int64_t)k) {
    for (int i = t; i < (int)k; i += kSelThreads) out[i] = i < len ? i : -1;
    return;
  }

  // ---- 1. boundary bin from the row's histogram; thread t owns bins
  //         4095-4t down to 4092-4t, so thread order is descending bin order
  const uint4 h4 = __ldcg(reinterpret_cast<const uint4*>(ws.hist + r * kCoarseBins) +
                          (kSelThreads - 1 - t));
  if (t == 0) {
    sm.s.bin = 0;
    sm.s.above = 0;
    sm.n_out = 0;
    sm.n_cand = 0;
  }
  const uint32_t local = h4.x + h4.y + h4.z + h4.w;
  const uint32_t excl = block_exclusive_scan(local, sm.s);
  if (excl < k && k <= excl + local) {
    const uint32_t hb[4] = {h4.w, h4.z, h4.y, h4.x};
    uint32_t run = excl;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (run < k && k <= run + hb[q]) {
        sm.s.bin = (uint32_t)(kCoarseBins - 1 - 4 * t - q);
        sm.s.above = run;
      }
      run += hb[q];
    }
  }
  __syncthreads();
  const uint32_t b1 = sm.s.bin;
  const uint32_t above = sm.s.above;

  // ---- 2. one pass over the row: above b1 -> out, b1 -> candidates.  Per
  //         chunk of 16K elements each thread holds its 16 keys in registers,
  //         counts them, and one block scan of the packed counts gives every
  //         thread its own output and candidate ranges (no atomics).
  const float* x = ws.logits + r * ws.ldw;  // 256-byte aligned
  constexpr int64_t kPass = (int64_t)kSelThreads * 4 * kSelVec;
  for (int64_t base = 0; base < len; base += kPass) {
    uint4 kv[kSelVec];
#pragma unroll
    for (int u = 0; u < kSelVec; ++u) {
      const int64_t i0 = base + 4 * ((int64_t)u * kSelThreads + t);
      float4 v;
      if (i0 + 3 < len) {
        v = __ldcg(reinterpret_cast<const float4*>(x + i0));
      } else {
        v.x = i0 + 0 < len ? __ldcg(x + i0 + 0) : -INFINITY;
        v.y = i0 + 1 < len ? __ldcg(x + i0 + 1) : -INFINITY;
        v.z = i0 + 2 < len ? __ldcg(x + i0 + 2) : -INFINITY;
        v.w = i0 + 3 < len ? __ldcg(x + i0 + 3) : -INFINITY;
      }
      kv[u] = make_uint4(float_key(v.x), float_key(v.y), float_key(v.z), float_key(v.w));
    }
    // positions past len hold key(-inf), whose bin (0x007) lies below any bin
    // that can hold the k-th largest of at least k + 1 finite logits
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int u = 0; u < kSelVec; ++u) {
      const uint32_t e4[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t bin = coarse_bin(e4[q]);
        n_gt += bin > b1 ? 1u : 0u;
        n_eq += bin == b1 ? 1u : 0u;
      }
    }
    // block sums fit 16 bits: fewer than k <= 2048 elements lie above b1 and a
    // chunk holds 16384 elements
    const uint32_t ex = block_exclusive_scan((n_gt << 16) | n_eq, sm.s);
    uint32_t o = sm.n_out + (ex >> 16);
    uint32_t c = sm.n_cand + (ex & 0xFFFFu);
#pragma unroll
    for (int u = 0; u < kSelVec; ++u) {
      const int64_t i0 = base + 4 * ((int64_t)u * kSelThreads + t);
      const uint32_t e4[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t bin = coarse_bin(e4[q]);
        if (bin > b1) {
          if (o < above) out[o] = (int32_t)(i0 + q);
          ++o;
        } else if (bin == b1) {
          if (c < (uint32_t)kSelCandCap) {
            sm.cand_keys[c] = e4[q];
            sm.cand_idx[c] = (int32_t)(i0 + q);
          }
          ++c;
        }
      }
    }
    __syncthreads();
    if (t == kSelThreads - 1) {  // the last thread's ends are the running totals
      sm.n_out = o;
      sm.n_cand = c;
    }
    __syncthreads();
  }
  if (t == 0) sm.slot = above;
  __syncthreads();

  // ---- 3. the exact remainder inside b1
  const uint32_t nb1 = sm.n_cand;
  const uint32_t need = k - above;
  auto emit = [&](uint32_t, int32_t i) {
    const uint32_t s = warp_claim(&sm.slot, true);
    if (s < k) out[s] = i;
  };
  if (nb1 <= (uint32_t)kSelCandCap) {
    const SmemPairs cand{sm.cand_keys, sm.cand_idx, (int)nb1};
    radix_select(sm.hist, sm.s, cand, need, b1 << kCoarseShift, 32 - kCoarseShift, emit);
  } else {
    const GlobalLogits<true> row{x, 0, len};
    radix_select(sm.hist, sm.s, row, need, b1 << kCoarseShift, 32 - kCoarseShift, emit);
  }
}

// Zeroes the work-item counter and the row histograms (n16 16-byte words).
__global__ void __launch_bounds__(256) paged_ws_zero_kernel(uint4* w, int64_t n16) {
  pdl_launch_dependents();
  pdl_wait();  // the previous call's select may still be reading them
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    w[i] = make_uint4(0u, 0u, 0u, 0u);
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
  const int64_t n16 = (int64_t)(ws.zero_bytes / 16);
  const unsigned zgrid = (unsigned)((n16 + 256 * 8 - 1) / (256 * 8));
  cudaError_t e = launch_dependent(paged_ws_zero_kernel, dim3(zgrid), dim3(256), 0, stream,
                                   reinterpret_cast<uint4*>(a.workspace), n16);
  if (e != cudaSuccess) return e;
  // scoring pass: the logits kernel writing into the workspace and counting
  // the row histograms, work items handed out by the counter
  PagedArgs s = a;
  s.logits = ws.logits;
  s.ld = ws.ldw;
  s.clean = 0;
  s.item_counter = ws.items;
  s.row_hist = ws.hist;
  e = launch_paged_logits(H, next_n, s, stream);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(SelSmem);
  e = cudaFuncSetAttribute(paged_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(paged_select_kernel, dim3((unsigned)rows), dim3(kSelThreads), smem,
                          stream, a, next_n);
}

}  // namespace idx
