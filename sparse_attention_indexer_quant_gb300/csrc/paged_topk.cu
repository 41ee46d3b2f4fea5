// Fused paged decode logits + top-k (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": paged_mqa_logits followed by
// top_k_per_row into topk_indices_buffer), without writing logits to memory.
//
// Each CTA scores a chunk of C = 8192 / next_n keys of one sequence with the
// shared TMA + tcgen05 main loop; its epilogue keeps the chunk's logits in
// shared memory.  At the end of the chunk the CTA emits, per query row, a
// superset of the chunk's k largest logits: every logit whose top 11 key bits
// are at or above those of the chunk's k-th largest (all of them when the chunk
// holds at most k).  Any member of the row's top k is in its chunk's top k, so
// the union of the supersets holds the row's top k.  The CTAs of a sequence
// then take a ticket; the last one selects the exact top k of each row from the
// candidates with the radix selection of top_k_per_row.
//
// Workspace (device, caller-owned):
//   u32 tickets[B] (zeroed before the launch)
//   u32 counts[rows][chunks]
//   u32 keys[rows][chunks][C], i32 idx[rows][chunks][C]
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"
#include "topk_select.cuh"

namespace idx {
namespace {

constexpr int kChunkFloats = 8192;  // per CTA: next_n rows x (8192 / next_n) keys

struct TopkWs {
  uint32_t* tickets;
  uint32_t* counts;
  uint32_t* keys;
  int32_t* idx;
  int64_t chunk_cap;  // C
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) / 256 * 256; }

__host__ __device__ inline TopkWs ws_layout(void* base, int32_t B, int32_t next_n,
                                            int32_t chunks, size_t* total) {
  const int64_t rows = (int64_t)B * next_n;
  const int64_t C = kChunkFloats / next_n;
  const size_t t_bytes = ws_align((size_t)B * 4);
  const size_t c_bytes = ws_align((size_t)rows * chunks * 4);
  const size_t e_bytes = ws_align((size_t)rows * chunks * C * 4);
  uint8_t* p = static_cast<uint8_t*>(base);
  TopkWs w;
  w.tickets = reinterpret_cast<uint32_t*>(p);
  w.counts = reinterpret_cast<uint32_t*>(p + t_bytes);
  w.keys = reinterpret_cast<uint32_t*>(p + t_bytes + c_bytes);
  w.idx = reinterpret_cast<int32_t*>(p + t_bytes + c_bytes + e_bytes);
  w.chunk_cap = C;
  if (total) *total = t_bytes + c_bytes + 2 * e_bytes;
  return w;
}

// Shared memory behind the main loop's buffers.
struct FusedExtra {
  float logits[kChunkFloats];    // [next_n][C]; reused as 4096 (key, idx) pairs by the merge
  SelectScratch sc;
  uint32_t ticket;
  uint32_t n_cand;
};

template <int H, int NEXT_N>
struct FusedEpilogue {
  static constexpr int NH = H * NEXT_N;
  static constexpr int C = kChunkFloats / NEXT_N;
  static constexpr size_t kExtraSmem = sizeof(FusedExtra);

  __device__ __forceinline__ static void tile(const PagedArgs&, const PagedCta& c,
                                              const float* w_smem, uint8_t* extra, int64_t key,
                                              const float (&d)[NH]) {
    FusedExtra& ex = *reinterpret_cast<FusedExtra*>(extra);
    float logit[NEXT_N];
    weighted_relu_sum<H, NEXT_N>(w_smem, d, logit);
    const int64_t off = key - c.k0;
    if (off < C) {
#pragma unroll
      for (int j = 0; j < NEXT_N; ++j) ex.logits[j * C + off] = logit[j];
    }
  }

  __device__ static void chunk_done(const PagedArgs& p, const PagedCta& c, uint8_t* extra,
                                    bool ok);
};

// Candidates of one row across all chunks, in global memory (read through L2).
struct RowCandidates {
  const uint32_t* keys;
  const int32_t* idx;
  const uint32_t* counts;
  int chunks;
  int64_t cap;
  template <class F>
  __device__ __forceinline__ void for_each(F f) const {
    for (int cx = 0; cx < chunks; ++cx) {
      const uint32_t n = __ldcg(counts + cx);
      const uint32_t* kk = keys + (int64_t)cx * cap;
      const int32_t* ii = idx + (int64_t)cx * cap;
      for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) f(__ldcg(kk + i), __ldcg(ii + i));
    }
  }
};

struct ChunkLogits {
  const float* x;
  int n;
  int64_t base;
  template <class F>
  __device__ __forceinline__ void for_each(F f) const {
    for (int i = threadIdx.x; i < n; i += blockDim.x) f(float_key(x[i]), (int32_t)(base + i));
  }
};

// Exact top-k of one row from its candidates (last CTA of the sequence).
__device__ void merge_row(FusedExtra& ex, const RowCandidates& src, int64_t n_valid, int32_t k,
                          int32_t* out) {
  if (threadIdx.x == 0) {
    ex.sc.out_count = 0;
    ex.n_cand = 0;
  }
  __syncthreads();
  auto emit = [&](uint32_t, int32_t i) { out[atomicAdd(&ex.sc.out_count, 1u)] = i; };
  if (n_valid <= k) {
    // every valid key is a candidate: list them, then pad
    src.for_each(emit);
    __syncthreads();
    const uint32_t m = ex.sc.out_count;
    for (int i = threadIdx.x; i < k; i += blockDim.x)
      if ((uint32_t)i >= m) out[i] = -1;
    __syncthreads();
    return;
  }
  uint32_t* ckeys = reinterpret_cast<uint32_t*>(ex.logits);
  int32_t* cidx = reinterpret_cast<int32_t*>(ex.logits) + kChunkFloats / 2;
  constexpr uint32_t kCap = kChunkFloats / 2;
  digit_histogram(ex.sc, src, 0, 0u, 0u);
  find_threshold_bin(ex.sc, kRadixBins, (uint32_t)k);
  const uint32_t b1 = ex.sc.bin;
  const uint32_t need = (uint32_t)k - ex.sc.above;
  const bool fits = ex.sc.hist[b1] <= kCap;
  __syncthreads();
  src.for_each([&](uint32_t key, int32_t i) {
    const uint32_t dg = key >> 21;
    if (dg > b1) {
      emit(key, i);
    } else if (dg == b1 && fits) {
      const uint32_t slot = atomicAdd(&ex.n_cand, 1u);
      ckeys[slot] = key;
      cidx[slot] = i;
    }
  });
  __syncthreads();
  const uint32_t prefix = b1 << 21, mask = 0x7FFu << 21;
  if (fits) {
    const SmemPairs cand{ckeys, cidx, (int)ex.n_cand};
    radix_select(ex.sc, cand, need, 1, prefix, mask, emit);
  } else {
    radix_select(ex.sc, src, need, 1, prefix, mask, emit);
  }
  __syncthreads();
}

template <int H, int NEXT_N>
__device__ void FusedEpilogue<H, NEXT_N>::chunk_done(const PagedArgs& p, const PagedCta& c,
                                                     uint8_t* extra, bool ok) {
  FusedExtra& ex = *reinterpret_cast<FusedExtra*>(extra);
  const TopkWs ws = ws_layout(p.workspace, p.B, NEXT_N, p.chunks, nullptr);
  const int cx = blockIdx.x;
  const uint32_t k = (uint32_t)p.topk;
  // ---- this chunk's candidates, row by row
  for (int j = 0; j < NEXT_N; ++j) {
    const int64_t r = (int64_t)c.b * NEXT_N + j;
    const int64_t len = c.L - NEXT_N + j + 1;
    int64_t n = len - c.k0;
    n = n < 0 ? 0 : (n > C ? C : n);
    if (!ok) n = 0;
    const int64_t seg = (r * p.chunks + cx) * ws.chunk_cap;
    uint32_t* okeys = ws.keys + seg;
    int32_t* oidx = ws.idx + seg;
    const ChunkLogits src{ex.logits + j * C, (int)n, c.k0};
    if (n <= (int64_t)k) {
      src.for_each([&](uint32_t key, int32_t i) {
        okeys[i - c.k0] = key;
        oidx[i - c.k0] = i;
      });
      if (threadIdx.x == 0) ws.counts[r * p.chunks + cx] = (uint32_t)n;
    } else {
      if (threadIdx.x == 0) ex.sc.out_count = 0;
      digit_histogram(ex.sc, src, 0, 0u, 0u);
      find_threshold_bin(ex.sc, kRadixBins, k);
      const uint32_t b1 = ex.sc.bin;
      src.for_each([&](uint32_t key, int32_t i) {
        if ((key >> 21) >= b1) {
          const uint32_t slot = atomicAdd(&ex.sc.out_count, 1u);
          okeys[slot] = key;
          oidx[slot] = i;
        }
      });
      __syncthreads();
      if (threadIdx.x == 0) ws.counts[r * p.chunks + cx] = ex.sc.out_count;
    }
    __syncthreads();
  }
  // ---- publish, then the last CTA of the sequence merges
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) ex.ticket = atomicAdd(ws.tickets + c.b, 1u);
  __syncthreads();
  if (ex.ticket != (uint32_t)p.chunks - 1) return;
  __threadfence();
  for (int j = 0; j < NEXT_N; ++j) {
    const int64_t r = (int64_t)c.b * NEXT_N + j;
    const int64_t len = c.L - NEXT_N + j + 1;
    const RowCandidates src{ws.keys + r * p.chunks * ws.chunk_cap,
                            ws.idx + r * p.chunks * ws.chunk_cap, ws.counts + r * p.chunks,
                            p.chunks, ws.chunk_cap};
    merge_row(ex, src, len < 0 ? 0 : len, p.topk, p.out_idx + r * p.topk);
  }
}

template <int H, int NEXT_N>
__global__ void __launch_bounds__(kPagedThreads, 1)
    paged_topk_kernel(const __grid_constant__ CUtensorMap tm_vals,
                      const __grid_constant__ CUtensorMap tm_scales, const PagedArgs p) {
  using Ep = FusedEpilogue<H, NEXT_N>;
  PagedCta c;
  if (!paged_cta_setup(p, c)) {
    // nothing to score in this chunk: publish empty candidate lists and take
    // part in the ticket so that the merge still happens exactly once
    uint8_t* sm = aligned_smem_base();
    Ep::chunk_done(p, c, sm + PagedLayout<H * NEXT_N>::kExtra, true);
    return;
  }
  paged_cta_run<H, NEXT_N, Ep>(&tm_vals, &tm_scales, p, c);
}

template <int H, int NEXT_N>
cudaError_t launch_one(const CUtensorMap& tv, const CUtensorMap& ts, const PagedArgs& a,
                       cudaStream_t stream) {
  using Ep = FusedEpilogue<H, NEXT_N>;
  const size_t smem = paged_smem_bytes<H * NEXT_N>() + Ep::kExtraSmem;
  auto kern = paged_topk_kernel<H, NEXT_N>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(a.workspace, 0, (size_t)a.B * 4, stream);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.chunks, (unsigned)a.B);
  kern<<<grid, kPagedThreads, smem, stream>>>(tv, ts, a);
  return cudaGetLastError();
}

}  // namespace

size_t paged_topk_workspace_bytes(int32_t B, int32_t next_n, int32_t max_blocks, int32_t k,
                                  int32_t* tiles_per_cta_out, int32_t* chunks_out) {
  (void)k;
  if (B <= 0 || (next_n != 1 && next_n != 2) || max_blocks <= 0) return 0;
  const int64_t C = kChunkFloats / next_n;
  const int64_t chunks = ((int64_t)max_blocks * kPage + C - 1) / C;
  if (tiles_per_cta_out) *tiles_per_cta_out = (int32_t)(C / kTileKeys);
  if (chunks_out) *chunks_out = (int32_t)chunks;
  size_t total = 0;
  ws_layout(nullptr, B, next_n, (int32_t)chunks, &total);
  return total;
}

cudaError_t launch_paged_logits_topk(const CUtensorMap& tv, const CUtensorMap& ts, int H,
                                     int next_n, const PagedArgs& a, cudaStream_t stream) {
  if (H == 32 && next_n == 1) return launch_one<32, 1>(tv, ts, a, stream);
  if (H == 32 && next_n == 2) return launch_one<32, 2>(tv, ts, a, stream);
  if (H == 64 && next_n == 1) return launch_one<64, 1>(tv, ts, a, stream);
  if (H == 64 && next_n == 2) return launch_one<64, 2>(tv, ts, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace idx
