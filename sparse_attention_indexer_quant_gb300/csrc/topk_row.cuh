// Top-k of one logits row per CTA (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": top_k_per_row into
// topk_indices_buffer; rows shorter than k are padded with -1).
//
// The row is processed in chunks of CHUNK elements staged in shared memory:
//   1. coarse histogram of the row (top 12 key bits: sign, exponent and three
//      mantissa bits) while the chunk is loaded; the bin b1 holding the k-th
//      largest value and the count above it follow from one block-wide scan;
//   2. every thread counts its elements above b1 and in b1; one block scan of
//      the packed counts gives each thread its output and candidate offsets, so
//      the elements above b1 go straight to out and b1's elements to a
//      shared-memory candidate list without atomics;
//   3. the exact remainder among b1's elements: their next 8 key bits give
//      the sub-bin holding the k-th largest (one warp scans the 256 counts);
//      the elements above it take the next slots, and the few in it are
//      ranked against each other (value, then position), or resolved by radix
//      digits on the low 12 key bits when there are many.
// A row of at most CHUNK elements is read from global memory once.  If b1
// holds more elements than the candidate list, step 3 runs its radix passes
// over the row itself, restricted to b1.
#pragma once

#include "common.cuh"
#include "topk_select.cuh"

namespace idx {

constexpr int kRowThreads = 512;
constexpr int kRowCandCap = 4096;
constexpr int kRowList2 = 2048;      // sub-bin list, in the spent staging buffer
constexpr int kRowRankDirect = 64;   // sub-bin lists ranked element by element

template <int CHUNK>
struct RowTopkSmem {
  SelectScratch sel;
  uint32_t cand_keys[kRowCandCap];
  int32_t cand_idx[kRowCandCap];
  uint32_t out_base;
  uint32_t cand_base;
  uint32_t slot;
  uint32_t n2;
  uint32_t keys[CHUNK];
  static_assert(CHUNK >= 2 * kRowList2, "the sub-bin list lives in the staging buffer");
};

// The k largest of x[0, len) -> out[0, k) as positions 0..len-1 (any order),
// -1 padded.  All threads of the CTA call it.
template <int CHUNK>
__device__ __forceinline__ void row_topk(RowTopkSmem<CHUNK>& sm, const float* __restrict__ x,
                                         int64_t len, int32_t k, int32_t* __restrict__ out) {
  if (len <= k) {
    for (int64_t i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < len ? (int32_t)i : -1;
    return;
  }
  const int n_chunks = (int)((len + CHUNK - 1) / CHUNK);
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) sm.sel.hist[i] = 0;
  if (threadIdx.x == 0) {
    sm.out_base = 0;
    sm.cand_base = 0;
  }
  __syncthreads();

  // stage chunk c's keys in shared memory; with hist, count them too
  auto stage = [&](int c, bool hist) {
    const int64_t c0 = (int64_t)c * CHUNK;
    const int n = (int)(len - c0 < CHUNK ? len - c0 : CHUNK);
    for (int base = 0; base < n; base += kBatch * kRowThreads) {
      float v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + u * kRowThreads + threadIdx.x;
        v[u] = i < n ? __ldcg(x + c0 + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + u * kRowThreads + threadIdx.x;
        if (i < n) {
          const uint32_t key = float_key(v[u]);
          sm.keys[i] = key;
          if (hist) atomicAdd(&sm.sel.hist[coarse_bin(key)], 1u);
        }
      }
    }
    return n;
  };

  // ---- 1. coarse histogram
  int n_last = 0;
  for (int c = 0; c < n_chunks; ++c) n_last = stage(c, true);
  __syncthreads();
  find_threshold_bin(sm.sel.hist, kCoarseBins, (uint32_t)k, sm.sel.s);
  const uint32_t b1 = sm.sel.s.bin;
  const uint32_t above = sm.sel.s.above;
  const uint32_t nb1 = sm.sel.hist[b1];
  const bool fits = nb1 <= (uint32_t)kRowCandCap;

  // ---- 2. elements above b1 to out, b1's elements to the candidate list
  for (int c = 0; c < n_chunks; ++c) {
    int n = n_last;
    if (n_chunks > 1) {
      __syncthreads();
      n = stage(c, false);
      __syncthreads();
    }
    // thread t takes elements t, t + 512, ... (conflict-free shared reads);
    // its outputs go to a range of its own
    uint32_t n_gt = 0, n_eq = 0;
    for (int i = threadIdx.x; i < n; i += kRowThreads) {
      const uint32_t bin = coarse_bin(sm.keys[i]);
      n_gt += bin > b1 ? 1u : 0u;
      n_eq += bin == b1 ? 1u : 0u;
    }
    // both block sums fit 16 bits: fewer than k <= 2048 elements of the row
    // lie above b1, and a chunk holds at most 32768 elements of b1
    const uint32_t packed = (n_gt << 16) | n_eq;
    const uint32_t excl = block_exclusive_scan(packed, sm.sel.s);
    uint32_t o = sm.out_base + (excl >> 16);
    uint32_t cc = sm.cand_base + (excl & 0xFFFFu);
    const int64_t c0 = (int64_t)c * CHUNK;
    for (int i = threadIdx.x; i < n; i += kRowThreads) {
      const uint32_t key = sm.keys[i];
      const uint32_t bin = coarse_bin(key);
      if (bin > b1) out[o++] = (int32_t)(c0 + i);
      if (bin == b1) {
        if (fits) {
          sm.cand_keys[cc] = key;
          sm.cand_idx[cc] = (int32_t)(c0 + i);
        }
        ++cc;
      }
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      sm.out_base = o;  // the last thread's offsets are the running totals
      sm.cand_base = cc;
    }
    __syncthreads();
  }

  // ---- 3. the exact remainder inside b1: b1's elements by their next 8 key
  //         bits (the sub-bin sb1 holding the k-th largest), those above sb1
  //         to the output, then among sb1's few elements by rank (key, then
  //         position), or by radix digits on the low 12 bits when there are
  //         many
  const uint32_t need = (uint32_t)k - above;
  if (threadIdx.x == 0) sm.slot = above;
  auto emit = [&](uint32_t, int32_t i) { out[warp_claim(&sm.slot, true)] = i; };
  if (!fits) {
    __syncthreads();
    const GlobalLogits<true> row{x, 0, len};
    radix_select(sm.sel.hist, sm.sel.s, row, need, b1 << kCoarseShift, 32 - kCoarseShift, emit);
    return;
  }
  uint32_t* const sub = sm.sel.hist;  // the coarse histogram is spent
  if (threadIdx.x < kSubBins) sub[threadIdx.x] = 0u;
  if (threadIdx.x == 0) sm.n2 = 0u;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < nb1; i += kRowThreads)
    atomicAdd(&sub[(sm.cand_keys[i] >> kSubShift) & (kSubBins - 1)], 1u);
  __syncthreads();
  if (threadIdx.x < 32) warp_find_sub_bin(sub, need, sm.sel.s);
  __syncthreads();
  const uint32_t sb1 = sm.sel.s.bin;
  const uint32_t above2 = sm.sel.s.above;  // b1's elements above sb1
  uint32_t* const keys2 = sm.keys;          // sb1's elements (the staging buffer is spent)
  int32_t* const idx2 = reinterpret_cast<int32_t*>(sm.keys + kRowList2);
  for (uint32_t i = threadIdx.x; i < nb1; i += kRowThreads) {
    const uint32_t key = sm.cand_keys[i];
    const int32_t pos = sm.cand_idx[i];
    const uint32_t sb = (key >> kSubShift) & (kSubBins - 1);
    const uint32_t s = warp_claim(&sm.slot, sb > sb1);
    if (sb > sb1) out[s] = pos;
    const uint32_t s2 = warp_claim(&sm.n2, sb == sb1);
    if (sb == sb1 && s2 < (uint32_t)kRowList2) {
      keys2[s2] = key;
      idx2[s2] = pos;
    }
  }
  __syncthreads();
  const uint32_t n2 = sm.n2;
  const uint32_t need2 = need - above2;
  if (n2 <= (uint32_t)kRowRankDirect) {
    if (threadIdx.x < n2) {
      const uint32_t key = keys2[threadIdx.x];
      const int32_t pos = idx2[threadIdx.x];
      uint32_t rank = 0;
      for (uint32_t q = 0; q < n2; ++q) {
        const uint32_t kq = keys2[q];
        rank += (kq > key || (kq == key && idx2[q] < pos)) ? 1u : 0u;
      }
      if (rank < need2) out[above + above2 + rank] = pos;
    }
    return;
  }
  const uint32_t prefix = (b1 << kCoarseShift) | (sb1 << kSubShift);
  if (n2 <= (uint32_t)kRowList2) {
    const SmemPairs cand{keys2, idx2, (int)n2};
    radix_select(sm.sel.hist, sm.sel.s, cand, need2, prefix, 32 - kSubShift, emit);
  } else {
    const SmemPairs cand{sm.cand_keys, sm.cand_idx, (int)nb1};
    radix_select(sm.sel.hist, sm.sel.s, cand, need2, prefix, 32 - kSubShift, emit);
  }
}

}  // namespace idx
