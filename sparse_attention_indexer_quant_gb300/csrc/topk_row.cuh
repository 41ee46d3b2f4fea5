// Top-k of one logits row per CTA (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": top_k_per_row into
// topk_indices_buffer; rows shorter than k are padded with -1).
//
// A row whose start is 16-byte aligned is streamed from global memory (L2 on
// the second pass) in rounds of float4 loads, eight of a thread's in flight;
// other rows are staged in shared memory in chunks of CHUNK elements:
//   1. coarse histogram of the row (top 12 key bits: sign, exponent and three
//      mantissa bits); the bin b1 holding the k-th largest value and the count
//      above it follow from one block-wide scan;
//   2. streamed rows: each thread classifies its elements of a round as above
//      b1 or in it (bit masks) and a warp takes its output and candidate slots
//      with one shared-memory atomic add per list; staged rows: per chunk, one
//      block scan of the packed counts gives each thread its offsets.  The
//      elements above b1 go straight to out, b1's elements to a shared-memory
//      candidate list;
//   3. the exact remainder among b1's elements: their next 8 key bits give
//      the sub-bin holding the k-th largest (one warp scans the 256 counts);
//      the elements above it take the next slots, and the few in it are
//      ranked against each other (value, then position), or resolved by radix
//      digits on the low 12 key bits when there are many.
// If b1 holds more elements than the candidate list, step 3 runs its radix
// passes over the row itself, restricted to b1.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "topk_select.cuh"

namespace idx {

constexpr int kRowThreads = 256;     // four CTAs (rows) per SM
constexpr int kRowCandCap = 2048;
constexpr int kRowVec = 8;           // float4 loads of a thread in flight per round
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

// Element `bit` (float4 bit >> 2, lane bit & 3) of a thread's round, picked by
// selects rather than an indexed (local-memory) array access.
__device__ __forceinline__ float round_value(const float4 (&v)[kRowVec], int bit) {
  static_assert(kRowVec == 8, "three select levels");
  const int u = bit >> 2;
  const float4 a01 = (u & 1) ? v[1] : v[0], a23 = (u & 1) ? v[3] : v[2];
  const float4 a45 = (u & 1) ? v[5] : v[4], a67 = (u & 1) ? v[7] : v[6];
  const float4 b0 = (u & 2) ? a23 : a01, b1 = (u & 2) ? a67 : a45;
  const float4 c = (u & 4) ? b1 : b0;
  const float lo = (bit & 1) ? c.y : c.x, hi = (bit & 1) ? c.w : c.z;
  return (bit & 2) ? hi : lo;
}

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

  // ---- 1. coarse histogram.  A 16-byte aligned row is streamed with float4
  //         loads, eight of a thread's in flight at once (8192 elements of
  //         the row per round); other rows are staged chunk by chunk.
  int n_last = 0;
  const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  // a round: thread t's float4 u covers elements base + 4 * (u * kRowThreads + t) ..+3
  auto load_round = [&](int64_t base, float4 (&v)[kRowVec], auto full) {
    constexpr bool kFull = decltype(full)::value;
#pragma unroll
    for (int u = 0; u < kRowVec; ++u) {
      const int64_t i0 = base + 4 * ((int64_t)u * kRowThreads + threadIdx.x);
      if (kFull || i0 + 3 < len) {
        v[u] = __ldcg(reinterpret_cast<const float4*>(x + i0));
      } else {
        v[u].x = i0 + 0 < len ? __ldcg(x + i0 + 0) : 0.f;
        v[u].y = i0 + 1 < len ? __ldcg(x + i0 + 1) : 0.f;
        v[u].z = i0 + 2 < len ? __ldcg(x + i0 + 2) : 0.f;
        v[u].w = i0 + 3 < len ? __ldcg(x + i0 + 3) : 0.f;
      }
    }
  };
  constexpr int64_t kRound = (int64_t)kRowVec * 4 * kRowThreads;
  if (aligned) {
    constexpr int kVec = kRowVec;
    // a round wholly inside the row skips the per-element bounds tests
    auto hist_round = [&](int64_t base, auto full) {
      constexpr bool kFull = decltype(full)::value;
      float4 v[kVec];
      load_round(base, v, full);
      // the next round's lines start on their way to L2 while this round's
      // keys are counted (no registers held for them)
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const int64_t i1 = base + kRound + 4 * ((int64_t)u * kRowThreads + threadIdx.x);
        if (i1 < len) asm volatile("prefetch.global.L2 [%0];" ::"l"(x + i1));
      }
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const int64_t i0 = base + 4 * ((int64_t)u * kRowThreads + threadIdx.x);
        const float e4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (kFull || i0 + q < len) {
            const uint32_t key = float_key(e4[q]);
            atomicAdd(&sm.sel.hist[coarse_bin(key)], 1u);
          }
        }
      }
    };
    for (int64_t base = 0; base < len; base += kRound) {
      if (base + kRound <= len)
        hist_round(base, std::integral_constant<bool, true>());
      else
        hist_round(base, std::integral_constant<bool, false>());
    }
    n_last = (int)(len - (int64_t)(n_chunks - 1) * CHUNK);
  } else {
    for (int c = 0; c < n_chunks; ++c) n_last = stage(c, true);
  }
  __syncthreads();
  find_threshold_bin(sm.sel.hist, kCoarseBins, (uint32_t)k, sm.sel.s);
  const uint32_t b1 = sm.sel.s.bin;
  const uint32_t above = sm.sel.s.above;
  const uint32_t nb1 = sm.sel.hist[b1];
  const bool fits = nb1 <= (uint32_t)kRowCandCap;

  // ---- 2. elements above b1 to out, b1's elements to the candidate list.
  //         An aligned row is streamed again (it is in L2): each thread
  //         classifies its elements of a round into bit masks, and a warp
  //         takes its slots with one shared-memory atomic add per list.
  if (aligned) {
    const uint32_t key_b1 = b1 << kCoarseShift;
    const uint32_t key_gt = key_b1 | ((1u << kCoarseShift) - 1u);
    const int lane = threadIdx.x & 31;
    auto classify_round = [&](int64_t base, auto full) {
      constexpr bool kFull = decltype(full)::value;
      float4 v[kRowVec];
      load_round(base, v, full);
      uint32_t gt = 0u, eq = 0u;
#pragma unroll
      for (int u = 0; u < kRowVec; ++u) {
        const int64_t i0 = base + 4 * ((int64_t)u * kRowThreads + threadIdx.x);
        const float e4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t key = float_key(e4[q]);
          const bool in = kFull || i0 + q < len;
          const uint32_t bit = 1u << (4 * u + q);
          gt |= (key > key_gt && in) ? bit : 0u;
          eq |= ((key ^ key_b1) < (1u << kCoarseShift) && in) ? bit : 0u;
        }
      }
      const uint32_t ng = __popc(gt), ne = __popc(eq);
      uint32_t ig = ng, ie = ne;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t yg = __shfl_up_sync(0xFFFFFFFFu, ig, o);
        const uint32_t ye = __shfl_up_sync(0xFFFFFFFFu, ie, o);
        if (lane >= o) {
          ig += yg;
          ie += ye;
        }
      }
      uint32_t bg = 0, be = 0;
      if (lane == 31) {
        if (ig != 0u) bg = atomicAdd(&sm.out_base, ig);
        if (ie != 0u) be = atomicAdd(&sm.cand_base, ie);
      }
      uint32_t o = __shfl_sync(0xFFFFFFFFu, bg, 31) + ig - ng;
      uint32_t cc = __shfl_sync(0xFFFFFFFFu, be, 31) + ie - ne;
      auto pos = [&](int bit) -> int64_t {
        return base + 4 * ((int64_t)(bit >> 2) * kRowThreads + threadIdx.x) + (bit & 3);
      };
      for (; gt != 0u; gt &= gt - 1u) out[o++] = (int32_t)pos(__ffs(gt) - 1);
      for (; eq != 0u; eq &= eq - 1u) {
        const int bit = __ffs(eq) - 1;
        if (fits) {
          sm.cand_keys[cc] = float_key(round_value(v, bit));
          sm.cand_idx[cc] = (int32_t)pos(bit);
        }
        ++cc;
      }
    };
    for (int64_t base = 0; base < len; base += kRound) {
      if (base + kRound <= len)
        classify_round(base, std::integral_constant<bool, true>());
      else
        classify_round(base, std::integral_constant<bool, false>());
    }
    __syncthreads();
  } else
  for (int c = 0; c < n_chunks; ++c) {
    int n = n_last;
    if (n_chunks > 1) {
      __syncthreads();
      n = stage(c, false);
      __syncthreads();
    }
    // thread t takes elements t, t + kRowThreads, ... (conflict-free shared reads);
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
  for (int i = threadIdx.x; i < kSubBins; i += kRowThreads) sub[i] = 0u;
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
