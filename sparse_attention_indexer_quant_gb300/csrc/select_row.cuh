// Exact top-k of one fp32 row by a thread-block cluster (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": top_k_per_row into
// topk_indices_buffer; rows of at most k elements list all of them, then -1).
//
// The P CTAs of a cluster each take a slice of the row, held in registers:
//   1. every CTA builds the coarse histogram of its slice (the top 12 bits of
//      each value's order-preserving key) in shared memory; summed over the
//      cluster through distributed shared memory it gives the bin b1 holding
//      the k-th largest value and the count above it;
//   2. each thread classifies its elements as above b1 or in it (bit masks);
//      a warp takes its output and candidate slots with one atomic add per
//      list on the leader's counters (through distributed shared memory); the
//      elements above go straight to the output, b1's elements (a few hundred
//      for smooth rows) with their keys into the leader's shared memory;
//   3. the leader takes the remaining ones from the candidates: by their next
//      8 key bits (the sub-bin holding the k-th largest), then among that
//      sub-bin's elements by rank (key, then position), or by a radix digit
//      on the low 12 bits when there are many.  A boundary bin larger than
//      the candidate list is resolved by radix passes over the row.
// Output positions are relative to the row start, in no particular order;
// equal values may be taken in any order.
#pragma once

#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "topk_select.cuh"

namespace idx {

constexpr int kSelThreads = 512;
constexpr int kSelVec = 4;                              // float4 loads per thread per chunk
constexpr int kSelChunk = kSelThreads * 4 * kSelVec;    // 8192 elements
constexpr int kCandSmem = 8192;                         // boundary-bin elements in the leader
constexpr int kMaxParts = 4;                            // CTAs per row at most
constexpr int kMinSlice = 4096;                         // elements per CTA at least
constexpr int kList2 = 2048;                            // boundary sub-bin list (leader)
constexpr int kRankDirect = 64;                         // sub-bin lists ranked element by element
static_assert(kCoarseBins == 8 * kSelThreads, "each select thread owns eight histogram bins");

struct SelSmem {
  uint32_t bins[kCoarseBins];  // coarse histogram of this CTA's slice
  uint32_t tsum[kSelThreads];  // per thread: its eight bins' slice count (read by the cluster)
  uint32_t sub[kSubBins];      // the candidates by their next 8 key bits (leader)
  uint32_t hist[kRadixBins];   // radix-digit scratch (leader)
  ScanScratch s;
  uint32_t nb1;                // the row's elements in the boundary bin
  uint32_t n_out;              // output slots handed out (leader; the cluster adds to it)
  uint32_t n_cand;             // candidate slots handed out (leader; likewise)
  uint32_t n2;                 // candidates in the boundary sub-bin (leader)
  uint32_t cand_keys[kCandSmem];
  int32_t cand_idx[kCandSmem];
  uint32_t keys2[kList2];      // the boundary sub-bin's candidates (leader)
  int32_t idx2[kList2];
};

// Keys of x[i] for this thread's 32 positions of the chunk pair at `base`
// (chunks base and base + kSelChunk; key(-inf) at positions from s1 on, which
// the passes below never count).  Four at a time when x is 16-byte aligned
// (base is a multiple of 4), else one by one; all of a thread's loads are
// issued before any key is formed, so they are in flight together.
__device__ __forceinline__ void load_pair_keys(const float* x, bool aligned, int32_t base,
                                               int32_t s1, int t, uint4 (&ka)[kSelVec],
                                               uint4 (&kb)[kSelVec]) {
  float4 v[2 * kSelVec];
#pragma unroll
  for (int j = 0; j < 2 * kSelVec; ++j) {
    const int32_t i0 = base + (j / kSelVec) * kSelChunk + 4 * ((j % kSelVec) * kSelThreads + t);
    if (aligned && i0 + 3 < s1) {
      v[j] = __ldca(reinterpret_cast<const float4*>(x + i0));
    } else {
      v[j].x = i0 + 0 < s1 ? __ldca(x + i0 + 0) : -INFINITY;
      v[j].y = i0 + 1 < s1 ? __ldca(x + i0 + 1) : -INFINITY;
      v[j].z = i0 + 2 < s1 ? __ldca(x + i0 + 2) : -INFINITY;
      v[j].w = i0 + 3 < s1 ? __ldca(x + i0 + 3) : -INFINITY;
    }
  }
#pragma unroll
  for (int u = 0; u < kSelVec; ++u) {
    const float4 a = v[u], b = v[kSelVec + u];
    ka[u] = make_uint4(float_key(a.x), float_key(a.y), float_key(a.z), float_key(a.w));
    kb[u] = make_uint4(float_key(b.x), float_key(b.y), float_key(b.z), float_key(b.w));
  }
}

// Key of mask bit `bit` of a chunk pair held in registers (chunk bit >> 4,
// float4 (bit >> 2) & 3, lane bit & 3), by selects rather than an indexed
// (local-memory) array access.
__device__ __forceinline__ uint32_t pair_key(const uint4 (&ka)[kSelVec], const uint4 (&kb)[kSelVec],
                                             int bit) {
  static_assert(kSelVec == 4, "four float4 per chunk");
  const bool u0 = (bit & 4) != 0, u1 = (bit & 8) != 0;
  const uint4 a = u1 ? (u0 ? ka[3] : ka[2]) : (u0 ? ka[1] : ka[0]);
  const uint4 b = u1 ? (u0 ? kb[3] : kb[2]) : (u0 ? kb[1] : kb[0]);
  const uint4 v = (bit & 16) ? b : a;
  const uint32_t lo = (bit & 1) ? v.y : v.x, hi = (bit & 1) ? v.w : v.z;
  return (bit & 2) ? hi : lo;
}

// Adds the chunk's positions below s1 to the CTA's histogram.
__device__ __forceinline__ void hist_keys(uint32_t* bins, const uint4 (&kv)[kSelVec], int32_t base,
                                          int32_t s1, int t) {
#pragma unroll
  for (int u = 0; u < kSelVec; ++u) {
    const int32_t i0 = base + 4 * (u * kSelThreads + t);
    const uint32_t e4[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
    if (i0 + 3 < s1) {
#pragma unroll
      for (int q = 0; q < 4; ++q) atomicAdd(&bins[coarse_bin(e4[q])], 1u);
    } else if (i0 < s1) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (i0 + q < s1) atomicAdd(&bins[coarse_bin(e4[q])], 1u);
    }
  }
}

// The k largest of x[0, len) -> out[0, k) (positions, -1 padded).  Called by
// every thread of every CTA of a cluster of `parts` CTAs (kSelThreads each)
// with the same arguments; every CTA takes the same branches and passes the
// same two cluster barriers.
__device__ __forceinline__ void cluster_select_row(SelSmem& sm, const float* x, int64_t len,
                                                   uint32_t k, int32_t* out, int parts) {
  const int part = (int)cluster_ctarank();
  const int t = threadIdx.x;
  const int lane = t & 31;
  const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  if (len <= (int64_t)k) {  // the whole cluster leaves here
    if (part == 0)
      for (int i = t; i < (int)k; i += kSelThreads) out[i] = i < len ? i : -1;
    return;
  }
  // positions within a row fit 32 bits (the output indices are int32)
  const int32_t n = (int32_t)len;
  const int32_t slice = ((n + parts - 1) / parts + 3) / 4 * 4;
  const int32_t s0 = part * slice;
  const int32_t s1 = s0 + slice < n ? s0 + slice : n;
  const int n_chunks = (slice + kSelChunk - 1) / kSelChunk;

  uint4 ka[kSelVec], kb[kSelVec];
  load_pair_keys(x, aligned, s0, s1, t, ka, kb);
#pragma unroll
  for (int q = 0; q < 8; ++q) sm.bins[8 * t + q] = 0u;
  if (t < kSubBins) sm.sub[t] = 0u;
  if (t == 0) {
    sm.s.bin = 0;
    sm.s.above = 0;
    sm.nb1 = 0;
    sm.n_out = 0;
    sm.n_cand = 0;
    sm.n2 = 0;
  }
  __syncthreads();

  // ---- 1. coarse histogram of the slice, then of the row
  for (int c = 0; c < n_chunks; c += 2) {  // (past two chunks the later pass reloads)
    if (c > 0) {
      load_pair_keys(x, aligned, s0 + c * kSelChunk, s1, t, ka, kb);
    }
    hist_keys(sm.bins, ka, s0 + c * kSelChunk, s1, t);
    hist_keys(sm.bins, kb, s0 + (c + 1) * kSelChunk, s1, t);
  }
  __syncthreads();  // the slice histogram is complete
  // thread t owns bins 4088 - 8t + j (j = 0..7): its slice counts, and their
  // sum, published for the cluster
  uint32_t h8[8];
  {
    const uint4 lo = *reinterpret_cast<const uint4*>(&sm.bins[kCoarseBins - 8 - 8 * t]);
    const uint4 hi = *reinterpret_cast<const uint4*>(&sm.bins[kCoarseBins - 4 - 8 * t]);
    h8[0] = lo.x;
    h8[1] = lo.y;
    h8[2] = lo.z;
    h8[3] = lo.w;
    h8[4] = hi.x;
    h8[5] = hi.y;
    h8[6] = hi.z;
    h8[7] = hi.w;
  }
  uint32_t local = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) local += h8[j];
  sm.tsum[t] = local;
  cluster_sync_all();  // #1: every CTA's slice sums are published, the counters zeroed
  {  // the row's count over thread t's bins (the other slices' sums in flight together)
    const uint32_t my = smem_u32(&sm.tsum[t]);
    uint32_t r[kMaxParts];
#pragma unroll
    for (int q = 0; q < kMaxParts; ++q)
      r[q] = q < parts && q != part ? ld_cluster_u32(cluster_map(my, (uint32_t)q)) : 0u;
#pragma unroll
    for (int q = 0; q < kMaxParts; ++q) local += r[q];
  }
  const uint32_t excl = block_exclusive_scan(local, sm.s);
  if (excl < k && k <= excl + local) {  // the thread holding the k-th largest
    // the row's counts of its eight bins: the other slices' through DSMEM
    const uint32_t my0 = smem_u32(&sm.bins[kCoarseBins - 8 - 8 * t]);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    uint4 v[2 * kMaxParts];
#pragma unroll
    for (int q = 0; q < kMaxParts; ++q) {
      const bool other = q < parts && q != part;
      v[2 * q] = other ? ld_cluster_v4(cluster_map(my0, (uint32_t)q)) : z;
      v[2 * q + 1] = other ? ld_cluster_v4(cluster_map(my0 + 16u, (uint32_t)q)) : z;
    }
#pragma unroll
    for (int q = 0; q < kMaxParts; ++q) {
      h8[0] += v[2 * q].x;
      h8[1] += v[2 * q].y;
      h8[2] += v[2 * q].z;
      h8[3] += v[2 * q].w;
      h8[4] += v[2 * q + 1].x;
      h8[5] += v[2 * q + 1].y;
      h8[6] += v[2 * q + 1].z;
      h8[7] += v[2 * q + 1].w;
    }
    uint32_t run = excl;
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // bins 4095 - 8t - q, highest first
      const uint32_t h = h8[7 - q];
      if (run < k && k <= run + h) {
        sm.s.bin = (uint32_t)(kCoarseBins - 1 - 8 * t - q);
        sm.s.above = run;
        sm.nb1 = h;
      }
      run += h;
    }
  }
  __syncthreads();
  const uint32_t b1 = sm.s.bin;
  const uint32_t above = sm.s.above;  // the row's elements in bins above b1
  const uint32_t nb = sm.nb1;         // ... and in b1

  // Each thread's elements of a chunk pair are 32 mask bits: bit 16*h + 4*u + q
  // is chunk h of the pair, float4 u, lane q of it.
  auto position = [&](int c, int bit) -> int32_t {  // chunk pair starting at chunk c
    return s0 + (c + (bit >> 4)) * kSelChunk + 4 * (((bit >> 2) & 3) * kSelThreads + t) + (bit & 3);
  };

  // ---- 2. each thread's elements above b1 go to the output, those in b1
  //         (key and position) to the leader's candidate list; a warp takes
  //         its slots with one atomic add per list on the leader's counters
  //         (positions past the slice are skipped: their key(-inf) padding is
  //         in b1 when the row's k-th largest value is itself -inf)
  const uint32_t n_out0 = cluster_map(smem_u32(&sm.n_out), 0);
  const uint32_t n_cand0 = cluster_map(smem_u32(&sm.n_cand), 0);
  const uint32_t cand_keys0 = cluster_map(smem_u32(sm.cand_keys), 0);
  const uint32_t cand_idx0 = cluster_map(smem_u32(sm.cand_idx), 0);
  const uint32_t key_b1 = b1 << kCoarseShift;                  // b1's keys share these top bits
  const uint32_t key_gt = key_b1 | ((1u << kCoarseShift) - 1u);  // keys above b1 exceed this
  const uint32_t pad_bin = coarse_bin(float_key(-INFINITY));   // the padding's bin
  const bool reload = n_chunks > 2;
  for (int c = 0; c < n_chunks; c += 2) {
    if (reload) {
      load_pair_keys(x, aligned, s0 + c * kSelChunk, s1, t, ka, kb);
    }
    uint32_t gt = 0u, eq = 0u;
    if (b1 > pad_bin) {  // the key(-inf) padding is neither above b1 nor in it
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int u = 0; u < kSelVec; ++u) {
          const uint4 v = h == 0 ? ka[u] : kb[u];
          const uint32_t e4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t bit = 1u << (16 * h + 4 * u + q);
            gt |= e4[q] > key_gt ? bit : 0u;
            eq |= (e4[q] ^ key_b1) < (1u << kCoarseShift) ? bit : 0u;
          }
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int u = 0; u < kSelVec; ++u) {
          const uint4 v = h == 0 ? ka[u] : kb[u];
          const uint32_t e4[4] = {v.x, v.y, v.z, v.w};
          const int32_t i0 = s0 + (c + h) * kSelChunk + 4 * (u * kSelThreads + t);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t bit = 1u << (16 * h + 4 * u + q);
            const bool in = i0 + q < s1;
            gt |= (e4[q] > key_gt && in) ? bit : 0u;
            eq |= ((e4[q] ^ key_b1) < (1u << kCoarseShift) && in) ? bit : 0u;
          }
        }
      }
    }
    const uint32_t ng = __popc(gt), ne = __popc(eq);
    uint32_t ig = ng, ie = ne;  // inclusive sums over the warp's lanes
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
    if (lane == 31) {  // the warp's totals
      if (ig != 0u) bg = atom_add_cluster_u32(n_out0, ig);
      if (ie != 0u) be = atom_add_cluster_u32(n_cand0, ie);
    }
    uint32_t o = __shfl_sync(0xFFFFFFFFu, bg, 31) + ig - ng;
    uint32_t ce = __shfl_sync(0xFFFFFFFFu, be, 31) + ie - ne;
    for (; gt != 0u; gt &= gt - 1u) {
      if (o < above) out[o] = position(c, __ffs(gt) - 1);
      ++o;
    }
    for (; eq != 0u; eq &= eq - 1u) {
      const int bit = __ffs(eq) - 1;
      if (ce < (uint32_t)kCandSmem) {
        st_cluster_u32(cand_keys0 + 4u * ce, pair_key(ka, kb, bit));
        st_cluster_u32(cand_idx0 + 4u * ce, (uint32_t)position(c, bit));
      }
      ++ce;
    }
  }
  cluster_sync_all();  // #2: the candidates are in the leader; no remote access follows
  if (part != 0) return;

  // ---- 3. the leader takes the remaining need = k - above of b1's nb
  //         elements: by their next 8 key bits (sub-bin sb1), then among
  //         sb1's few elements by rank (key, then position), or by a radix
  //         digit on the low 12 bits when there are many.  Its output
  //         counter stands at `above` and hands out the remaining slots.
  const uint32_t need = k - above;
  auto emit = [&](uint32_t, int32_t i) {
    const uint32_t s = warp_claim(&sm.n_out, true);
    if (s < k) out[s] = i;
  };
  if (nb > (uint32_t)kCandSmem) {
    // more such elements than the list holds: radix passes over the row
    const GlobalLogits<true> row{x, 0, (int64_t)n};
    radix_select(sm.hist, sm.s, row, need, b1 << kCoarseShift, 32 - kCoarseShift, emit);
    return;
  }
  for (uint32_t i = t; i < nb; i += kSelThreads)
    atomicAdd(&sm.sub[(sm.cand_keys[i] >> kSubShift) & (kSubBins - 1)], 1u);
  __syncthreads();
  if (t < 32) warp_find_sub_bin(sm.sub, need, sm.s);
  __syncthreads();
  const uint32_t sb1 = sm.s.bin;
  const uint32_t above2 = sm.s.above;  // b1's elements above sb1
  for (uint32_t i = t; i < nb; i += kSelThreads) {
    const uint32_t key = sm.cand_keys[i];
    const int32_t pos = sm.cand_idx[i];
    const uint32_t sub = (key >> kSubShift) & (kSubBins - 1);
    const uint32_t s = warp_claim(&sm.n_out, sub > sb1);
    if (sub > sb1 && s < k) out[s] = pos;
    const uint32_t s2 = warp_claim(&sm.n2, sub == sb1);
    if (sub == sb1 && s2 < (uint32_t)kList2) {
      sm.keys2[s2] = key;
      sm.idx2[s2] = pos;
    }
  }
  __syncthreads();
  const uint32_t n2 = sm.n2;
  const uint32_t need2 = need - above2;
  if (n2 <= (uint32_t)kRankDirect) {
    if ((uint32_t)t < n2) {
      const uint32_t key = sm.keys2[t];
      const int32_t pos = sm.idx2[t];
      uint32_t rank = 0;
      for (uint32_t q = 0; q < n2; ++q) {
        const uint32_t kq = sm.keys2[q];
        rank += (kq > key || (kq == key && sm.idx2[q] < pos)) ? 1u : 0u;
      }
      if (rank < need2) out[above + above2 + rank] = pos;
    }
    return;
  }
  const uint32_t prefix = (b1 << kCoarseShift) | (sb1 << kSubShift);
  if (n2 <= (uint32_t)kList2) {
    const SmemPairs cand{sm.keys2, sm.idx2, (int)n2};
    radix_select(sm.hist, sm.s, cand, need2, prefix, 32 - kSubShift, emit);
  } else {
    const SmemPairs cand{sm.cand_keys, sm.cand_idx, (int)nb};
    radix_select(sm.hist, sm.s, cand, need2, prefix, 32 - kSubShift, emit);
  }
}

// Parts per row for a cluster select kernel: the most (up to kMaxParts,
// slices of at least kMinSlice elements, at most one CTA per SM) for which
// every row's cluster can be resident at once, so the launch is a single wave.
// The cluster capacities come from the occupancy API, once per device and
// kernel (`slot` names the kernel: 0 fused decode, 1 rows).
template <class Kern>
int select_parts(Kern kern, int slot, int64_t rows, int64_t ldw, int sms, size_t smem) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int capacity[2][kMaxDevices][kMaxParts + 1];  // 0: not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
  int64_t best = 1;
  for (int P = 2; P <= kMaxParts; ++P) {
    if (ldw / P < kMinSlice || rows * P > (int64_t)sms) break;
    int cap = 0;
    if (dev >= 0) {
      std::lock_guard<std::mutex> lock(mu);
      if (capacity[slot][dev][P] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)P);
        cfg.blockDim = dim3(kSelThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)P;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
          (void)cudaGetLastError();
          n = -1;
        }
        capacity[slot][dev][P] = n > 0 ? n : -1;
      }
      cap = capacity[slot][dev][P];
    }
    if (cap >= rows) best = P;
  }
  return (int)best;
}

}  // namespace idx
