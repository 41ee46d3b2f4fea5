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
//      one block scan and one exchange of CTA totals give every thread its
//      output and candidate slots; the elements above go straight to the
//      output, b1's elements (a few hundred for smooth rows) with their keys
//      into the cluster leader's shared memory;
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
constexpr int kSubShift = 12;                           // sub-bin: key bits 19..12
constexpr int kSubBins = 256;
constexpr int kMaskPairs = 8;                           // chunk pairs whose masks are kept
constexpr int kList2 = kMaskPairs * kSelThreads;        // boundary sub-bin list (the mask space)
constexpr int kRankDirect = 64;                         // sub-bin lists ranked element by element
static_assert(kCoarseBins == 8 * kSelThreads, "each select thread owns eight histogram bins");

struct SelSmem {
  uint32_t bins[kCoarseBins];  // coarse histogram of this CTA's slice
  uint32_t row_bins[kCoarseBins];  // ... and of the row (sum over the cluster)
  uint32_t sub[kSubBins];      // this CTA's b1 elements by the next 8 key bits
  uint32_t mgt[kMaskPairs][kSelThreads];  // per thread and chunk pair: taken outright
  uint32_t meq[kMaskPairs][kSelThreads];  // ... and boundary candidates
  uint32_t n2;                 // candidates in the boundary sub-bin (leader)
  uint32_t hist[kRadixBins];   // radix-digit scratch (leader)
  ScanScratch s;
  uint32_t warp_gt[kSelThreads / 32], warp_eq[kSelThreads / 32];
  uint32_t cta_gt, cta_eq;     // this CTA's counts above / in b1 (read by the cluster)
  uint32_t o_base, c_base;     // this CTA's first output / candidate slot
  uint32_t all_eq;             // the row's elements in b1
  uint32_t slot;               // next output slot of the exact pass
  uint32_t cand_keys[kCandSmem];
  int32_t cand_idx[kCandSmem];
};

// Keys of x[i] for this thread's 16 positions of the chunk at `base`
// (key(-inf) at positions from s1 on, which the passes below never count).
// Four at a time when x is 16-byte aligned (base is a multiple of 4), else
// one by one.
__device__ __forceinline__ void load_chunk_keys(const float* x, bool aligned, int32_t base,
                                                int32_t s1, int t, uint4 (&kv)[kSelVec]) {
#pragma unroll
  for (int u = 0; u < kSelVec; ++u) {
    const int32_t i0 = base + 4 * (u * kSelThreads + t);
    float4 v;
    if (aligned && i0 + 3 < s1) {
      v = __ldca(reinterpret_cast<const float4*>(x + i0));
    } else {
      v.x = i0 + 0 < s1 ? __ldca(x + i0 + 0) : -INFINITY;
      v.y = i0 + 1 < s1 ? __ldca(x + i0 + 1) : -INFINITY;
      v.z = i0 + 2 < s1 ? __ldca(x + i0 + 2) : -INFINITY;
      v.w = i0 + 3 < s1 ? __ldca(x + i0 + 3) : -INFINITY;
    }
    kv[u] = make_uint4(float_key(v.x), float_key(v.y), float_key(v.z), float_key(v.w));
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
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (i0 + q < s1) atomicAdd(&bins[coarse_bin(e4[q])], 1u);
  }
}

// Exclusive prefix sums of a and b over the block's threads (ea, eb) and their
// block totals (ta, tb).  The caller syncs before the scratch is reused.
__device__ __forceinline__ void block_scan2(SelSmem& sm, uint32_t a, uint32_t b, uint32_t& ea,
                                            uint32_t& eb, uint32_t& ta, uint32_t& tb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t xa = a, xb = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t ya = __shfl_up_sync(0xFFFFFFFFu, xa, o);
    const uint32_t yb = __shfl_up_sync(0xFFFFFFFFu, xb, o);
    if (lane >= o) {
      xa += ya;
      xb += yb;
    }
  }
  if (lane == 31) {
    sm.warp_gt[warp] = xa;
    sm.warp_eq[warp] = xb;
  }
  __syncthreads();
  uint32_t pa = 0, pb = 0, sa = 0, sb = 0;
#pragma unroll
  for (int w = 0; w < kSelThreads / 32; ++w) {
    const uint32_t va = sm.warp_gt[w], vb = sm.warp_eq[w];
    pa += w < warp ? va : 0u;
    pb += w < warp ? vb : 0u;
    sa += va;
    sb += vb;
  }
  ea = pa + xa - a;
  eb = pb + xb - b;
  ta = sa;
  tb = sb;
}

// The k largest of x[0, len) -> out[0, k) (positions, -1 padded).  Called by
// every thread of every CTA of a cluster of `parts` CTAs (kSelThreads each)
// with the same arguments; every CTA takes the same branches and passes the
// same three cluster barriers.
__device__ __forceinline__ void cluster_select_row(SelSmem& sm, const float* x, int64_t len,
                                                   uint32_t k, int32_t* out, int parts) {
  const int part = (int)cluster_ctarank();
  const int t = threadIdx.x;
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
  load_chunk_keys(x, aligned, s0, s1, t, ka);
  load_chunk_keys(x, aligned, s0 + kSelChunk, s1, t, kb);
#pragma unroll
  for (int q = 0; q < 8; ++q) sm.bins[8 * t + q] = 0u;
  if (t < kSubBins) sm.sub[t] = 0u;
  if (t == 0) {
    sm.s.bin = 0;
    sm.s.above = 0;
    sm.n2 = 0;
  }
  __syncthreads();

  // ---- 1. coarse histogram of the slice, then of the row
  for (int c = 0; c < n_chunks; c += 2) {  // (past two chunks the later passes reload)
    if (c > 0) {
      load_chunk_keys(x, aligned, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, aligned, s0 + (c + 1) * kSelChunk, s1, t, kb);
    }
    hist_keys(sm.bins, ka, s0 + c * kSelChunk, s1, t);
    hist_keys(sm.bins, kb, s0 + (c + 1) * kSelChunk, s1, t);
  }
  cluster_sync_all();  // #1: every CTA's slice histogram is complete
  // thread t's bins 4095 - 8t down to 4088 - 8t, summed over the cluster (all
  // of a thread's remote loads are issued before any is used)
  uint32_t local = 0;
#pragma unroll
  for (int half = 0; half < 2; ++half) {  // 4 bins at a time
    const uint32_t my = smem_u32(&sm.bins[kCoarseBins - 8 - 8 * t + 4 * half]);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 v0 = ld_cluster_v4(cluster_map(my, 0));
    const uint4 v1 = parts > 1 ? ld_cluster_v4(cluster_map(my, 1)) : z;
    const uint4 v2 = parts > 2 ? ld_cluster_v4(cluster_map(my, 2)) : z;
    const uint4 v3 = parts > 3 ? ld_cluster_v4(cluster_map(my, 3)) : z;
    const uint4 acc = make_uint4(v0.x + v1.x + v2.x + v3.x, v0.y + v1.y + v2.y + v3.y,
                                 v0.z + v1.z + v2.z + v3.z, v0.w + v1.w + v2.w + v3.w);
    *reinterpret_cast<uint4*>(&sm.row_bins[kCoarseBins - 8 - 8 * t + 4 * half]) = acc;
    local += acc.x + acc.y + acc.z + acc.w;
  }
  const uint32_t excl = block_exclusive_scan(local, sm.s);
  if (excl < k && k <= excl + local) {
    uint32_t run = excl;
    for (int q = 0; q < 8; ++q) {  // bins 4095 - 8t - q, highest first
      const uint32_t h = sm.row_bins[kCoarseBins - 1 - 8 * t - q];
      if (run < k && k <= run + h) {
        sm.s.bin = (uint32_t)(kCoarseBins - 1 - 8 * t - q);
        sm.s.above = run;
      }
      run += h;
    }
  }
  __syncthreads();
  const uint32_t b1 = sm.s.bin;
  const uint32_t above = sm.s.above;  // the row's elements in bins above b1

  // Each thread's elements of a chunk pair are 32 mask bits: bit 16*h + 4*u + q
  // is chunk h of the pair, float4 u, lane q of it.
  auto position = [&](int c, int bit) -> int32_t {  // chunk pair starting at chunk c
    return s0 + (c + (bit >> 4)) * kSelChunk + 4 * (((bit >> 2) & 3) * kSelThreads + t) + (bit & 3);
  };
  // masks of the elements above b1 and in b1 (positions past the slice are
  // skipped: their key(-inf) padding is in b1 when the row's k-th largest
  // value is itself -inf)
  auto coarse_masks = [&](int c, uint32_t& gt, uint32_t& eq) {
    gt = 0u;
    eq = 0u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int u = 0; u < kSelVec; ++u) {
        const uint4 v = h == 0 ? ka[u] : kb[u];
        const uint32_t e4[4] = {v.x, v.y, v.z, v.w};
        const int32_t i0 = s0 + (c + h) * kSelChunk + 4 * (u * kSelThreads + t);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t bin = i0 + q < s1 ? coarse_bin(e4[q]) : 0u;
          const uint32_t bit = 1u << (16 * h + 4 * u + q);
          gt |= bin > b1 ? bit : 0u;
          eq |= (bin == b1 && i0 + q < s1) ? bit : 0u;
        }
      }
    }
  };

  // ---- 2. masks and counts of each thread's elements above b1 (taken
  //         outright) and in b1 (candidates); the masks of up to kMaskPairs
  //         chunk pairs are kept for the scatter
  const bool reload = n_chunks > 2;
  uint32_t n_gt = 0, n_eq = 0;
  for (int c = 0; c < n_chunks; c += 2) {
    if (reload) {
      load_chunk_keys(x, aligned, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, aligned, s0 + (c + 1) * kSelChunk, s1, t, kb);
    }
    uint32_t gt, eq;
    coarse_masks(c, gt, eq);
    n_gt += __popc(gt);
    n_eq += __popc(eq);
    if (c / 2 < kMaskPairs) {
      sm.mgt[c / 2][t] = gt;
      sm.meq[c / 2][t] = eq;
    }
  }

  // ---- 3. slots: block scan, then the CTAs of the row trade totals
  uint32_t eg, ee, tg, te;
  block_scan2(sm, n_gt, n_eq, eg, ee, tg, te);
  if (t == 0) {
    sm.cta_gt = tg;
    sm.cta_eq = te;
  }
  cluster_sync_all();  // #2: every CTA's totals are visible
  if (t < 32) {  // lane q reads CTA q's totals, all in flight together
    uint32_t g = 0, e = 0;
    if (t < parts) {
      g = ld_cluster_u32(cluster_map(smem_u32(&sm.cta_gt), t));
      e = ld_cluster_u32(cluster_map(smem_u32(&sm.cta_eq), t));
    }
    const uint32_t bg = __reduce_add_sync(0xFFFFFFFFu, t < part ? g : 0u);
    const uint32_t be = __reduce_add_sync(0xFFFFFFFFu, t < part ? e : 0u);
    const uint32_t ae = __reduce_add_sync(0xFFFFFFFFu, e);
    if (t == 0) {
      sm.o_base = bg;
      sm.c_base = be;
      sm.all_eq = ae;
    }
  }
  __syncthreads();

  // ---- 4. elements above b1 -> out, b1's elements (key and position) ->
  //         the leader's candidate list
  const uint32_t cand_keys0 = cluster_map(smem_u32(sm.cand_keys), 0);
  const uint32_t cand_idx0 = cluster_map(smem_u32(sm.cand_idx), 0);
  uint32_t o = sm.o_base + eg;
  uint32_t ce = sm.c_base + ee;
  for (int c = 0; c < n_chunks; c += 2) {
    uint32_t gt, eq;
    bool in_regs = !reload;  // the pair's keys are in ka / kb
    if (c / 2 < kMaskPairs) {
      gt = sm.mgt[c / 2][t];
      eq = sm.meq[c / 2][t];
    } else {
      load_chunk_keys(x, aligned, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, aligned, s0 + (c + 1) * kSelChunk, s1, t, kb);
      coarse_masks(c, gt, eq);
      in_regs = true;
    }
    for (; gt != 0u; gt &= gt - 1u) {
      if (o < above) out[o] = position(c, __ffs(gt) - 1);
      ++o;
    }
    for (; eq != 0u; eq &= eq - 1u) {
      const int bit = __ffs(eq) - 1;
      const int32_t i = position(c, bit);
      if (ce < (uint32_t)kCandSmem) {
        const uint32_t key = in_regs ? pair_key(ka, kb, bit) : float_key(__ldca(x + i));
        st_cluster_u32(cand_keys0 + 4u * ce, key);
        st_cluster_u32(cand_idx0 + 4u * ce, (uint32_t)i);
      }
      ++ce;
    }
  }
  cluster_sync_all();  // #3: the candidates are in the leader; no remote access follows
  if (part != 0) return;

  // ---- 5. the leader takes the remaining need = k - above of b1's nb
  //         elements: by their next 8 key bits (sub-bin sb1), then among
  //         sb1's few elements by rank (key, then position), or by a radix
  //         digit on the low 12 bits when there are many
  const uint32_t nb = sm.all_eq;
  const uint32_t need = k - above;
  if (t == 0) sm.slot = above;
  auto emit = [&](uint32_t, int32_t i) {
    const uint32_t s = warp_claim(&sm.slot, true);
    if (s < k) out[s] = i;
  };
  if (nb > (uint32_t)kCandSmem) {
    // more such elements than the list holds: a radix pass over the row
    __syncthreads();
    const GlobalLogits<true> row{x, 0, (int64_t)n};
    radix_select(sm.hist, sm.s, row, need, b1 << kCoarseShift, 32 - kCoarseShift, emit);
    return;
  }
  for (uint32_t i = t; i < nb; i += kSelThreads)
    atomicAdd(&sm.sub[(sm.cand_keys[i] >> kSubShift) & (kSubBins - 1)], 1u);
  __syncthreads();
  find_threshold_bin(sm.sub, kSubBins, need, sm.s);
  const uint32_t sb1 = sm.s.bin;
  const uint32_t above2 = sm.s.above;  // b1's elements above sb1
  uint32_t* const keys2 = &sm.mgt[0][0];  // sb1's elements (the masks are spent)
  int32_t* const idx2 = reinterpret_cast<int32_t*>(&sm.meq[0][0]);
  for (uint32_t i = t; i < nb; i += kSelThreads) {
    const uint32_t key = sm.cand_keys[i];
    const int32_t pos = sm.cand_idx[i];
    const uint32_t sub = (key >> kSubShift) & (kSubBins - 1);
    const uint32_t s = warp_claim(&sm.slot, sub > sb1);
    if (sub > sb1 && s < k) out[s] = pos;
    const uint32_t s2 = warp_claim(&sm.n2, sub == sb1);
    if (sub == sb1 && s2 < (uint32_t)kList2) {
      keys2[s2] = key;
      idx2[s2] = pos;
    }
  }
  __syncthreads();
  const uint32_t n2 = sm.n2;
  const uint32_t need2 = need - above2;
  if (n2 <= (uint32_t)kRankDirect) {
    if ((uint32_t)t < n2) {
      const uint32_t key = keys2[t];
      const int32_t pos = idx2[t];
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
  if (n2 <= (uint32_t)kList2) {
    const SmemPairs cand{keys2, idx2, (int)n2};
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
