// Exact top-k of one fp32 row by a thread-block cluster (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": top_k_per_row into
// topk_indices_buffer; rows of at most k elements list all of them, then -1).
//
// The P CTAs of a cluster each take a slice of the row, held in registers:
//   1. every CTA builds the coarse histogram of its slice (the top 12 bits of
//      each value's order-preserving key) in shared memory; summed over the
//      cluster through distributed shared memory it gives the bin b1 holding
//      the k-th largest value and the count above it;
//   2. the CTAs count b1's elements by the next 8 key bits, which gives the
//      sub-bin sb1 the same way;
//   3. each thread classifies its elements as above (b1, sb1) or in it (bit
//      masks), one block scan and one exchange of CTA totals give every thread
//      its output and candidate slots; the elements above go straight to the
//      output, the few in (b1, sb1) into the cluster leader's shared memory;
//   4. the leader ranks the candidates by key and position (a radix pass on the
//      low 12 bits when there are many).
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
static_assert(kCoarseBins == 8 * kSelThreads, "each select thread owns eight histogram bins");

struct SelSmem {
  uint32_t bins[kCoarseBins];  // coarse histogram of this CTA's slice
  uint32_t row_bins[kCoarseBins];  // ... and of the row (sum over the cluster)
  uint32_t sub[kSubBins];      // this CTA's b1 elements by the next 8 key bits
  uint32_t mgt[kMaskPairs][kSelThreads];  // per thread and chunk pair: taken outright
  uint32_t meq[kMaskPairs][kSelThreads];  // ... and boundary candidates
  uint32_t sb1, above2;        // the boundary sub-bin, b1's elements above it
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
// same four cluster barriers.
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
    sm.sb1 = 0;
    sm.above2 = 0;
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
  const uint32_t above = sm.s.above;

  // Each thread's elements of a chunk pair are 32 mask bits: bit 16*h + 4*u + q
  // is chunk h of the pair, float4 u, lane q of it.
  auto position = [&](int c, int bit) -> int32_t {  // chunk pair starting at chunk c
    return s0 + (c + (bit >> 4)) * kSelChunk + 4 * (((bit >> 2) & 3) * kSelThreads + t) + (bit & 3);
  };
  // masks of the elements above b1 and in b1; b1's elements also counted by
  // their next 8 key bits
  // (positions past the slice are skipped: their key(-inf) padding is in b1
  // when the row's k-th largest value is itself -inf)
  auto coarse_masks = [&](int c, uint32_t& gt, uint32_t& eq, bool count_sub) {
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
          if (bin == b1 && i0 + q < s1) {
            eq |= bit;
            if (count_sub) atomicAdd(&sm.sub[(e4[q] >> kSubShift) & (kSubBins - 1)], 1u);
          }
        }
      }
    }
  };

  // ---- 2. the boundary sub-bin sb1: b1's elements by key bits 19..12,
  //         summed over the cluster; the coarse masks are kept (up to
  //         kMaskPairs chunk pairs) for the passes below
  const bool reload = n_chunks > 2;
  for (int c = 0; c < n_chunks; c += 2) {
    if (reload) {
      load_chunk_keys(x, aligned, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, aligned, s0 + (c + 1) * kSelChunk, s1, t, kb);
    }
    uint32_t gt, eq;
    coarse_masks(c, gt, eq, true);
    if (c / 2 < kMaskPairs) {
      sm.mgt[c / 2][t] = gt;
      sm.meq[c / 2][t] = eq;
    }
  }
  cluster_sync_all();  // #2: every CTA's sub-bin counts are complete
  {
    uint32_t sv = 0;  // thread t < 256 holds sub-bin 255 - t (highest first)
    if (t < kSubBins) {
      const uint32_t my = smem_u32(&sm.sub[kSubBins - 1 - t]);
      const uint32_t v0 = ld_cluster_u32(cluster_map(my, 0));
      const uint32_t v1 = parts > 1 ? ld_cluster_u32(cluster_map(my, 1)) : 0u;
      const uint32_t v2 = parts > 2 ? ld_cluster_u32(cluster_map(my, 2)) : 0u;
      const uint32_t v3 = parts > 3 ? ld_cluster_u32(cluster_map(my, 3)) : 0u;
      sv = v0 + v1 + v2 + v3;
    }
    const uint32_t need1 = k - above;
    const uint32_t ex = block_exclusive_scan(sv, sm.s);
    if (t < kSubBins && ex < need1 && need1 <= ex + sv) {
      sm.sb1 = (uint32_t)(kSubBins - 1 - t);
      sm.above2 = ex;
    }
    __syncthreads();
  }
  const uint32_t sb1 = sm.sb1;
  const uint32_t taken = above + sm.above2;  // elements above (b1, sb1)

  // ---- 3a. final masks: an element is taken outright when its (bin, sub-bin)
  //         is above (b1, sb1), a candidate when equal to it; only b1's few
  //         elements need their sub-bin, read back from the logits
  auto final_masks = [&](int c, uint32_t& gt, uint32_t& eq) {
    if (c / 2 < kMaskPairs) {
      gt = sm.mgt[c / 2][t];
      eq = sm.meq[c / 2][t];
    } else {
      load_chunk_keys(x, aligned, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, aligned, s0 + (c + 1) * kSelChunk, s1, t, kb);
      coarse_masks(c, gt, eq, false);
    }
    uint32_t in = 0u;
    for (uint32_t m = eq; m != 0u; m &= m - 1u) {
      const int bit = __ffs(m) - 1;
      const uint32_t sub = (float_key(__ldca(x + position(c, bit))) >> kSubShift) & (kSubBins - 1);
      if (sub > sb1) gt |= 1u << bit;
      else if (sub == sb1) in |= 1u << bit;
    }
    eq = in;
  };
  uint32_t n_gt = 0, n_eq = 0;
  for (int c = 0; c < n_chunks; c += 2) {
    uint32_t gt, eq;
    final_masks(c, gt, eq);
    n_gt += __popc(gt);
    n_eq += __popc(eq);
    if (c / 2 < kMaskPairs) {
      sm.mgt[c / 2][t] = gt;
      sm.meq[c / 2][t] = eq;
    }
  }

  // ---- 3b. slots: block scan, then the CTAs of the row trade totals
  uint32_t eg, ee, tg, te;
  block_scan2(sm, n_gt, n_eq, eg, ee, tg, te);
  if (t == 0) {
    sm.cta_gt = tg;
    sm.cta_eq = te;
  }
  cluster_sync_all();  // #3: every CTA's totals are visible
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

  // ---- 3c. elements above (b1, sb1) -> out, its elements -> the leader's list
  const uint32_t cand_keys0 = cluster_map(smem_u32(sm.cand_keys), 0);
  const uint32_t cand_idx0 = cluster_map(smem_u32(sm.cand_idx), 0);
  uint32_t o = sm.o_base + eg;
  uint32_t ce = sm.c_base + ee;
  for (int c = 0; c < n_chunks; c += 2) {
    uint32_t gt, eq;
    if (c / 2 < kMaskPairs) {
      gt = sm.mgt[c / 2][t];
      eq = sm.meq[c / 2][t];
    } else {
      final_masks(c, gt, eq);
    }
    for (; gt != 0u; gt &= gt - 1u) {
      if (o < taken) out[o] = position(c, __ffs(gt) - 1);
      ++o;
    }
    for (; eq != 0u; eq &= eq - 1u) {
      const int32_t i = position(c, __ffs(eq) - 1);
      if (ce < (uint32_t)kCandSmem) {
        st_cluster_u32(cand_keys0 + 4u * ce, float_key(__ldca(x + i)));
        st_cluster_u32(cand_idx0 + 4u * ce, (uint32_t)i);
      }
      ++ce;
    }
  }
  cluster_sync_all();  // #4: the candidates are in the leader; no remote access follows
  if (part != 0) return;

  // ---- 4. the leader takes the remaining k - taken of the candidates, which
  //         share their top 20 key bits: by rank (key, then position) when
  //         there are few, else by a radix digit on the low 12 bits
  const uint32_t nb = sm.all_eq;
  const uint32_t need = k - taken;
  if (nb <= (uint32_t)kSelThreads) {
    if ((uint32_t)t < nb) {
      const uint32_t key = sm.cand_keys[t];
      const int32_t pos = sm.cand_idx[t];
      uint32_t rank = 0;
      for (uint32_t q = 0; q < nb; ++q) {
        const uint32_t kq = sm.cand_keys[q];
        rank += (kq > key || (kq == key && sm.cand_idx[q] < pos)) ? 1u : 0u;
      }
      if (rank < need) out[taken + rank] = pos;
    }
    return;
  }
  if (t == 0) sm.slot = taken;
  __syncthreads();
  auto emit = [&](uint32_t, int32_t i) {
    const uint32_t s = warp_claim(&sm.slot, true);
    if (s < k) out[s] = i;
  };
  const uint32_t prefix = (b1 << kCoarseShift) | (sb1 << kSubShift);
  if (nb <= (uint32_t)kCandSmem) {
    const SmemPairs cand{sm.cand_keys, sm.cand_idx, (int)nb};
    radix_select(sm.hist, sm.s, cand, need, prefix, 32 - kSubShift, emit);
  } else {
    // more such elements than the list holds: a radix pass over the row
    const GlobalLogits<true> row{x, 0, (int64_t)n};
    radix_select(sm.hist, sm.s, row, need, prefix, 32 - kSubShift, emit);
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
