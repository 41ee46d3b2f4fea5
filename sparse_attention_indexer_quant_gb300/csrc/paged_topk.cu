// Paged decode logits + top-k (vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer":
// paged_mqa_logits followed by top_k_per_row into topk_indices_buffer), in
// launches that hand the logits over through the caller's workspace instead of
// a logits tensor:
//
//   1. zero     the scoring pass's work-item counter;
//   2. score    the persistent cp.async + tcgen05 logits kernel, taking work items
//               from the counter and writing each row's valid logits to a
//               row-major scratch that stays in L2 for these sizes;
//   3. select   one thread-block cluster of P CTAs per row, each CTA over a
//               slice of the row held in registers: every CTA builds the coarse
//               histogram of its slice (the top 12 bits of each logit's
//               order-preserving key) in shared memory; summed over the
//               cluster through distributed shared memory it gives the bin b1
//               holding the k-th largest logit and the count above it; each
//               CTAs then count b1's elements by the next 8 key bits, which
//               gives the sub-bin sb1 the same way; each thread counts its
//               elements above and in (b1, sb1), one block scan and one
//               exchange of CTA totals give every thread its output and
//               candidate slots; the elements above (b1, sb1) go straight to
//               the output and its own few elements into the cluster leader's
//               shared memory, where they are ranked by key and position.
// All three are dependent launches, so each one's start overlaps the previous
// one's tail.
//
// Workspace (device, caller-owned), 256-byte aligned pieces: the u32 work-item
// counter (zeroed per call), then f32 logits [rows][ldw], ldw = max_blocks * 64.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"
#include "topk_select.cuh"

namespace idx {
namespace {

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

struct TopkWs {
  uint32_t* items;    // work-item counter of the scoring pass
  float* logits;      // [rows][ldw]
  int64_t ldw;
  size_t zero_bytes;  // the counter
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) / 256 * 256; }

__host__ __device__ inline TopkWs ws_layout(void* base, int64_t rows, int32_t max_blocks,
                                            size_t* total) {
  const int64_t ldw = (int64_t)max_blocks * kPage;
  const size_t o_lg = 256;
  uint8_t* p = static_cast<uint8_t*>(base);
  TopkWs w;
  w.items = reinterpret_cast<uint32_t*>(p);
  w.logits = reinterpret_cast<float*>(p + o_lg);
  w.ldw = ldw;
  w.zero_bytes = 16;
  if (total) *total = o_lg + ws_align((size_t)rows * ldw * 4);
  return w;
}

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
// (key(-inf) outside [base, s1): its bin lies below the bin of any finite
// logit, so such positions are never counted above or in b1).
__device__ __forceinline__ void load_chunk_keys(const float* x, int32_t base, int32_t s1, int t,
                                                uint4 (&kv)[kSelVec]) {
#pragma unroll
  for (int u = 0; u < kSelVec; ++u) {
    const int32_t i0 = base + 4 * (u * kSelThreads + t);
    float4 v;
    if (i0 + 3 < s1) {
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

// Launched as clusters of `parts` CTAs, one cluster per row.  Every CTA of a
// cluster takes the same branches and passes the same four cluster barriers.
__global__ void __launch_bounds__(kSelThreads, 1) paged_select_kernel(const PagedArgs p, int next_n,
                                                                      int parts) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  pdl_wait();  // the scoring pass's logits
  const int64_t rows = (int64_t)p.B * next_n;
  const TopkWs ws = ws_layout(p.workspace, rows, p.max_blocks, nullptr);
  const int64_t r = blockIdx.x / parts;
  const int part = (int)cluster_ctarank();
  const int b = (int)(r / next_n), j = (int)(r % next_n);
  int64_t L = __ldg(p.context_lens + b);
  const int64_t cap = (int64_t)p.max_blocks * kPage;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  int64_t len = L - next_n + j + 1;
  len = len < 0 ? 0 : len;
  const uint32_t k = (uint32_t)p.topk;
  int32_t* out = p.out_idx + r * p.topk;
  const int t = threadIdx.x;
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
  const float* x = ws.logits + r * ws.ldw;  // 256-byte aligned; slices 16-byte aligned

  uint4 ka[kSelVec], kb[kSelVec];
  load_chunk_keys(x, s0, s1, t, ka);
  load_chunk_keys(x, s0 + kSelChunk, s1, t, kb);
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
      load_chunk_keys(x, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, s0 + (c + 1) * kSelChunk, s1, t, kb);
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
  auto coarse_masks = [&](uint32_t& gt, uint32_t& eq, bool count_sub) {
    gt = 0u;
    eq = 0u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int u = 0; u < kSelVec; ++u) {
        const uint4 v = h == 0 ? ka[u] : kb[u];
        const uint32_t e4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t bin = coarse_bin(e4[q]);
          const uint32_t bit = 1u << (16 * h + 4 * u + q);
          gt |= bin > b1 ? bit : 0u;
          if (bin == b1) {
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
      load_chunk_keys(x, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, s0 + (c + 1) * kSelChunk, s1, t, kb);
    }
    uint32_t gt, eq;
    coarse_masks(gt, eq, true);
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
      load_chunk_keys(x, s0 + c * kSelChunk, s1, t, ka);
      load_chunk_keys(x, s0 + (c + 1) * kSelChunk, s1, t, kb);
      coarse_masks(gt, eq, false);
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

// Zeroes the scoring pass's work-item counter.
__global__ void __launch_bounds__(32) paged_ws_zero_kernel(uint32_t* counter) {
  pdl_launch_dependents();
  pdl_wait();  // the previous call's kernels are done with the workspace
  if (threadIdx.x == 0) *counter = 0u;
}

// Parts per row for the select: the most (up to kMaxParts, slices of at
// least kMinSlice elements, at most one CTA per SM) for which every row's
// cluster can be resident at once, so the launch is a single wave.  The
// cluster capacities come from the occupancy API, once per device.
int select_parts(int64_t rows, int64_t ldw, int sms, size_t smem) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int capacity[kMaxDevices][kMaxParts + 1];  // 0: not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
  int64_t best = 1;
  for (int P = 2; P <= kMaxParts; ++P) {
    if (ldw / P < kMinSlice || rows * P > (int64_t)sms) break;
    int cap = 0;
    if (dev >= 0) {
      std::lock_guard<std::mutex> lock(mu);
      if (capacity[dev][P] == 0) {
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
        if (cudaOccupancyMaxActiveClusters(&n, paged_select_kernel, &cfg) != cudaSuccess) {
          (void)cudaGetLastError();
          n = -1;
        }
        capacity[dev][P] = n > 0 ? n : -1;
      }
      cap = capacity[dev][P];
    }
    if (cap >= rows) best = P;
  }
  return (int)best;
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

cudaError_t launch_paged_logits_topk(int H, int next_n, const PagedArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.B * next_n;
  const TopkWs ws = ws_layout(a.workspace, rows, a.max_blocks, nullptr);
  const size_t smem = sizeof(SelSmem);
  // the three kernels share one shared-memory carveout, so no SM has to be
  // reconfigured between them
  cudaError_t e = cudaFuncSetAttribute(paged_ws_zero_kernel,
                                       cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(paged_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(paged_select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  e = launch_dependent(paged_ws_zero_kernel, dim3(1), dim3(32), 0, stream, ws.items);
  if (e != cudaSuccess) return e;
  // scoring pass: the logits kernel writing into the workspace, work items
  // handed out by the counter
  PagedArgs s = a;
  s.logits = ws.logits;
  s.ld = ws.ldw;
  s.clean = 0;
  s.item_counter = ws.items;
  e = launch_paged_logits(H, next_n, s, stream);
  if (e != cudaSuccess) return e;
  const int parts = select_parts(rows, ws.ldw, a.sms > 0 ? a.sms : 1, smem);
  return launch_dependent_cluster(paged_select_kernel, dim3((unsigned)(rows * parts)),
                                  dim3(kSelThreads), smem, stream, (unsigned)parts, a, next_n,
                                  parts);
}

}  // namespace idx
