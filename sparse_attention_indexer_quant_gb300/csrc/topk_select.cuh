// Block-wide selection of the k largest fp32 values (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": top_k_per_row).
//
// Values are mapped to order-preserving uint32 keys.  A coarse histogram over
// the top 12 key bits (sign, exponent and 3 mantissa bits: 8 bins per octave
// at any magnitude) locates the bin holding the k-th largest value; everything
// in higher bins is selected outright, and the exact threshold inside the
// boundary bin is found by radix passes over the boundary elements only, on
// the 20 key bits below the bin (two 10-bit digits).  Elements equal to the final threshold key
// fill the remaining slots in arrival order, so equal values may be taken in
// any order.
//
// A source visits (key, index) pairs: `src.for_each(f)` calls f(key, idx) for
// this thread's share of the elements.  Every thread of the block must call
// the routines below together.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace idx {

constexpr int kCoarseShift = 20;
constexpr int kCoarseBins = 1 << (32 - kCoarseShift);   // 4096
constexpr int kRadixBins = 2048;

__device__ __forceinline__ uint32_t coarse_bin(uint32_t key) { return key >> kCoarseShift; }

struct ScanScratch {
  uint32_t warp_sums[32];
  uint32_t bin;
  uint32_t above;
  uint32_t count;
  uint32_t tie_count;
};

struct SelectScratch {
  uint32_t hist[kCoarseBins];
  ScanScratch s;
};

// atomicAdd(&hist[bin], 1) for every lane with pred.  The 12-bit bins spread
// a warp's 32 logits over many bins, so plain shared-memory atomics see few
// same-address conflicts; per-warp aggregation (match.any) costs more than
// it saves here.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool pred) {
  if (pred) atomicAdd(&hist[bin], 1u);
}

// Returns a distinct slot from *counter for every lane with pred (one atomic
// per warp), or 0xFFFFFFFF for lanes without.
__device__ __forceinline__ uint32_t warp_claim(uint32_t* counter, bool pred) {
  const uint32_t active = __activemask();
  const uint32_t want = __ballot_sync(active, pred);
  if (!pred) return 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(want) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(want));
  base = __shfl_sync(want, base, leader);
  return base + __popc(want & ((1u << lane) - 1u));
}

// Exclusive prefix sum of v over the threads of the block, in thread order.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, ScanScratch& sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sc.warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < nwarps ? sc.warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nwarps) sc.warp_sums[lane] = t;
  }
  __syncthreads();
  const uint32_t before = warp == 0 ? 0u : sc.warp_sums[warp - 1];
  const uint32_t r = before + x - v;
  __syncthreads();
  return r;
}

// Finds the bin b of hist[0, nbins) with count(bins > b) < need <= count(bins >= b)
// and stores b and count(bins > b) in sc.bin / sc.above.  Requires
// 1 <= need <= total count.  Warp w sums the w-th segment of bins from the
// top (its lanes on consecutive bins, so the reads are free of bank
// conflicts); the warp whose segment holds the need-th element then walks
// it from the top, 32 bins a step, with a warp scan.
__device__ __forceinline__ void find_threshold_bin(const uint32_t* hist, int nbins, uint32_t need,
                                                   ScanScratch& sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (int)(blockDim.x >> 5);
  const int seg = (nbins + nw - 1) / nw;
  const int hi = nbins - warp * seg;   // the warp's bins: [lo, hi)
  const int lo = hi - seg > 0 ? hi - seg : 0;
  uint32_t sum = 0;
  for (int i = lo + lane; i < hi; i += 32) sum += hist[i];
  sum = __reduce_add_sync(0xFFFFFFFFu, sum);
  if (lane == 0) sc.warp_sums[warp] = sum;
  __syncthreads();
  uint32_t above = 0;  // elements in the segments above this warp's
  for (int q = 0; q < warp; ++q) above += sc.warp_sums[q];
  if (above < need && need <= above + sum) {
    uint32_t run = above;
    for (int top = hi; top > lo; top -= 32) {
      const int bin = top - 1 - lane;  // lane 0 on the row's highest bin
      const uint32_t h = bin >= lo ? hist[bin] : 0u;
      uint32_t incl = h;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t hit = __ballot_sync(0xFFFFFFFFu, run + incl >= need);
      if (hit != 0u) {
        const int l = __ffs(hit) - 1;
        const uint32_t before = __shfl_sync(0xFFFFFFFFu, incl - h, l);
        if (lane == 0) {
          sc.bin = (uint32_t)(top - 1 - l);
          sc.above = run + before;
        }
        break;
      }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  __syncthreads();
}

// Emits (through emit(key, idx)) exactly `need` elements: the `need` largest
// keys among those of src whose top `known` bits equal those of `prefix`.
// The remaining low bits are resolved in one, two or three radix digits of at
// most 11 bits.  hist must hold at least kRadixBins words of scratch.
template <class Src, class Emit>
__device__ __forceinline__ void radix_select(uint32_t* hist, ScanScratch& sc, const Src& src,
                                             uint32_t need, uint32_t prefix, int known,
                                             Emit emit) {
  uint32_t mask = known == 0 ? 0u : (0xFFFFFFFFu << (32 - known));
  prefix &= mask;
  while (known < 32 && need > 0) {
    const int rest = 32 - known;
    const int width = rest <= 11 ? rest : (rest <= 22 ? (rest + 1) / 2 : 11);
    const int sh = rest - width;
    const uint32_t dm = (1u << width) - 1u;
    const int nb = 1 << width;
    for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    src.for_each([&](uint32_t key, int32_t) {
      hist_add(hist, (key >> sh) & dm, (key & mask) == prefix);
    });
    __syncthreads();
    find_threshold_bin(hist, nb, need, sc);
    const uint32_t b = sc.bin, above = sc.above;
    if (above > 0) {
      src.for_each([&](uint32_t key, int32_t idx) {
        if ((key & mask) == prefix && ((key >> sh) & dm) > b) emit(key, idx);
      });
    }
    need -= above;
    prefix |= b << sh;
    mask |= dm << sh;
    known += width;
    __syncthreads();
  }
  if (need == 0) return;
  if (threadIdx.x == 0) sc.tie_count = 0;
  __syncthreads();
  src.for_each([&](uint32_t key, int32_t idx) {
    if (key == prefix) {
      const uint32_t t = atomicAdd(&sc.tie_count, 1u);
      if (t < need) emit(key, idx);
    }
  });
  __syncthreads();
}

// Sub-bin of a boundary bin: the next 8 key bits below the coarse 12.
constexpr int kSubShift = 12;
constexpr int kSubBins = 256;
static_assert(kSubBins == 8 * 32, "one warp resolves the sub-bin, eight bins a lane");

// In warp 0 of the block: the bin b of hist[0, kSubBins) with
// count(bins > b) < need <= count(bins >= b) -> sc.bin, and count(bins > b)
// -> sc.above.  Requires 1 <= need <= the total count.
__device__ __forceinline__ void warp_find_sub_bin(const uint32_t* hist, uint32_t need,
                                                  ScanScratch& sc) {
  const int lane = threadIdx.x & 31;
  uint32_t h[8], local = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {  // bins kSubBins - 1 - 8 * lane - q, highest first
    h[q] = hist[kSubBins - 1 - 8 * lane - q];
    local += h[q];
  }
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t run = incl - local;
  if (run < need && need <= incl) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (run < need && need <= run + h[q]) {
        sc.bin = (uint32_t)(kSubBins - 1 - 8 * lane - q);
        sc.above = run;
      }
      run += h[q];
    }
  }
}

// Elements of a shared-memory array of keys with their indices.
struct SmemPairs {
  const uint32_t* keys;
  const int32_t* idx;
  int n;
  template <class F>
  __device__ __forceinline__ void for_each(F f) const {
    for (int i = threadIdx.x; i < n; i += blockDim.x) f(keys[i], idx[i]);
  }
};

// Global-memory sources load a batch of kBatch elements per thread into
// registers before handing any of them to f, so that every thread keeps
// kBatch independent loads in flight (f's atomics and stores would otherwise
// keep the next load from issuing before the previous element is done).
constexpr int kBatch = 8;

// Elements of a global-memory array of keys with their indices (read through L2).
struct GlobalPairs {
  const uint32_t* keys;
  const int32_t* idx;
  int64_t n;
  template <class F>
  __device__ __forceinline__ void for_each(F f) const {
    for (int64_t base = 0; base < n; base += (int64_t)kBatch * blockDim.x) {
      uint32_t kk[kBatch];
      int32_t ii[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t i = base + (int64_t)u * blockDim.x + threadIdx.x;
        kk[u] = i < n ? __ldcg(keys + i) : 0u;
        ii[u] = i < n ? __ldcg(idx + i) : 0;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t i = base + (int64_t)u * blockDim.x + threadIdx.x;
        if (i < n) f(kk[u], ii[u]);
      }
    }
  }
};

// fp32 logits x[lo, hi) as keys with their positions; loads through L2 (ld.cg)
// or the read-only path.
template <bool kCg>
struct GlobalLogits {
  const float* x;
  int64_t lo, hi;
  template <class F>
  __device__ __forceinline__ void for_each(F f) const {
    const int64_t n = hi - lo;
    for (int64_t base = 0; base < n; base += (int64_t)kBatch * blockDim.x) {
      float v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t i = base + (int64_t)u * blockDim.x + threadIdx.x;
        v[u] = i < n ? (kCg ? __ldcg(x + lo + i) : __ldg(x + lo + i)) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int64_t i = base + (int64_t)u * blockDim.x + threadIdx.x;
        if (i < n) f(float_key(v[u]), (int32_t)(lo + i));
      }
    }
  }
};

}  // namespace idx
