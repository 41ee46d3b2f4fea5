// Block-wide radix selection of the k largest fp32 values (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": top_k_per_row).
//
// Values are mapped to order-preserving uint32 keys and the threshold key is
// found digit by digit (11, 11 and 10 bits, most significant first) from
// shared-memory histograms.  At every digit the elements whose digit is above
// the threshold digit are certainly selected and are emitted at once; the
// rest of the search continues among the elements that share the threshold
// prefix.  Elements equal to the final threshold key fill the remaining slots
// in arrival order, so equal values may be taken in any order.
//
// A source visits (key, index) pairs: `src.for_each(f)` calls f(key, idx) for
// this thread's share of the elements.  Every thread of the block must call
// the routines below together.
#pragma once

#include "common.cuh"

namespace idx {

constexpr int kRadixBins = 2048;

struct SelectScratch {
  uint32_t hist[kRadixBins];
  uint32_t warp_sums[32];
  uint32_t bin;
  uint32_t above;
  uint32_t out_count;
  uint32_t tie_count;
  uint32_t aux;
};

__device__ __forceinline__ constexpr int digit_shift(int d) { return d == 0 ? 21 : d == 1 ? 10 : 0; }
__device__ __forceinline__ constexpr uint32_t digit_mask(int d) { return d == 2 ? 0x3FFu : 0x7FFu; }

// Exclusive prefix sum of v over the threads of the block, in thread order.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, SelectScratch& sc) {
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
    if (lane < nwarps) sc.warp_sums[lane] = t;  // inclusive totals
  }
  __syncthreads();
  const uint32_t before = warp == 0 ? 0u : sc.warp_sums[warp - 1];
  const uint32_t r = before + x - v;
  __syncthreads();
  return r;
}

// Finds the bin b of hist[0, nbins) with count(bins > b) < need <= count(bins >= b)
// and stores b and count(bins > b) in sc.bin / sc.above.  Requires
// 1 <= need <= total count.
__device__ __forceinline__ void find_threshold_bin(SelectScratch& sc, int nbins, uint32_t need) {
  const int nt = blockDim.x;
  const int per = (nbins + nt - 1) / nt;
  // thread t owns bins (hi - per, hi] counted from the top
  const int hi = nbins - 1 - threadIdx.x * per;
  uint32_t local = 0;
  for (int q = 0; q < per; ++q) {
    const int bin = hi - q;
    if (bin >= 0) local += sc.hist[bin];
  }
  const uint32_t excl = block_exclusive_scan(local, sc);
  if (excl < need && need <= excl + local) {
    uint32_t run = excl;
    for (int q = 0; q < per; ++q) {
      const int bin = hi - q;
      if (bin < 0) break;
      const uint32_t h = sc.hist[bin];
      if (run + h >= need) {
        sc.bin = (uint32_t)bin;
        sc.above = run;
        break;
      }
      run += h;
    }
  }
  __syncthreads();
}

// Histogram of digit d over the elements matching (key & mask) == prefix.
template <class Src>
__device__ __forceinline__ void digit_histogram(SelectScratch& sc, const Src& src, int d,
                                                uint32_t prefix, uint32_t mask) {
  const int nb = (int)digit_mask(d) + 1;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) sc.hist[i] = 0;
  __syncthreads();
  const int sh = digit_shift(d);
  const uint32_t dm = digit_mask(d);
  src.for_each([&](uint32_t key, int32_t) {
    if ((key & mask) == prefix) atomicAdd(&sc.hist[(key >> sh) & dm], 1u);
  });
  __syncthreads();
}

// Emits (through emit(key, idx)) exactly `need` elements: the `need` largest
// keys among those matching (key & mask) == prefix, searching from digit d0.
template <class Src, class Emit>
__device__ __forceinline__ void radix_select(SelectScratch& sc, const Src& src, uint32_t need,
                                             int d0, uint32_t prefix, uint32_t mask,
                                             Emit emit) {
  for (int d = d0; d < 3 && need > 0; ++d) {
    digit_histogram(sc, src, d, prefix, mask);
    find_threshold_bin(sc, (int)digit_mask(d) + 1, need);
    const uint32_t b = sc.bin, above = sc.above;
    const int sh = digit_shift(d);
    const uint32_t dm = digit_mask(d);
    if (above > 0) {
      src.for_each([&](uint32_t key, int32_t idx) {
        if ((key & mask) == prefix && ((key >> sh) & dm) > b) emit(key, idx);
      });
    }
    need -= above;
    prefix |= b << sh;
    mask |= dm << sh;
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

}  // namespace idx
