// Main loop shared by the paged decode kernels (unfused logits and fused
// logits + top-k): TMA producer, tcgen05 MMA issuer and TMEM epilogue.  The
// epilogue policy `Ep` decides what happens to each key's dot products.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace idx {

constexpr int kPagedThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kStages = 6;
constexpr int kMaxTilesPerCta = 64;
constexpr int kTileKeys = 128;       // MMA M: two pages
constexpr int kTileValBytes = kTileKeys * kValBytes;  // 8192

__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t used) {
  return used <= 32 ? 32 : used <= 64 ? 64 : used <= 128 ? 128 : used <= 256 ? 256 : 512;
}
__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory and tensor-memory plan for N = NH query-head columns.
template <int NH>
struct PagedLayout {
  // accumulator buffers: as many as keep a CTA within 128 TMEM columns (N = 32,
  // 64) or 256 columns (N = 128), so that 2-4 CTAs share an SM
  static constexpr int kAccBufs = NH == 32 ? 3 : 1;
  static constexpr uint32_t kSfbCol = kAccBufs * NH;     // 4 columns
  static constexpr uint32_t kSfaCol = kSfbCol + 4;       // 4 columns per accumulator
  static constexpr uint32_t kTmemCols = tmem_cols_for(kSfaCol + 4 * kAccBufs);
  static constexpr size_t kA = 0;                                   // stages x 8192 (SW64)
  static constexpr size_t kB = kA + (size_t)kStages * kTileValBytes; // NH x 64 (SW64)
  static constexpr size_t kSfRaw = kB + (size_t)NH * kValBytes;      // stages x 512
  static constexpr size_t kSfa = kSfRaw + (size_t)kStages * 512;     // stages x 512
  static constexpr size_t kSfb = kSfa + (size_t)kStages * 512;       // 512
  static constexpr size_t kW = kSfb + 512;                           // NH floats
  static constexpr size_t kBt = kW + (size_t)NH * 4;                 // 2 x 64 page ids
  static constexpr size_t kBars = align_up(kBt + 2 * kMaxTilesPerCta * 4, 16);
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs;
  static constexpr size_t kMisc = kBars + (size_t)kNumBars * 8;      // tmem base, abort
  static constexpr size_t kExtra = align_up(kMisc + 16, 1024);       // epilogue's region
};

template <int NH>
__host__ __device__ constexpr size_t paged_smem_bytes() {
  return PagedLayout<NH>::kExtra + 1024;  // + slack to align the base to 1024
}

struct PagedCta {
  int b;
  int64_t L;        // context length after validation
  int64_t k0;       // first key of this CTA's chunk
  int64_t k_end;    // end of the chunk's column range
  int n_tiles;      // tiles of 128 keys holding at least one key < L
};

__device__ __forceinline__ bool paged_cta_setup(const PagedArgs& p, PagedCta& c) {
  c.b = blockIdx.y;
  const int64_t chunk_keys = (int64_t)p.tiles_per_cta * kTileKeys;
  c.k0 = (int64_t)blockIdx.x * chunk_keys;
  c.k_end = c.k0 + chunk_keys;
  int64_t L = __ldg(p.context_lens + c.b);
  int64_t cap = (int64_t)p.max_blocks * kPage;
  if (p.logits != nullptr && p.ld < cap) cap = p.ld;
  if (L < 0 || L > cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) count_bad_input(p.errors);
    L = L < 0 ? 0 : cap;
  }
  c.L = L;
  const int64_t k1 = L < c.k_end ? L : c.k_end;
  c.n_tiles = k1 > c.k0 ? (int)((k1 - c.k0 + kTileKeys - 1) / kTileKeys) : 0;
  return c.n_tiles > 0;
}

// -inf into the columns of this CTA's chunk that no tile covers.
template <int NEXT_N>
__device__ __forceinline__ void clean_tail(const PagedArgs& p, const PagedCta& c) {
  const int64_t lo = c.k0 + (int64_t)c.n_tiles * kTileKeys;
  const int64_t hi = c.k_end < p.ld ? c.k_end : p.ld;
  for (int j = 0; j < NEXT_N; ++j) {
    float* row = p.logits + ((int64_t)c.b * NEXT_N + j) * p.ld;
    for (int64_t s = lo + threadIdx.x; s < hi; s += blockDim.x) row[s] = -INFINITY;
  }
}

// out[j] = sum_h w[j*H + h] * max(0, d[j*H + h]), h ascending.
template <int H, int NEXT_N>
__device__ __forceinline__ void weighted_relu_sum(const float* w, const float (&d)[H * NEXT_N],
                                                  float (&out)[NEXT_N]) {
#pragma unroll
  for (int j = 0; j < NEXT_N; ++j) {
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < H; h += 4) {
      const float4 ww = *reinterpret_cast<const float4*>(w + j * H + h);
      acc = fmaf(ww.x, fmaxf(d[j * H + h + 0], 0.f), acc);
      acc = fmaf(ww.y, fmaxf(d[j * H + h + 1], 0.f), acc);
      acc = fmaf(ww.z, fmaxf(d[j * H + h + 2], 0.f), acc);
      acc = fmaf(ww.w, fmaxf(d[j * H + h + 3], 0.f), acc);
    }
    out[j] = acc;
  }
}

__device__ __forceinline__ uint8_t* aligned_smem_base() {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t a = smem_u32(smem_raw);
  return smem_raw + ((1024u - (a & 1023u)) & 1023u);
}

template <int H, int NEXT_N, class Ep>
__device__ __forceinline__ void paged_cta_run(const CUtensorMap* tm_vals,
                                              const CUtensorMap* tm_scales, const PagedArgs& p,
                                              const PagedCta& c) {
  constexpr int NH = H * NEXT_N;
  using Lay = PagedLayout<NH>;
  constexpr int ACC = Lay::kAccBufs;
  static_assert(NH % 32 == 0 && NH <= 128, "N must be 32, 64 or 128");

  uint8_t* sm = aligned_smem_base();
  uint8_t* sA = sm + Lay::kA;
  uint8_t* sB = sm + Lay::kB;
  uint8_t* sSfRaw = sm + Lay::kSfRaw;
  uint8_t* sSfa = sm + Lay::kSfa;
  uint8_t* sSfb = sm + Lay::kSfb;
  float* sW = reinterpret_cast<float*>(sm + Lay::kW);
  const uint32_t bars = smem_u32(sm + Lay::kBars);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bars + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bars + 8u * (2 * kStages + ACC + a); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::kMisc + 4);
  uint8_t* extra = sm + Lay::kExtra;
  int32_t* sBt = reinterpret_cast<int32_t*>(sm + Lay::kBt);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- setup: TMEM, barriers, the sequence's query heads and weights
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Lay::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    *abort = 0;
    fence_mbar_init();
  }
  {
    // B operand: row n = j*H + h of this sequence's query heads, 64 bytes,
    // stored with the 64-byte swizzle (16-byte chunk c of row n at chunk
    // c ^ ((n >> 1) & 3)).
    const uint8_t* qv = p.q_vals + (int64_t)c.b * NH * kValBytes;
    for (int i = threadIdx.x; i < NH * 4; i += kPagedThreads) {
      const int n = i >> 2, ch = i & 3;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(qv + n * kValBytes) + ch);
      *reinterpret_cast<uint4*>(sB + n * kValBytes + ((ch ^ ((n >> 1) & 3)) << 4)) = v;
    }
    // B scale factors in the 32x16-byte atom: row n's 4 bytes at
    // 16*(n % 32) + 4*(n / 32); rows past NH are zero.
    const uint32_t* qs = reinterpret_cast<const uint32_t*>(p.q_scales) + (int64_t)c.b * NH;
    for (int n = threadIdx.x; n < 128; n += kPagedThreads) {
      const uint32_t wv = n < NH ? __ldg(qs + n) : 0u;
      *reinterpret_cast<uint32_t*>(sSfb + 16 * (n % 32) + 4 * (n / 32)) = wv;
    }
    for (int n = threadIdx.x; n < NH; n += kPagedThreads)
      sW[n] = __ldg(p.weights + (int64_t)c.b * NH + n);
    // the chunk's page ids; pages past the context are not read
    const int32_t* bt = p.block_table + (int64_t)c.b * p.max_blocks + c.k0 / kPage;
    const int n_pages = (int)((c.L - c.k0 + kPage - 1) / kPage);
    for (int i = threadIdx.x; i < 2 * c.n_tiles; i += kPagedThreads)
      sBt[i] = i < n_pages ? __ldg(bt + i) : 0;
    Ep::init(extra);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(tm_vals);
      tma_prefetch_desc(tm_scales);
      int issued = 0;
      for (int i = 0; i < c.n_tiles; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(empty_bar(s), ((i / kStages) & 1) ^ 1, abort)) {
          flag_timeout(p.errors, kTimeoutProducer);
          break;
        }
        const bool two = c.k0 + (int64_t)(2 * i + 1) * kPage < c.L;
        const int32_t id0 = sBt[2 * i];
        const int32_t id1 = sBt[2 * i + 1];
        // out-of-range ids load the TMA fill (zeros) instead of faulting
        if (id0 < 0 || id0 >= p.num_blocks) count_bad_input(p.errors);
        if (two && (id1 < 0 || id1 >= p.num_blocks)) count_bad_input(p.errors);
        const uint32_t bytes = (two ? 2u : 1u) * (kPageValBytes + 256u);
        const uint32_t fb = full_bar(s);
        mbar_arrive_expect_tx(fb, bytes);
        const uint32_t a_dst = smem_u32(sA + (size_t)s * kTileValBytes);
        const uint32_t sf_dst = smem_u32(sSfRaw + (size_t)s * 512);
        tma_load_3d(a_dst, tm_vals, 0, 0, id0, fb);
        tma_load_2d(sf_dst, tm_scales, 0, id0, fb);
        if (two) {
          tma_load_3d(a_dst + kPageValBytes, tm_vals, 0, 0, id1, fb);
          tma_load_2d(sf_dst + 256, tm_scales, 0, id1, fb);
        }
        ++issued;
      }
      // every copy this thread issued must land before the CTA can exit
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        if (!mbar_wait_drain(full_bar(i % kStages), (i / kStages) & 1))
          flag_timeout(p.errors, kTimeoutDrain);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t sfb_t = tmem + Lay::kSfbCol;
    if (lane == 0) tmem_cp_32x128b_x4(sfb_t, smem_desc(smem_u32(sSfb), 16, 128, kLayoutNone));
    __syncwarp();
    const uint64_t b_desc = smem_desc(smem_u32(sB), 16, 512, kLayoutSw64);
    int issued = 0;
    for (int i = 0; i < c.n_tiles; ++i) {
      const int s = i % kStages;
      const int a = i % ACC;
      const bool ok = mbar_wait(full_bar(s), (i / kStages) & 1, abort) &&
                      mbar_wait(tempty_bar(a), ((i / ACC) & 1) ^ 1, abort);
      if (!ok) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutMma);
        break;
      }
      tc_fence_after();
      // scale-factor atom: row l holds the 4-byte scale words of tile keys
      // l, l+32, l+64, l+96 (key k's word is word k of the two pages' scale
      // areas as loaded)
      const uint32_t* raw = reinterpret_cast<const uint32_t*>(sSfRaw + (size_t)s * 512);
      const uint4 row = make_uint4(raw[lane], raw[lane + 32], raw[lane + 64], raw[lane + 96]);
      *reinterpret_cast<uint4*>(sSfa + (size_t)s * 512 + 16 * lane) = row;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const uint32_t sfa_t = tmem + Lay::kSfaCol + 4u * a;
        tmem_cp_32x128b_x4(sfa_t,
                           smem_desc(smem_u32(sSfa + (size_t)s * 512), 16, 128, kLayoutNone));
        const uint32_t d_t = tmem + (uint32_t)(a * NH);
        const uint64_t a_desc =
            smem_desc(smem_u32(sA + (size_t)s * kTileValBytes), 16, 512, kLayoutSw64);
        // K = 0..63 uses scale bytes 0,1 of each row; K = 64..127 bytes 2,3.
        // The second half of each 64-byte row starts 32 bytes in (+2 in the
        // descriptor's 16-byte units).
        mma_mxf4(d_t, a_desc, b_desc, mxf4_idesc(NH, 0, 0), sfa_t, sfb_t, 0u);
        mma_mxf4(d_t, a_desc + 2, b_desc + 2, mxf4_idesc(NH, 2, 2), sfa_t, sfb_t, 1u);
        mma_commit(empty_bar(s));
        mma_commit(tfull_bar(a));
      }
      __syncwarp();
      ++issued;
    }
    // the last MMAs must have finished before TMEM is released
    if (lane == 0 && issued > 0) {
      const int i = issued - 1;
      if (!mbar_wait_drain(tfull_bar(i % ACC), (i / ACC) & 1))
        flag_timeout(p.errors, kTimeoutDrain);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
    const int m = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    for (int i = 0; i < c.n_tiles; ++i) {
      const int a = i % ACC;
      if (!mbar_wait(tfull_bar(a), (i / ACC) & 1, abort)) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutEpilogue);
        break;
      }
      tc_fence_after();
      float d[NH];
#pragma unroll
      for (int part = 0; part < NH / 32; ++part)
        tmem_ld32_sync(lane_addr + (uint32_t)(a * NH + 32 * part),
                       *reinterpret_cast<float(*)[32]>(&d[32 * part]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(a));
      Ep::tile(p, c, sW, extra, c.k0 + (int64_t)i * kTileKeys + m, d);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
  const bool ok = *abort == 0;
  Ep::chunk_done(p, c, extra, ok);
}

}  // namespace idx
