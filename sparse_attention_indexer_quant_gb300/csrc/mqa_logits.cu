// Prefill MQA logits over contiguous MXFP4 keys (vLLM API docs
// "vllm.models.glm5next.nvidia.sparse_indexer": mqa_logits; the keys come from
// the gather of the block-split cache, vLLM PR #48558 "Live validation").
//
//     logit[t, s] = sum_h w[t, h] * max(0, q^[t, h] . k^[s]),  s in [start_t, end_t)
//
// One CTA per group of G = 256 / H query tokens: the group's G*H query heads
// are the MMA's B operand (N = 256).  Keys stream through 128-key tiles from
// the union of the group's windows:
//   warp 0      producer: one 128 x 64-byte TMA box per tile (64-byte swizzle,
//               rows past S filled with zeros) and the tile's 128 key scale
//               words by 4-byte cp.async straight into the 32x16-byte
//               scale-factor layout, all completing on the stage's barrier;
//   warp 1      MMA issuer: tcgen05.cp of the tile's scale factors to one of
//               two TMEM slots (before it waits for the accumulator), then two
//               tcgen05.mma kind::mxf4 (K = 64 each) into a 128 x 256 fp32
//               accumulator;
//   warps 2-17  epilogue: TMEM lane = key; the four warps on a lane quarter
//               split the G queries; w * max(0, .) summed over heads, masked
//               to each query's window.
// The CTA order is reversed so that the largest groups (the end of a causal
// prefill) start first.
//
// With TOPK (idx_mqa_logits_topk) no logits row is written: the epilogue keeps,
// per query row, a histogram of the top 10 key bits (sign, exponent, one
// mantissa bit) of the logits it has admitted and a threshold tau, the lower
// edge of the histogram bin that holds the k-th largest admitted logit once k
// are admitted.  A logit is admitted (appended to the row's candidate list,
// value and position, with one shared-memory slot claim per warp) iff its key
// is >= tau.  Every logit >= tau is therefore in the list and at least k of
// them are, so the row's k largest are in the list; tau only grows (one warp
// per query pair recomputes it every kTkEvery tiles from a possibly stale, never
// over-counted histogram).  A second kernel selects the exact top-k of each
// list (topk.cu).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"

namespace idx {
namespace {

constexpr int kMqaThreads = 576;   // warp 0 TMA, warp 1 MMA, warps 2-17 epilogue
constexpr int kMqaStages = 4;
constexpr int kN = 256;            // query-head columns per CTA
constexpr int kEpiWarps = 16;

constexpr int kTkBins = 1024;      // candidate histogram: top 10 key bits
constexpr int kTkShift = 22;
constexpr int kTkEvery = 32;       // tiles between threshold updates (per query pair; an
                                   // update holds up its warp, and so the next tile)

// shared memory of the candidate state, per query of the group
struct TopkState {
  uint32_t hist[kTkBins];
  uint32_t cnt;                    // candidates appended
  uint32_t tau;                    // admission threshold (an order-preserving key)
  uint32_t pad[2];
};

struct MqaLayout {
  static constexpr uint32_t kAccCol = 0;            // 256 fp32 columns
  static constexpr uint32_t kSfbCol = kN;           // 8 columns (two 128-row atoms)
  static constexpr uint32_t kSfaCol = kN + 8;       // 2 x 4 columns (tiles alternate)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr size_t kA = 0;                                        // stages x 8192
  static constexpr size_t kB = kA + (size_t)kMqaStages * kTileValBytes;  // 256 x 64
  static constexpr size_t kSfa = kB + (size_t)kN * kValBytes;            // stages x 512
  static constexpr size_t kSfb = kSfa + (size_t)kMqaStages * 512;        // 2 x 512
  static constexpr size_t kW = kSfb + 1024;                              // 256 floats
  static constexpr size_t kWin = kW + (size_t)kN * 4;                    // 2 x 8 int32
  static constexpr size_t kBars = align_up(kWin + 64, 16);
  static constexpr int kNumBars = 2 * kMqaStages + 2;
  static constexpr size_t kMisc = kBars + (size_t)kNumBars * 8;
  static constexpr size_t kEnd = align_up(kMisc + 16, 1024);
};

// The threshold of query q: the lower edge of the highest bin b with
// count(bins >= b) >= k, or 0 while fewer than k are admitted.  One warp;
// lane l reads bins [32 (31 - l), 32 (32 - l)) with eight 16-byte loads (the
// counts may be stale, never over-counted: the threshold can only be low).
__device__ __forceinline__ void update_tau(TopkState& ts, uint32_t k) {
  const int lane = threadIdx.x & 31;
  uint32_t c[32];  // c[i]: bin 32 (32 - lane) - 1 - i (highest first)
  uint32_t sum = 0;
  const uint32_t base = 32u * (31u - (uint32_t)lane);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    uint4 q;
    asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
                 : "r"(smem_u32(ts.hist + base + 4 * v)));
    c[31 - 4 * v] = q.x;
    c[30 - 4 * v] = q.y;
    c[29 - 4 * v] = q.z;
    c[28 - 4 * v] = q.w;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) sum += c[i];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t run = incl - sum;
  if (run < k && k <= incl) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (run < k && k <= run + c[i]) {
        const uint32_t t = (base + 31u - (uint32_t)i) << kTkShift;
        if (t > ts.tau) ts.tau = t;
      }
      run += c[i];
    }
  }
  __syncwarp();
}

template <int H, bool TOPK>
__global__ void __launch_bounds__(kMqaThreads, 1)
    mqa_logits_kernel(const __grid_constant__ CUtensorMap tm_k, const MqaArgs p) {
  constexpr int G = kN / H;       // queries per CTA
  constexpr int GH = G / 4;       // queries per epilogue warp
  using Lay = MqaLayout;
  const int64_t n_groups = (p.T + G - 1) / G;
  const int64_t g = n_groups - 1 - (int64_t)blockIdx.x;
  const int64_t t0 = g * G;

  uint8_t* sm = aligned_smem_base();
  uint8_t* sA = sm + Lay::kA;
  uint8_t* sB = sm + Lay::kB;
  uint8_t* sSfa = sm + Lay::kSfa;
  uint8_t* sSfb = sm + Lay::kSfb;
  float* sW = reinterpret_cast<float*>(sm + Lay::kW);
  int32_t* sStart = reinterpret_cast<int32_t*>(sm + Lay::kWin);
  int32_t* sEnd = sStart + 8;
  const uint32_t bars = smem_u32(sm + Lay::kBars);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kMqaStages + s); };
  const uint32_t tfull = bars + 8u * (2 * kMqaStages);
  const uint32_t tempty = bars + 8u * (2 * kMqaStages + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::kMisc + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- windows of the group's queries (clamped to [0, S])
  if (threadIdx.x < G) {
    const int64_t t = t0 + threadIdx.x;
    int32_t st = 0, en = 0;
    if (t < p.T) {
      const int32_t st0 = __ldg(p.row_start + t), en0 = __ldg(p.row_end + t);
      st = st0 < 0 ? 0 : (st0 > p.S ? (int32_t)p.S : st0);
      en = en0 < st ? st : (en0 > p.S ? (int32_t)p.S : en0);
      if (st != st0 || en != en0) count_bad_input(p.errors);
    }
    sStart[threadIdx.x] = st;
    sEnd[threadIdx.x] = en;
  }
  TopkState* tks = reinterpret_cast<TopkState*>(sm + Lay::kEnd);  // TOPK only
  if (TOPK) {
    for (int i = threadIdx.x; i < G * (int)(sizeof(TopkState) / 4); i += kMqaThreads)
      reinterpret_cast<uint32_t*>(tks)[i] = 0u;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Lay::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMqaStages; ++s) {
      mbar_init(full_bar(s), 1 + 32);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps);
    *abort = 0;
    fence_mbar_init();
  }
  {
    // B operand: query heads (t0 + j, h) as rows n = j*H + h, 64-byte swizzle;
    // rows of queries past T are zero.
    const int64_t rows_avail = (p.T - t0) * H;
    const uint8_t* qv = p.q_vals + t0 * H * kValBytes;
    for (int i = threadIdx.x; i < kN * 4; i += kMqaThreads) {
      const int n = i >> 2, ch = i & 3;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < rows_avail) v = __ldg(reinterpret_cast<const uint4*>(qv + n * kValBytes) + ch);
      *reinterpret_cast<uint4*>(sB + n * kValBytes + ((ch ^ ((n >> 1) & 3)) << 4)) = v;
    }
    const uint32_t* qs = reinterpret_cast<const uint32_t*>(p.q_scales) + t0 * H;
    for (int n = threadIdx.x; n < kN; n += kMqaThreads) {
      const uint32_t wv = n < rows_avail ? __ldg(qs + n) : 0u;
      const int a = n >> 7, r = n & 127;
      *reinterpret_cast<uint32_t*>(sSfb + a * 512 + 16 * (r % 32) + 4 * (r / 32)) = wv;
      sW[n] = n < rows_avail ? __ldg(p.weights + t0 * H + n) : 0.f;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- key tiles covering the union of the windows
  int32_t kmin = INT32_MAX, kmax = 0;
  for (int j = 0; j < G; ++j) {
    if (sEnd[j] > sStart[j]) {
      kmin = min(kmin, sStart[j]);
      kmax = max(kmax, sEnd[j]);
    }
  }
  const int tile_lo = kmax > 0 ? kmin / kTileKeys : 0;
  const int tile_hi = kmax > 0 ? (kmax + kTileKeys - 1) / kTileKeys : 0;
  const int n_tiles = tile_hi - tile_lo;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (n_tiles > 0) {
      if (lane == 0) tma_prefetch_desc(&tm_k);
      const uint32_t* ksc = reinterpret_cast<const uint32_t*>(p.k_scales);
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kMqaStages;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_bar(s), ((i / kMqaStages) & 1) ^ 1, abort))) {
          if (lane == 0) flag_timeout(p.errors, kTimeoutProducer);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(full_bar(s), kTileValBytes);
          tma_load_2d(smem_u32(sA + (size_t)s * kTileValBytes), &tm_k, 0,
                      (tile_lo + i) * kTileKeys, full_bar(s));
        }
        const uint32_t dst = smem_u32(sSfa + (size_t)s * 512);
        const int64_t k0 = (int64_t)(tile_lo + i) * kTileKeys + lane;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          // keys past S (zero values from the TMA fill) take the last key's scales
          const int64_t kk = k0 + 32 * u < p.S ? k0 + 32 * u : p.S - 1;
          cp_async_4(dst + 16 * lane + 4 * u, ksc + kk, pol);
        }
        cp_async_arrive_noinc(full_bar(s));
        ++issued;
      }
      cp_async_wait_all();
      if (lane == 0)
        for (int i = issued > kMqaStages ? issued - kMqaStages : 0; i < issued; ++i)
          if (!mbar_wait_drain(full_bar(i % kMqaStages), (i / kMqaStages) & 1))
            flag_timeout(p.errors, kTimeoutDrain);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t sfb_t = tmem + Lay::kSfbCol;
    const uint32_t sfa_t = tmem + Lay::kSfaCol;
    if (lane == 0 && n_tiles > 0) {
      tmem_cp_32x128b_x4(sfb_t, smem_desc(smem_u32(sSfb), 16, 128, kLayoutNone));
      tmem_cp_32x128b_x4(sfb_t + 4, smem_desc(smem_u32(sSfb + 512), 16, 128, kLayoutNone));
    }
    __syncwarp();
    const uint64_t b_desc = smem_desc(smem_u32(sB), 16, 512, kLayoutSw64);
    int issued = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % kMqaStages;
      if (!mbar_wait(full_bar(s), (i / kMqaStages) & 1, abort)) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutMma);
        break;
      }
      fence_proxy_async_smem();
      __syncwarp();
      const uint32_t sfa_i = sfa_t + 4u * (uint32_t)(i & 1);
      if (lane == 0)
        tmem_cp_32x128b_x4(sfa_i, smem_desc(smem_u32(sSfa + (size_t)s * 512), 16, 128, kLayoutNone));
      if (!mbar_wait(tempty, (i & 1) ^ 1, abort)) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutMma);
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint64_t a_desc =
            smem_desc(smem_u32(sA + (size_t)s * kTileValBytes), 16, 512, kLayoutSw64);
        mma_mxf4(tmem + Lay::kAccCol, a_desc, b_desc, mxf4_idesc(kN, 0, 0), sfa_i, sfb_t, 0u);
        mma_mxf4(tmem + Lay::kAccCol, a_desc + 2, b_desc + 2, mxf4_idesc(kN, 2, 2), sfa_i, sfb_t,
                 1u);
        mma_commit(empty_bar(s));
        mma_commit(tfull);
      }
      __syncwarp();
      ++issued;
    }
    if (lane == 0 && issued > 0 && !mbar_wait_drain(tfull, (issued - 1) & 1))
      flag_timeout(p.errors, kTimeoutDrain);
  } else {
    // ---------------------------------------------------------- epilogue
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int half = e / 4;                 // which quarter of the group's queries
    const int m = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    int32_t st[GH], en[GH];
#pragma unroll
    for (int j = 0; j < GH; ++j) {
      st[j] = sStart[half * GH + j];
      en[j] = sEnd[half * GH + j];
    }
    // the warp's queries' logits rows, and the keys inside every one of their
    // windows: a tile wholly in there stores without per-query tests
    float* rows_p[GH];
    int32_t in_lo = 0, in_hi = 0x7FFFFFFF;
    const bool all_rows = t0 + half * GH + GH <= p.T;
#pragma unroll
    for (int j = 0; j < GH; ++j) {
      const int64_t t = t0 + half * GH + j;
      rows_p[j] = p.logits + (t < p.T ? t : 0) * p.ld;
      in_lo = st[j] > in_lo ? st[j] : in_lo;
      in_hi = en[j] < in_hi ? en[j] : in_hi;
    }
    for (int i = 0; i < n_tiles; ++i) {
      if (!mbar_wait(tfull, i & 1, abort)) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutEpilogue);
        break;
      }
      tc_fence_after();
      float d[GH * H];
#pragma unroll
      for (int part = 0; part < GH * H / 32; ++part)
        tmem_ld32(lane_addr + Lay::kAccCol + (uint32_t)(half * GH * H + 32 * part),
                  *reinterpret_cast<float(*)[32]>(&d[32 * part]));
      tmem_wait_ld();
      tmem_take(d);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      const int64_t key = (int64_t)(tile_lo + i) * kTileKeys + m;
      float logit[GH];
      weighted_relu_sum<H, GH>(sW + half * GH * H, d, logit);
      const int32_t k_tile = (tile_lo + i) * kTileKeys;
      if (!TOPK && all_rows && k_tile >= in_lo && k_tile + kTileKeys <= in_hi) {
#pragma unroll
        for (int j = 0; j < GH; ++j) rows_p[j][k_tile + m] = logit[j];
        continue;
      }
#pragma unroll
      for (int j = 0; j < GH; ++j) {
        const int64_t t = t0 + half * GH + j;
        if (t >= p.T) break;
        if (TOPK) {
          // admit the logit if it reaches the row's threshold: one slot claim
          // per warp (the warp's 32 keys belong to the same query)
          TopkState& ts = tks[half * GH + j];
          const uint32_t kk = float_key(logit[j]);
          const bool take = key >= st[j] && key < en[j] && kk >= *(volatile uint32_t*)&ts.tau;
          const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, take);
          if (ballot != 0u) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(&ts.cnt, (uint32_t)__popc(ballot));
            base = __shfl_sync(0xFFFFFFFFu, base, 0);
            if (take) {
              const int64_t slot = t * p.cand_ld + base + __popc(ballot & ((1u << lane) - 1u));
              p.cand_vals[slot] = logit[j];
              p.cand_idx[slot] = (int32_t)(key - st[j]);
              // (one atomic per lane: grouping the warp's equal bins with a
              // match instruction first was slower)
              atomicAdd(&ts.hist[kk >> kTkShift], 1u);
            }
          }
        } else {
          float* row = p.logits + t * p.ld;
          if (key >= st[j] && key < en[j])
            row[key] = logit[j];
          else if (p.clean && key < p.S)
            row[key] = -INFINITY;
        }
      }
      // one warp of the query pair raises the thresholds every kTkEvery
      // tiles, the four lane quarters' warps taking turns
      if (TOPK && (i % kTkEvery) == kTkEvery - 1 && ((i / kTkEvery) & 3) == quarter) {
#pragma unroll
        for (int j = 0; j < GH; ++j) update_tau(tks[half * GH + j], (uint32_t)p.topk);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
  if (TOPK) {
    if (threadIdx.x < G && t0 + threadIdx.x < p.T) p.cand_cnt[t0 + threadIdx.x] = tks[threadIdx.x].cnt;
    return;
  }
  if (p.clean) {
    // -inf for the columns of [0, S) that no tile covers
    const int64_t lo_end = (int64_t)tile_lo * kTileKeys;
    const int64_t hi_begin = (int64_t)tile_hi * kTileKeys;
    for (int j = 0; j < G; ++j) {
      const int64_t t = t0 + j;
      if (t >= p.T) break;
      float* row = p.logits + t * p.ld;
      const int64_t lo1 = n_tiles > 0 ? lo_end : p.S;
      for (int64_t s = threadIdx.x; s < lo1 && s < p.S; s += kMqaThreads) row[s] = -INFINITY;
      if (n_tiles > 0)
        for (int64_t s = hi_begin + threadIdx.x; s < p.S; s += kMqaThreads) row[s] = -INFINITY;
    }
  }
}

template <int H, bool TOPK>
cudaError_t launch_h(const CUtensorMap& tm, const MqaArgs& a, cudaStream_t stream) {
  const size_t smem = MqaLayout::kEnd + (TOPK ? (kN / H) * sizeof(TopkState) : 0) + 1024;
  auto kern = mqa_logits_kernel<H, TOPK>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int G = kN / H;
  const int64_t groups = (a.T + G - 1) / G;
  kern<<<(unsigned)groups, kMqaThreads, smem, stream>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mqa_logits(const CUtensorMap& tm_kvals, int H, const MqaArgs& a,
                              cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const bool topk = a.cand_vals != nullptr;
  if (H == 32) return topk ? launch_h<32, true>(tm_kvals, a, stream) : launch_h<32, false>(tm_kvals, a, stream);
  if (H == 64) return topk ? launch_h<64, true>(tm_kvals, a, stream) : launch_h<64, false>(tm_kvals, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace idx
