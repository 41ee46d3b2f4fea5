// Persistent main loop shared by the paged decode kernels (unfused logits and
// the scoring pass of logits + top-k): each CTA loops over work items
// (sequence b, chunk of tiles_per_item 128-key tiles) with four warp roles:
//   warps 0-3   epilogue: one thread per key (TMEM lane) loads its row of D and
//               hands the next_n*H dot products to the epilogue policy `Ep`
//               (at N = 128, warps 0-7, each with one query's 64 columns);
//   warp 4      MMA issuer: tcgen05.cp of the tile's key scale factors to TMEM
//               and two tcgen05.mma kind::mxf4 block-scaled MMAs (K = 64 each)
//               giving D[key, j*H + h] in TMEM (fp32);
//   warp 5      item loader (the warp numbers of these roles shift by four at
//               N = 128): picks the next item (a fixed chunk-major
//               round-robin, or a global counter when `dynamic`), stages the
//               sequence's query heads (the MMA's B operand, N = next_n*H), their
//               scale factors, weights and the chunk's page ids into one of two
//               buffers, and publishes the item descriptor;
//   warps 6-7   copy producers: per tile, the two pages' value rows (16-byte
//               cp.async into the 64-byte-swizzled K-major layout the MMA reads)
//               and their scale words (4-byte cp.async straight into the
//               32x16-byte scale-factor layout), into a ring of stages.
// Each producer thread ends a tile with cp.async.mbarrier.arrive, so the
// stage's barrier completes when the 64 threads' copies have landed, without
// the producers waiting on them; the MMA thread fences the generic-proxy
// writes to the async proxy after its wait.  Page ids outside the cache are skipped (and counted) instead of
// being read.  The stage ring, the accumulator ring and the two item buffers
// run across items, so the copy stream does not drain between items.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "mxfp4_encode.cuh"

namespace idx {

constexpr int kCopyThreads = 64;
constexpr int kTileKeys = 128;        // MMA M: two pages
constexpr int kTileValBytes = kTileKeys * kValBytes;  // 8192
constexpr int kMaxTilesPerCta = 64;   // tiles per work item
constexpr int kClCache = 1024;        // context lengths kept in shared memory

__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t used) {
  return used <= 32 ? 32 : used <= 64 ? 64 : used <= 128 ? 128 : used <= 256 ? 256 : 512;
}
__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Occupancy plan per N = next_n * H.  Streaming random pages reaches HBM rate
// only with about 200 KB of copies in flight per SM (loaded latency is several
// microseconds), so each shape gets as many stage buffers as its CTAs-per-SM
// allow: N = 32 three CTAs of 7 stages, N = 64 two of 10, N = 128 two of 10
// (with one accumulator each: the two CTAs' MMAs and epilogues interleave on
// the SM, which streams faster than one CTA of 20 stages with three).
__host__ __device__ constexpr int paged_ctas_per_sm(int nh) { return nh == 32 ? 3 : 2; }
__host__ __device__ constexpr int paged_stages(int nh) { return nh == 32 ? 7 : 10; }
// Epilogue warps: four (one per TMEM lane quarter) take all N columns of their
// keys; at N = 128 eight, a pair per lane quarter, each taking one query's 64
// heads, so that each SM sub-partition has four warps forming sums.  Then the
// MMA warp, the item loader and two copy producers.
__host__ __device__ constexpr int paged_epi_warps(int nh) { return nh == 128 ? 8 : 4; }
__host__ __device__ constexpr int paged_threads(int nh) { return 32 * (paged_epi_warps(nh) + 4); }

struct ItemDesc {
  int64_t L;        // context length after validation
  int64_t k0;       // first key of the item
  int64_t k_end;    // end of the item's column range
  int32_t b;        // sequence
  int32_t n_tiles;  // tiles holding a key < L; -1 ends the item stream
};

// Shared-memory and tensor-memory plan for N = NH query-head columns.
template <int NH>
struct PagedLayout {
  static constexpr int kStages = paged_stages(NH);
  // accumulators: as many as fit the TMEM share of a CTA (512 columns per SM:
  // 128 for each of three N = 32 CTAs, 256 for each of two N = 64 or N = 128
  // CTAs): three at N = 32 and 64, so that three tiles' MMAs can be in flight
  // while the epilogue reads a fourth's; one at N = 128, where the SM's other
  // CTA covers the wait
  static constexpr int kAccBufs = NH == 128 ? 1 : 3;
  static constexpr uint32_t kSfbCol = kAccBufs * NH;        // 2 x 4 columns
  static constexpr uint32_t kSfaCol = kSfbCol + 8;          // 4 columns per accumulator
  static constexpr uint32_t kTmemCols = tmem_cols_for(kSfaCol + 4 * kAccBufs);
  static constexpr size_t kA = 0;                                      // stages x 8192 (SW64)
  static constexpr size_t kB = kA + (size_t)kStages * kTileValBytes;   // 2 x NH x 64 (SW64)
  static constexpr size_t kSfa = kB + 2 * (size_t)NH * kValBytes;      // stages x 512
  static constexpr size_t kSfb = kSfa + (size_t)kStages * 512;         // 2 x 512
  static constexpr size_t kW = kSfb + 2 * 512;                         // 2 x NH floats
  static constexpr size_t kBt = kW + 2 * (size_t)NH * 4;               // 2 x 128 page ids
  static constexpr size_t kCl = kBt + 2 * 2 * kMaxTilesPerCta * 4;     // context lengths
  static constexpr size_t kItem = align_up(kCl + kClCache * 4, 16);
  static constexpr size_t kBars = kItem + 2 * sizeof(ItemDesc);
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 4;
  static constexpr size_t kMisc = kBars + (size_t)kNumBars * 8;        // tmem base, abort
  static constexpr size_t kExtra = align_up(kMisc + 16, 1024);         // epilogue's region
};

template <int NH>
__host__ __device__ constexpr size_t paged_smem_bytes() {
  return PagedLayout<NH>::kExtra + 1024;  // + slack to align the base to 1024
}

// Keys of a sequence the kernels read: its context length clamped to the
// block table (and to the logits row when there is one).
__device__ __forceinline__ int64_t len_cap(const PagedArgs& p) {
  int64_t cap = (int64_t)p.max_blocks * kPage;
  if (p.logits != nullptr && p.ld < cap) cap = p.ld;
  return cap;
}

// Work item w in chunk-major order: w = c * B + b.
__device__ __forceinline__ ItemDesc paged_item(const PagedArgs& p, int64_t w, const int32_t* cl,
                                               bool count_errors) {
  ItemDesc it;
  it.b = (int32_t)(w % p.B);
  const int64_t c = w / p.B;
  const int64_t C = (int64_t)p.tiles_per_cta * kTileKeys;
  it.k0 = c * C;
  it.k_end = it.k0 + C;
  int64_t L = it.b < kClCache ? cl[it.b] : __ldg(p.context_lens + it.b);
  const int64_t cap = len_cap(p);
  if (L < 0 || L > cap) {
    if (count_errors && c == 0) count_bad_input(p.errors);
    L = L < 0 ? 0 : cap;
  }
  it.L = L;
  const int64_t k1 = L < it.k_end ? L : it.k_end;
  it.n_tiles = k1 > it.k0 ? (int32_t)((k1 - it.k0 + kTileKeys - 1) / kTileKeys) : 0;
  return it;
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

// Work-item counter of the dynamic schedule, kept in a workspace that calls
// reuse: the top 40 bits hold the call's generation, the low kItemBits the
// items handed out.  A call's first claim finds an older generation's value
// (or whatever a fresh workspace held) and installs its own, so the counter
// needs no clearing between calls.  Returns the call's next item index;
// 0xFFFFFFFF (past every item) if the installing race does not settle.
constexpr int kItemBits = 24;
__device__ __forceinline__ uint32_t claim_item(unsigned long long* ctr, unsigned long long gen,
                                               idx_device_errors* errors) {
  constexpr unsigned long long kCount = (1ull << kItemBits) - 1ull;
  unsigned long long v = atomicAdd(ctr, 1ull);
  if ((v >> kItemBits) == gen) return (uint32_t)(v & kCount);
  unsigned long long cur = v + 1ull;  // the stale value, as this thread left it
  for (int i = 0; i < (1 << 16); ++i) {
    const unsigned long long prev = atomicCAS(ctr, cur, (gen << kItemBits) | 1ull);
    if (prev == cur) return 0u;  // installed, with item 0 claimed
    if ((prev >> kItemBits) == gen) return (uint32_t)(atomicAdd(ctr, 1ull) & kCount);
    cur = prev;  // other claims moved the stale value on
  }
  flag_timeout(errors, kTimeoutProducer);
  return 0xFFFFFFFFu;
}

// Installs this call's generation in the counter ahead of the first claims
// (one thread of the grid, while its warp has nothing else to do yet), so
// that the claims find it in place and take one atomic add each; claims that
// come first install it themselves.
__device__ __forceinline__ void install_generation(unsigned long long* ctr, unsigned long long gen) {
  unsigned long long cur = atomicAdd(ctr, 0ull);
  for (int i = 0; i < 64 && (cur >> kItemBits) != gen; ++i) {
    const unsigned long long prev = atomicCAS(ctr, cur, gen << kItemBits);
    if (prev == cur) return;
    cur = prev;
  }
}

// The decode step's preparation (a scoring pass that also does the step's
// insert and query quantisation), spread over the grid's item loaders: the
// work is cut into chunks of kStepChunkPasses warp passes (two 128-element
// vectors a pass: the sequence's NEXT_N * H query heads, then its NEXT_N new
// keys), B * step_chunks() in all, claimed from a generation-tagged counter
// in the workspace by each loader before its first item.  A loader that
// finishes a chunk of sequence b adds one to b's generation-tagged done count;
// before staging an item of b a loader waits, for at most kWaitLimitNs, until
// that count reaches b's chunk total.  Every chunk is claimed by a running
// CTA that waits on nothing while doing it, so the waits need no
// co-residency of the grid.  A new key whose position is outside the block
// table or whose page id is outside the cache is skipped and counted.
constexpr int kStepChunkPasses = 2;

template <int H, int NEXT_N>
__host__ __device__ constexpr int step_chunks() {
  return ((NEXT_N * H + NEXT_N + 1) / 2 + kStepChunkPasses - 1) / kStepChunkPasses;
}

// Chunk ci of sequence b, by the whole loader warp (the encoder's shuffles
// need converged warps: a 16-lane group past the end encodes zeros and stores
// nothing).  All of a lane's loads are issued before any is encoded.
template <int H, int NEXT_N>
__device__ __forceinline__ void step_prepare_chunk(const PagedArgs& p, int32_t b, int ci,
                                                   int lane) {
  constexpr int kQ = NEXT_N * H;
  constexpr int kB = kStepChunkPasses;
  const int part = lane & 15;
  const int64_t cap = (int64_t)p.max_blocks * kPage;
  int64_t L = __ldg(p.context_lens + b);
  L = L < 0 ? 0 : (L > cap ? cap : L);  // (an over-long context is counted by the loop)
  uint4 raw[kB];
  int32_t id[kB];
#pragma unroll
  for (int u = 0; u < kB; ++u) {
    const int v = 2 * (ci * kB + u) + (lane >> 4);
    raw[u] = make_uint4(0, 0, 0, 0);
    id[u] = -1;
    if (v < kQ) {
      raw[u] = __ldg(reinterpret_cast<const uint4*>(p.q_bf16 + ((int64_t)b * kQ + v) * kHeadDim) +
                     part);
    } else if (v < kQ + NEXT_N) {
      const int j = v - kQ;
      const int64_t pos = L - NEXT_N + j;
      if (pos >= 0) {
        id[u] = __ldg(p.block_table + (int64_t)b * p.max_blocks + pos / kPage);
        raw[u] = __ldg(reinterpret_cast<const uint4*>(p.k_new + ((int64_t)b * NEXT_N + j) * kHeadDim) +
                       part);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kB; ++u) {
    const int v = 2 * (ci * kB + u) + (lane >> 4);
    uint8_t* vdst = nullptr;
    uint8_t* sdst = nullptr;
    if (v < kQ) {
      const int64_t row = (int64_t)b * kQ + v;
      vdst = p.q_vals_w + row * kValBytes;
      sdst = p.q_scales_w + row * kScaleBytes;
    } else if (v < kQ + NEXT_N) {
      const int64_t pos = L - NEXT_N + (v - kQ);
      if (pos >= 0 && id[u] >= 0 && id[u] < p.num_blocks) {
        uint8_t* pg = p.kcache_w + (int64_t)id[u] * kPageBytes;
        vdst = pg + (pos % kPage) * kValBytes;
        sdst = pg + kPageValBytes + (pos % kPage) * kScaleBytes;
      } else if (part == 0) {
        count_bad_input(p.errors);
      }
    }
    uint32_t sw;
    const uint32_t packed = encode8(raw[u], &sw);
    if (vdst != nullptr) {
      reinterpret_cast<uint32_t*>(vdst)[part] = packed;
      if (part == 0) *reinterpret_cast<uint32_t*>(sdst) = sw;
    }
  }
}

// The decode step: by the loader warp, before it stages an item of sequence
// b, a wait until every chunk of b is done (returns false, raising *abort,
// if the wait gives up).
template <int H, int NEXT_N>
__device__ __forceinline__ bool step_wait_sequence(const PagedArgs& p, int32_t b, int lane,
                                                   volatile int* abort) {
  constexpr unsigned long long kCount = (1ull << kItemBits) - 1ull;
  uint32_t ok = 1;
  if (lane == 0) {
    const unsigned long long* st = p.seq_state + b;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
      unsigned long long c;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(c) : "l"(st) : "memory");
      if ((c >> kItemBits) == p.item_gen && (c & kCount) >= (unsigned long long)step_chunks<H, NEXT_N>())
        break;
      if ((it & 15u) == 15u && (*abort || global_timer_ns() - t0 > kWaitLimitNs)) {
        flag_timeout(p.errors, kTimeoutProducer);
        *abort = 1;
        ok = 0;
        break;
      }
    }
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  return ok != 0;
}

// Barrier among the epilogue warps only, returning pred ORed (AND = false:
// ANDed) over the epilogue threads, so that every epilogue warp takes the
// same decision.
template <int EPI_THREADS, bool AND = false>
__device__ __forceinline__ bool epilogue_sync_reduce(bool pred) {
  uint32_t r;
  if (AND)
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)pred), "n"(EPI_THREADS) : "memory");
  else
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)pred), "n"(EPI_THREADS) : "memory");
  return r != 0;
}

template <int H, int NEXT_N, class Ep, bool STEP = false>
__device__ __forceinline__ void paged_persistent_run(const PagedArgs& p, const uint8_t* kcache,
                                                     bool dynamic, bool pass_empty,
                                                     unsigned long long* item_counter) {
  constexpr int NH = H * NEXT_N;
  using Lay = PagedLayout<NH>;
  constexpr int ACC = Lay::kAccBufs;
  constexpr int kStages = Lay::kStages;
  constexpr int EPI = paged_epi_warps(NH);   // warps [0, EPI): epilogue
  constexpr int kMmaWarp = EPI, kLoaderWarp = EPI + 1, kCopyWarp0 = EPI + 2;
  constexpr int kThreads = paged_threads(NH);
  static_assert(NH % 32 == 0 && NH <= 128, "N must be 32, 64 or 128");
  static_assert(Lay::kTmemCols * paged_ctas_per_sm(NH) <= 512, "TMEM over-subscribed");

  uint8_t* sm = aligned_smem_base();
  uint8_t* sA = sm + Lay::kA;
  uint8_t* sB = sm + Lay::kB;
  uint8_t* sSfa = sm + Lay::kSfa;
  uint8_t* sSfb = sm + Lay::kSfb;
  float* sW = reinterpret_cast<float*>(sm + Lay::kW);
  int32_t* sBt = reinterpret_cast<int32_t*>(sm + Lay::kBt);
  int32_t* sCl = reinterpret_cast<int32_t*>(sm + Lay::kCl);
  ItemDesc* sItem = reinterpret_cast<ItemDesc*>(sm + Lay::kItem);
  const uint32_t bars = smem_u32(sm + Lay::kBars);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bars + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bars + 8u * (2 * kStages + ACC + a); };
  auto qfull_bar = [&](int q) { return bars + 8u * (2 * kStages + 2 * ACC + q); };
  auto qempty_bar = [&](int q) { return bars + 8u * (2 * kStages + 2 * ACC + 2 + q); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::kMisc + 4);
  uint8_t* extra = sm + Lay::kExtra;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), Lay::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), kCopyThreads);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), EPI);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(qfull_bar(q), 1);
      mbar_init(qempty_bar(q), 1 + EPI);  // the MMA commit + the epilogue warps
    }
    *abort = 0;
    fence_mbar_init();
  }
  // up to here only this CTA's shared and tensor memory was touched: with a
  // dependent launch that overlaps the previous kernel's tail; every input is
  // read after the wait
  if (p.wait_first) {
    pdl_wait();
    pdl_launch_dependents();
  } else {
    pdl_launch_dependents();
    pdl_wait();
  }
  // The item loader's operands (warp 5), read into registers before they are
  // staged, all loads of a lane in flight together:
  //   B operand: row r = j*H + h of the sequence's query heads, 64 bytes,
  //   stored with the 64-byte swizzle (16-byte chunk c of row r at chunk
  //   c ^ ((r >> 1) & 3)); its scale factors in the 32x16-byte atom (row r's
  //   4 bytes at 16*(r % 32) + 4*(r / 32), rows past NH zero); the weights;
  //   the page ids of the item's first n_tiles tiles (entries past the
  //   sequence's last page are never used: the producers skip those pages).
  constexpr int kQv = NH * 4 / 32;
  uint4 qv_r[kQv];
  uint32_t sf_r[4];
  float w_r[NH / 32];
  int32_t id_r[4];
  auto load_operands = [&](int32_t b, int64_t k0, int32_t n_tiles) {
    const uint4* qv = reinterpret_cast<const uint4*>(p.q_vals + (int64_t)b * NH * kValBytes);
    // (in the decode step this launch's preparation chunks wrote them: loads
    // through L2)
#pragma unroll
    for (int u = 0; u < kQv; ++u) qv_r[u] = STEP ? __ldcg(qv + lane + 32 * u) : __ldg(qv + lane + 32 * u);
    const uint32_t* qs = reinterpret_cast<const uint32_t*>(p.q_scales) + (int64_t)b * NH;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      sf_r[u] = lane + 32 * u < NH ? (STEP ? __ldcg(qs + lane + 32 * u) : __ldg(qs + lane + 32 * u))
                                   : 0u;
#pragma unroll
    for (int u = 0; u < NH / 32; ++u) w_r[u] = __ldg(p.weights + (int64_t)b * NH + lane + 32 * u);
    const int32_t* bt = p.block_table + (int64_t)b * p.max_blocks + k0 / kPage;
    const int64_t in_row = (int64_t)p.max_blocks - k0 / kPage;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = lane + 32 * u;
      id_r[u] = i < 2 * n_tiles && i < in_row ? __ldg(bt + i) : 0;
    }
  };
  // The loader's first item is this CTA's own index: its operands are read
  // now, for all of the item's tiles, while the block fills the context-length
  // cache that decides how many of them are used.
  // (not in the decode step: there the operands exist once the item's
  // sequence has been prepared)
  const bool preloaded =
      !STEP && warp == kLoaderWarp && (int64_t)blockIdx.x < (int64_t)p.B * p.chunks;
  if (preloaded)
    load_operands((int32_t)(blockIdx.x % p.B),
                  (int64_t)(blockIdx.x / p.B) * p.tiles_per_cta * kTileKeys, p.tiles_per_cta);
  for (int i = threadIdx.x; i < p.B && i < kClCache; i += kThreads)
    sCl[i] = __ldg(p.context_lens + i);
  Ep::init(extra);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t n_items = (int64_t)p.B * p.chunks;
  if (dynamic && blockIdx.x == 0 && threadIdx.x == 0) install_generation(item_counter, p.item_gen);

  if (warp == kLoaderWarp) {
    // ---------------------------------------------------------- item loader
    constexpr uint32_t kAll = 0xFFFFFFFFu;
    if (STEP) {
      // the decode step's preparation chunks, claimed until none is left
      constexpr uint32_t kCh = (uint32_t)step_chunks<H, NEXT_N>();
      const uint32_t total = (uint32_t)p.B * kCh;
      while (true) {
        uint32_t c = 0;
        if (lane == 0) c = claim_item(p.prep_counter, p.item_gen, p.errors);
        c = __shfl_sync(kAll, c, 0);
        if (c >= total) break;
        step_prepare_chunk<H, NEXT_N>(p, (int32_t)(c / kCh), (int)(c % kCh), lane);
        __threadfence();  // the chunk's stores before the count that publishes them
        __syncwarp();
        if (lane == 0) (void)claim_item(p.seq_state + c / kCh, p.item_gen, p.errors);
      }
    }
    int n = 0;
    int64_t w = (int64_t)blockIdx.x - (int64_t)gridDim.x;
    bool first = true;
    while (true) {
      ItemDesc it;
      it.n_tiles = -1;
      // the next item with work (with pass_empty: the next item); the first
      // item of a CTA is its own index, later ones come from the counter
      while (true) {
        if (dynamic && !first) {
          uint32_t t = 0;
          if (lane == 0) t = claim_item(item_counter, p.item_gen, p.errors);
          w = (int64_t)gridDim.x + (int64_t)__shfl_sync(kAll, t, 0);
        } else {
          w += gridDim.x;
        }
        first = false;
        if (w >= n_items) {
          it.n_tiles = -1;
          break;
        }
        it = paged_item(p, w, sCl, lane == 0);
        if (it.n_tiles > 0 || pass_empty) break;
      }
      // the decode step: the sequence's query heads and new keys first (an
      // item stream that gives up there ends here for every role)
      if (STEP && it.n_tiles > 0 && !step_wait_sequence<H, NEXT_N>(p, it.b, lane, abort))
        it.n_tiles = -1;
      if (it.n_tiles > 0 && !(preloaded && w == (int64_t)blockIdx.x))
        load_operands(it.b, it.k0, it.n_tiles);
      const int qb = n & 1;
      if (!__all_sync(kAll, mbar_wait(qempty_bar(qb), ((n >> 1) & 1) ^ 1, abort))) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutProducer);
        break;
      }
      if (it.n_tiles > 0) {
        uint8_t* b_dst = sB + (size_t)qb * NH * kValBytes;
#pragma unroll
        for (int u = 0; u < kQv; ++u) {
          const int i = lane + 32 * u;
          const int r = i >> 2, ch = i & 3;
          *reinterpret_cast<uint4*>(b_dst + r * kValBytes + ((ch ^ ((r >> 1) & 3)) << 4)) = qv_r[u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)  // row lane + 32u
          *reinterpret_cast<uint32_t*>(sSfb + qb * 512 + 16 * lane + 4 * u) = sf_r[u];
#pragma unroll
        for (int u = 0; u < NH / 32; ++u) sW[qb * NH + lane + 32 * u] = w_r[u];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = lane + 32 * u;
          if (i < 2 * it.n_tiles) sBt[qb * 2 * kMaxTilesPerCta + i] = id_r[u];
        }
      }
      if (lane == 0) sItem[qb] = it;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(qfull_bar(qb));
      ++n;
      if (it.n_tiles < 0) break;
    }
  } else if (warp >= kCopyWarp0) {
    // ---------------------------------------------------------- copy producers
    const int pt = threadIdx.x - kCopyWarp0 * 32;  // 0..63
    // the cache is streamed once per call: its lines go first, so that the
    // logits written meanwhile stay in L2 for whatever reads them next
    const uint64_t pol = l2_evict_first_policy();
    int issued = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int qb = n & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(qfull_bar(qb), (n >> 1) & 1, abort))) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutProducer);
        break;
      }
      const ItemDesc it = sItem[qb];
      if (it.n_tiles < 0) break;
      const int32_t* ids = sBt + qb * 2 * kMaxTilesPerCta;
      for (int t = 0; t < it.n_tiles; ++t) {
        const int s = issued % kStages;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(empty_bar(s), ((issued / kStages) & 1) ^ 1, abort));
        if (!ok) {
          if (lane == 0) flag_timeout(p.errors, kTimeoutProducer);
          break;
        }
        const bool two = it.k0 + (int64_t)(2 * t + 1) * kPage < it.L;
        const int32_t id0 = ids[2 * t], id1 = ids[2 * t + 1];
        const bool ok0 = id0 >= 0 && id0 < p.num_blocks;
        const bool ok1 = two && id1 >= 0 && id1 < p.num_blocks;
        if (pt == 0) {
          if (!ok0) count_bad_input(p.errors);
          if (two && !ok1) count_bad_input(p.errors);
        }
        const uint8_t* pg0 = kcache + (int64_t)(ok0 ? id0 : 0) * kPageBytes;
        const uint8_t* pg1 = kcache + (int64_t)(ok1 ? id1 : 0) * kPageBytes;
        const uint32_t a_dst = smem_u32(sA + (size_t)s * kTileValBytes);
        // values: 512 chunks of 16 bytes; chunk q is key q/4, 16-byte column q%4
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int q = pt + kCopyThreads * u;
          const int key = q >> 2, c = q & 3;
          const bool second = key >= kPage;
          if (second ? ok1 : ok0) {
            const uint8_t* src = (second ? pg1 : pg0) + (key & (kPage - 1)) * kValBytes + c * 16;
            cp_async_16(a_dst + key * kValBytes + ((c ^ ((key >> 1) & 3)) << 4), src, pol);
          }
        }
        // scales: key k's 4-byte word to 16*(k % 32) + 4*(k / 32) of the atom
        const uint32_t sf_dst = smem_u32(sSfa + (size_t)s * 512);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int key = pt + kCopyThreads * u;
          const bool second = key >= kPage;
          if (second ? ok1 : ok0) {
            const uint8_t* src =
                (second ? pg1 : pg0) + kPageValBytes + (key & (kPage - 1)) * kScaleBytes;
            cp_async_4(sf_dst + 16 * (key % 32) + 4 * (key / 32), src, pol);
          }
        }
        // the stage fills once all 64 threads' copies have landed; the thread
        // holds no tile back, so its waits never depend on its own copies
        cp_async_arrive_noinc(full_bar(s));
        ++issued;
      }
    }
    // nothing may still be writing shared memory when the CTA exits
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    int tiles = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int qb = n & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(qfull_bar(qb), (n >> 1) & 1, abort))) {
        if (lane == 0) flag_timeout(p.errors, kTimeoutMma);
        break;
      }
      const ItemDesc it = sItem[qb];
      if (it.n_tiles < 0) break;
      tc_fence_after();
      const uint32_t sfb_t = tmem + Lay::kSfbCol + 4u * qb;
      if (lane == 0 && it.n_tiles > 0)
        tmem_cp_32x128b_x4(sfb_t, smem_desc(smem_u32(sSfb + qb * 512), 16, 128, kLayoutNone));
      __syncwarp();
      const uint64_t b_desc =
          smem_desc(smem_u32(sB + (size_t)qb * NH * kValBytes), 16, 512, kLayoutSw64);
      for (int t = 0; t < it.n_tiles; ++t) {
        const int s = tiles % kStages;
        const int a = tiles % ACC;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(full_bar(s), (tiles / kStages) & 1, abort) &&
                                         mbar_wait(tempty_bar(a), ((tiles / ACC) & 1) ^ 1, abort));
        if (!ok) {
          if (lane == 0) flag_timeout(p.errors, kTimeoutMma);
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          // the stage was written by cp.async (generic proxy); the MMA and
          // tcgen05.cp read it through the async proxy
          fence_proxy_async_smem();
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
        ++tiles;
      }
      // the item's B buffer is free once its MMAs are done
      if (lane == 0) mma_commit(qempty_bar(qb));
      __syncwarp();
    }
    // the last MMAs must have finished before TMEM is released
    if (lane == 0 && tiles > 0) {
      const int i = tiles - 1;
      if (!mbar_wait_drain(tfull_bar(i % ACC), (i / ACC) & 1))
        flag_timeout(p.errors, kTimeoutDrain);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    // warp w: TMEM lanes [32 (w % 4), +32) (its keys) and columns
    // [NC (w / 4), +NC) (queries j0 .. j0 + NJ - 1 of the item's NEXT_N)
    constexpr int NC = NH * 4 / EPI;
    constexpr int NJ = NEXT_N * 4 / EPI;
    static_assert(NC == NJ * H, "an epilogue warp takes whole queries");
    const int quarter = warp & 3;
    const int cpart = warp >> 2;
    const int j0 = cpart * NJ;
    const int m = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(cpart * NC);
    int tiles = 0;
    for (int n = 0;; ++n) {
      const int qb = n & 1;
      // every epilogue warp takes the same branches: the item's wait is
      // agreed over the epilogue warps, a wait that gives up raises *abort,
      // the item loop still runs to its end (later waits return at once), and
      // the epilogue warps leave together, on one agreed decision (two warps
      // that read *abort apart would otherwise part at the barrier below)
      const bool have = epilogue_sync_reduce<EPI * 32, true>(
          mbar_wait(qfull_bar(qb), (n >> 1) & 1, abort));
      const ItemDesc it = sItem[qb];
      const bool stop = !have || it.n_tiles < 0;
      const int n_tiles = stop ? 0 : it.n_tiles;
      const float* w = sW + qb * NH + j0 * H;
      for (int t = 0; t < n_tiles; ++t) {
        const int a = tiles % ACC;
        ++tiles;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(tfull_bar(a), ((tiles - 1) / ACC) & 1, abort))) {
          if (lane == 0) flag_timeout(p.errors, kTimeoutEpilogue);
          continue;
        }
        tc_fence_after();
        float d[NC];
#pragma unroll
        for (int part = 0; part < NC / 32; ++part)
          tmem_ld32_sync(lane_addr + (uint32_t)(a * NH + 32 * part),
                         *reinterpret_cast<float(*)[32]>(&d[32 * part]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(a));
        Ep::template tile<NJ>(p, it, w, extra, it.k0 + (int64_t)t * kTileKeys + m, d, j0);
      }
      if (epilogue_sync_reduce<EPI * 32>(stop || *abort)) break;
      Ep::item_done(p, it, extra, EPI * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty_bar(qb));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

}  // namespace idx
