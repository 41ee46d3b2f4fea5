// C ABI of libidx (declared in include/idx.h): argument validation, the
// fail-closed architecture gate, TMA tensor-map encoding and kernel dispatch.
// Nothing here allocates device memory or synchronises.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "idx.h"
#include "common.cuh"
#include "launch.h"
#include "paged_core.cuh"

namespace {
thread_local char g_detail[512] = "";
}  // namespace

namespace idx {

idx_status fail(idx_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof g_detail, fmt, ap);
  va_end(ap);
  return s;
}

idx_status ok() {
  g_detail[0] = '\0';
  return IDX_OK;
}

}  // namespace idx

namespace {

using idx::fail;
using idx::ok;

// Generations of the fused call's work-item counter: distinct per call (of the
// process), nonzero (a zero-filled workspace matches no call), below 2^40.
unsigned long long next_item_generation() {
  static std::atomic<unsigned long long> g_next{1};
  constexpr unsigned long long kMask = (1ull << (64 - idx::kItemBits)) - 1ull;
  unsigned long long g = g_next.fetch_add(1) & kMask;
  while (g == 0) g = g_next.fetch_add(1) & kMask;
  return g;
}

idx_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(IDX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- device gate, cached per device
constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 ok, 2 rejected
std::atomic<int> g_dev_sms[kMaxDevices];

idx_status current_device_ok_impl(int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(IDX_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
  int st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, sms = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return from_cuda(e, "cudaDeviceGetAttribute");
    st = idx_arch_supported(major, minor) == IDX_OK ? 1 : 2;
    g_dev_sms[dev].store(sms, std::memory_order_relaxed);
    g_dev_state[dev].store(st, std::memory_order_release);
  }
  if (st != 1)
    return fail(IDX_ERR_UNSUPPORTED_DEVICE, "device %d is not sm_103 (GB300); refusing", dev);
  if (sms_out) *sms_out = g_dev_sms[dev].load(std::memory_order_relaxed);
  return IDX_OK;
}

// ---- tensor maps through the driver entry point (no link-time libcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The prefill kernels' 2-D tensor map over the contiguous key values: 64 bytes
// x S rows, boxes of 128 rows, 64-byte swizzle (rows past S read as zeros).
idx_status key_tensor_map(const uint8_t* k_vals, int64_t S, CUtensorMap* tk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {64, (cuuint64_t)S};
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(k_vals), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IDX_ERR_CUDA, "tensor map (keys): CUresult %d", (int)r);
  return IDX_OK;
}

// Workspace of the prefill logits + top-k: per row a list length, then
// [rows][ld] candidate values and [rows][ld] positions (ld = S rounded up to 4).
struct MqaTopkWs {
  uint32_t* cnt;
  float* vals;
  int32_t* idx;
  int64_t ld;
};
size_t ws_round(size_t x) { return (x + 255) / 256 * 256; }
MqaTopkWs mqa_topk_ws(void* base, int64_t T, int64_t S, size_t* total) {
  const int64_t ld = (S + 3) / 4 * 4;
  const size_t o_cnt = 256, o_vals = o_cnt + ws_round((size_t)T * 4);
  const size_t o_idx = o_vals + ws_round((size_t)T * ld * 4);
  uint8_t* p = static_cast<uint8_t*>(base);
  MqaTopkWs w{reinterpret_cast<uint32_t*>(p + o_cnt), reinterpret_cast<float*>(p + o_vals),
              reinterpret_cast<int32_t*>(p + o_idx), ld};
  if (total) *total = o_idx + ws_round((size_t)T * ld * 4);
  return w;
}

idx_status check_paged_common(const uint8_t* q_vals, const uint8_t* q_scales, int32_t B,
                              int32_t next_n, int32_t H, const uint8_t* kcache,
                              int64_t num_blocks, int32_t page_size, const int32_t* block_table,
                              int32_t max_blocks, const int32_t* context_lens,
                              const float* weights) {
  if (B < 0 || B > 65535) return fail(IDX_ERR_INVALID_ARG, "B=%d outside [0, 65535]", B);
  if (next_n != 1 && next_n != 2) return fail(IDX_ERR_INVALID_ARG, "next_n=%d not in {1,2}", next_n);
  if (H != 32 && H != 64) return fail(IDX_ERR_INVALID_ARG, "H=%d not in {32,64}", H);
  if (page_size != 64) return fail(IDX_ERR_INVALID_ARG, "page_size=%d (only 64)", page_size);
  if (max_blocks <= 0 || max_blocks > (1 << 24))
    return fail(IDX_ERR_INVALID_ARG, "max_blocks=%d", max_blocks);
  if (num_blocks <= 0 || num_blocks > (int64_t)INT32_MAX)
    return fail(IDX_ERR_INVALID_ARG, "num_blocks=%lld", (long long)num_blocks);
  if (B == 0) return IDX_OK;
  if (!q_vals || !q_scales || !kcache || !block_table || !context_lens || !weights)
    return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q_vals, 16) || !aligned(kcache, 16) || !aligned(q_scales, 4) ||
      !aligned(weights, 16))
    return fail(IDX_ERR_INVALID_ARG,
                "alignment: q_vals/kcache/weights need 16 bytes, q_scales 4 bytes");
  return IDX_OK;
}

// Work items for the persistent paged kernels: each sequence's columns
// [0, cols) are cut into items of whole 128-key tiles, about twelve items per
// CTA over the batch (2..64 tiles each; the static round-robin assignment
// evens out sequences shorter than the block table over many small items),
// and the grid holds as many CTAs as fit on the device at once (or fewer when
// there are fewer items).
void set_paged_chunking(idx::PagedArgs& a, int64_t cols, int sms, int nh, int fixed_tiles = 0) {
  const int64_t ctas = (int64_t)sms * idx::paged_ctas_per_sm(nh);
  const int64_t tiles = (cols + 127) / 128;
  int64_t per = (tiles * a.B + 12 * ctas - 1) / (12 * ctas);
  per = per < 2 ? 2 : (per > idx::kMaxTilesPerCta ? idx::kMaxTilesPerCta : per);
  if (fixed_tiles > 0) per = fixed_tiles;
  a.sms = sms;
  a.tiles_per_cta = (int32_t)per;
  const int64_t chunks = (cols + per * 128 - 1) / (per * 128);
  a.chunks = chunks > INT32_MAX ? -1 : (int32_t)chunks;
  const int64_t items = chunks * a.B;
  a.grid = (int32_t)(items < ctas ? items : ctas);
}

}  // namespace

namespace idx {
idx_status current_device_ok(int* sms_out) { return current_device_ok_impl(sms_out); }
}  // namespace idx

extern "C" {

int idx_version(void) { return 100; }

const char* idx_status_string(idx_status s) {
  switch (s) {
    case IDX_OK: return "ok";
    case IDX_ERR_INVALID_ARG: return "invalid argument";
    case IDX_ERR_UNSUPPORTED_DEVICE: return "unsupported device (sm_103 required)";
    case IDX_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case IDX_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* idx_last_error_detail(void) { return g_detail; }

idx_status idx_arch_supported(int major, int minor) {
  return (major == 10 && minor == 3) ? IDX_OK : IDX_ERR_UNSUPPORTED_DEVICE;
}

idx_status idx_check_device(int device) {
  int major = 0, minor = 0;
  cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  if (e != cudaSuccess) return from_cuda(e, "cudaDeviceGetAttribute");
  idx_status s = idx_arch_supported(major, minor);
  if (s != IDX_OK) return fail(s, "device %d has compute capability %d.%d", device, major, minor);
  return ok();
}

idx_status idx_quant_insert(const void* k_bf16, int64_t n_tokens, int64_t k_row_stride,
                            const int64_t* slot_mapping, uint8_t* kcache, int64_t num_blocks,
                            int32_t page_size, idx_device_errors* errors, idx_stream_t stream) {
  if (n_tokens < 0 || n_tokens > (int64_t)INT32_MAX * 16)
    return fail(IDX_ERR_INVALID_ARG, "n_tokens=%lld", (long long)n_tokens);
  if (page_size != 64) return fail(IDX_ERR_INVALID_ARG, "page_size=%d (only 64)", page_size);
  if (num_blocks <= 0) return fail(IDX_ERR_INVALID_ARG, "num_blocks=%lld", (long long)num_blocks);
  if (k_row_stride < 128 || (k_row_stride % 8) != 0)
    return fail(IDX_ERR_INVALID_ARG, "k_row_stride=%lld (>= 128, multiple of 8)",
                (long long)k_row_stride);
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (n_tokens == 0) return ok();
  if (!k_bf16 || !slot_mapping || !kcache) return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k_bf16, 16) || !aligned(kcache, 16) || !aligned(slot_mapping, 8))
    return fail(IDX_ERR_INVALID_ARG, "alignment: k_bf16/kcache need 16 bytes, slots 8");
  return from_cuda(idx::launch_quant_insert(k_bf16, n_tokens, k_row_stride, slot_mapping, kcache,
                                            num_blocks, errors, (cudaStream_t)stream),
                   "quant_insert launch");
}

idx_status idx_quant_q(const void* q_bf16, int64_t rows, uint8_t* q_vals, uint8_t* q_scales,
                       idx_stream_t stream) {
  if (rows < 0 || rows > (int64_t)INT32_MAX * 16)
    return fail(IDX_ERR_INVALID_ARG, "rows=%lld", (long long)rows);
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (rows == 0) return ok();
  if (!q_bf16 || !q_vals || !q_scales) return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q_bf16, 16) || !aligned(q_vals, 4) || !aligned(q_scales, 4))
    return fail(IDX_ERR_INVALID_ARG, "alignment: q_bf16 16 bytes, outputs 4 bytes");
  return from_cuda(idx::launch_quant_q(q_bf16, rows, q_vals, q_scales, (cudaStream_t)stream),
                   "quant_q launch");
}

idx_status idx_rope_quant_q(const void* q_bf16, int64_t T, int32_t H, const int32_t* positions,
                            const float* cos_table, const float* sin_table, int32_t num_pos,
                            int32_t rot_dim, uint8_t* q_vals, uint8_t* q_scales,
                            idx_device_errors* errors, idx_stream_t stream) {
  if (T < 0 || T > (int64_t)INT32_MAX) return fail(IDX_ERR_INVALID_ARG, "T=%lld", (long long)T);
  if (H <= 0 || H > 1024) return fail(IDX_ERR_INVALID_ARG, "H=%d outside [1, 1024]", H);
  if (rot_dim < 0 || rot_dim > 128 || (rot_dim % 2) != 0)
    return fail(IDX_ERR_INVALID_ARG, "rot_dim=%d (even, 0..128)", rot_dim);
  if (num_pos < 0) return fail(IDX_ERR_INVALID_ARG, "num_pos=%d", num_pos);
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (T == 0) return ok();
  if (!q_bf16 || !q_vals || !q_scales ||
      (rot_dim > 0 && (!positions || !cos_table || !sin_table)))
    return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q_bf16, 16) || !aligned(q_vals, 4) || !aligned(q_scales, 4) ||
      !aligned(positions, 4) || !aligned(cos_table, 4) || !aligned(sin_table, 4))
    return fail(IDX_ERR_INVALID_ARG, "alignment: q_bf16 16 bytes, the rest 4 bytes");
  return from_cuda(idx::launch_rope_quant_q(q_bf16, T, H, positions, cos_table, sin_table,
                                            num_pos, rot_dim, q_vals, q_scales, errors,
                                            (cudaStream_t)stream),
                   "rope_quant_q launch");
}

idx_status idx_kpool_insert(const void* k_bf16, const float* gate, const float* ape,
                            const int64_t* slot_mapping, int64_t n, int32_t kpool,
                            uint8_t* kcache, int64_t num_blocks, int32_t page_size,
                            float* pooled, idx_device_errors* errors, idx_stream_t stream) {
  if (n < 0 || n > (int64_t)INT32_MAX) return fail(IDX_ERR_INVALID_ARG, "n=%lld", (long long)n);
  if (kpool < 1 || kpool > 128) return fail(IDX_ERR_INVALID_ARG, "kpool=%d outside [1, 128]", kpool);
  if (page_size != 64) return fail(IDX_ERR_INVALID_ARG, "page_size=%d (only 64)", page_size);
  if (num_blocks <= 0) return fail(IDX_ERR_INVALID_ARG, "num_blocks=%lld", (long long)num_blocks);
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (n < kpool) return ok();  // no pool completes in this batch
  if (!k_bf16 || !gate || !ape || !slot_mapping || !kcache)
    return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k_bf16, 16) || !aligned(kcache, 16) || !aligned(slot_mapping, 8) ||
      !aligned(gate, 4) || !aligned(ape, 4) || !aligned(pooled, 4))
    return fail(IDX_ERR_INVALID_ARG, "alignment: k_bf16/kcache 16 bytes, slots 8, floats 4");
  return from_cuda(idx::launch_kpool_insert(k_bf16, gate, ape, slot_mapping, n, kpool, kcache,
                                            num_blocks, pooled, errors, (cudaStream_t)stream),
                   "kpool_insert launch");
}

idx_status idx_paged_mqa_logits(const uint8_t* q_vals, const uint8_t* q_scales, int32_t B,
                                int32_t next_n, int32_t H, const uint8_t* kcache,
                                int64_t num_blocks, int32_t page_size,
                                const int32_t* block_table, int32_t max_blocks,
                                const int32_t* context_lens, const float* weights,
                                float* logits, int64_t ld, int clean, idx_device_errors* errors,
                                idx_stream_t stream) {
  idx_status s = check_paged_common(q_vals, q_scales, B, next_n, H, kcache, num_blocks, page_size,
                                    block_table, max_blocks, context_lens, weights);
  if (s != IDX_OK) return s;
  if (ld <= 0) return fail(IDX_ERR_INVALID_ARG, "ld=%lld", (long long)ld);
  int sms = 0;
  s = idx::current_device_ok(&sms);
  if (s != IDX_OK) return s;
  if (B == 0) return ok();
  if (!logits) return fail(IDX_ERR_INVALID_ARG, "null logits");
  idx::PagedArgs a{};
  a.kcache = kcache;
  a.q_vals = q_vals;
  a.q_scales = q_scales;
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.weights = weights;
  a.logits = logits;
  a.ld = ld;
  a.num_blocks = num_blocks;
  a.B = B;
  a.max_blocks = max_blocks;
  a.clean = clean ? 1 : 0;
  a.errors = errors;
  const int64_t cap = (int64_t)max_blocks * 64;
  set_paged_chunking(a, a.clean ? ld : (ld < cap ? ld : cap), sms, H * next_n);
  if (a.chunks <= 0) return fail(IDX_ERR_INVALID_ARG, "ld too large");
  return from_cuda(idx::launch_paged_logits(H, next_n, a, (cudaStream_t)stream),
                   "paged_mqa_logits launch");
}

idx_status idx_mqa_logits(const uint8_t* q_vals, const uint8_t* q_scales, int64_t T, int32_t H,
                          const uint8_t* k_vals, const uint8_t* k_scales, int64_t S,
                          const float* weights, const int32_t* row_start,
                          const int32_t* row_end, float* logits, int64_t ld, int clean,
                          idx_device_errors* errors, idx_stream_t stream) {
  if (T < 0 || T > (int64_t)INT32_MAX * 4) return fail(IDX_ERR_INVALID_ARG, "T=%lld", (long long)T);
  if (H != 32 && H != 64) return fail(IDX_ERR_INVALID_ARG, "H=%d not in {32,64}", H);
  if (S < 0 || S > (int64_t)INT32_MAX - 256) return fail(IDX_ERR_INVALID_ARG, "S=%lld", (long long)S);
  if (ld < S || ld <= 0) return fail(IDX_ERR_INVALID_ARG, "ld=%lld < S=%lld", (long long)ld, (long long)S);
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (T == 0 || S == 0) return ok();
  if (!q_vals || !q_scales || !k_vals || !k_scales || !weights || !row_start || !row_end || !logits)
    return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q_vals, 16) || !aligned(k_vals, 16) || !aligned(q_scales, 4) ||
      !aligned(k_scales, 4) || !aligned(weights, 4))
    return fail(IDX_ERR_INVALID_ARG, "alignment: q_vals/k_vals 16 bytes, scales/weights 4");
  CUtensorMap tk;
  if ((s = key_tensor_map(k_vals, S, &tk)) != IDX_OK) return s;
  idx::MqaArgs a{};
  a.q_vals = q_vals;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  a.weights = weights;
  a.row_start = row_start;
  a.row_end = row_end;
  a.logits = logits;
  a.T = T;
  a.S = S;
  a.ld = ld;
  a.clean = clean ? 1 : 0;
  a.errors = errors;
  return from_cuda(idx::launch_mqa_logits(tk, H, a, (cudaStream_t)stream), "mqa_logits launch");
}

size_t idx_mqa_logits_topk_workspace_bytes(int64_t T, int64_t S, int32_t k) {
  (void)k;
  if (T <= 0 || S <= 0) return 0;
  size_t total = 0;
  mqa_topk_ws(nullptr, T, S, &total);
  return total;
}

idx_status idx_mqa_logits_topk(const uint8_t* q_vals, const uint8_t* q_scales, int64_t T,
                               int32_t H, const uint8_t* k_vals, const uint8_t* k_scales,
                               int64_t S, const float* weights, const int32_t* row_start,
                               const int32_t* row_end, int32_t k, int32_t* out_idx,
                               void* workspace, size_t workspace_bytes,
                               idx_device_errors* errors, idx_stream_t stream) {
  if (T < 0 || T > (int64_t)INT32_MAX) return fail(IDX_ERR_INVALID_ARG, "T=%lld", (long long)T);
  if (H != 32 && H != 64) return fail(IDX_ERR_INVALID_ARG, "H=%d not in {32,64}", H);
  if (S < 0 || S > (int64_t)INT32_MAX - 256) return fail(IDX_ERR_INVALID_ARG, "S=%lld", (long long)S);
  if (k < 1 || k > 2048) return fail(IDX_ERR_INVALID_ARG, "k=%d outside [1, 2048]", k);
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (T == 0) return ok();
  if (!out_idx || !row_start || !row_end) return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (S == 0)  // every window is empty: every slot is -1
    return from_cuda(cudaMemsetAsync(out_idx, 0xFF, (size_t)T * k * sizeof(int32_t),
                                     (cudaStream_t)stream),
                     "mqa_logits_topk (no keys)");
  if (!q_vals || !q_scales || !k_vals || !k_scales || !weights)
    return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q_vals, 16) || !aligned(k_vals, 16) || !aligned(q_scales, 4) ||
      !aligned(k_scales, 4) || !aligned(weights, 4))
    return fail(IDX_ERR_INVALID_ARG, "alignment: q_vals/k_vals 16 bytes, scales/weights 4");
  size_t need = 0;
  const MqaTopkWs ws = mqa_topk_ws(workspace, T, S, &need);
  if (workspace_bytes < need || workspace == nullptr)
    return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(IDX_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  CUtensorMap tk;
  if ((s = key_tensor_map(k_vals, S, &tk)) != IDX_OK) return s;
  idx::MqaArgs a{};
  a.q_vals = q_vals;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  a.weights = weights;
  a.row_start = row_start;
  a.row_end = row_end;
  a.T = T;
  a.S = S;
  a.ld = S;
  a.errors = errors;
  a.topk = k;
  a.cand_vals = ws.vals;
  a.cand_idx = ws.idx;
  a.cand_cnt = ws.cnt;
  a.cand_ld = ws.ld;
  cudaError_t e = idx::launch_mqa_logits(tk, H, a, (cudaStream_t)stream);
  if (e == cudaSuccess)
    e = idx::launch_cand_topk(ws.vals, ws.idx, ws.cnt, ws.ld, T, k, out_idx, (cudaStream_t)stream);
  return from_cuda(e, "mqa_logits_topk launch");
}

idx_status idx_topk_rows(const float* logits, int64_t rows, int64_t ld, const int32_t* row_start,
                         const int32_t* row_end, int32_t k, int32_t* out_idx,
                         idx_stream_t stream) {
  if (rows < 0 || rows > (int64_t)INT32_MAX) return fail(IDX_ERR_INVALID_ARG, "rows=%lld", (long long)rows);
  if (k < 1 || k > 2048) return fail(IDX_ERR_INVALID_ARG, "k=%d outside [1, 2048]", k);
  if (ld <= 0) return fail(IDX_ERR_INVALID_ARG, "ld=%lld", (long long)ld);
  int sms = 0;
  idx_status s = idx::current_device_ok(&sms);
  if (s != IDX_OK) return s;
  if (rows == 0) return ok();
  if (!logits || !row_end || !out_idx) return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(logits, 4)) return fail(IDX_ERR_INVALID_ARG, "logits not 4-byte aligned");
  return from_cuda(idx::launch_topk_rows(logits, rows, ld, row_start, row_end, k, out_idx, sms,
                                         (cudaStream_t)stream),
                   "topk_rows launch");
}

size_t idx_paged_logits_topk_workspace_bytes(int32_t B, int32_t next_n, int32_t max_blocks,
                                             int32_t page_size, int32_t k) {
  (void)page_size;
  return idx::paged_topk_workspace_bytes(B, next_n, max_blocks, k);
}

idx_status idx_paged_logits_topk(const uint8_t* q_vals, const uint8_t* q_scales, int32_t B,
                                 int32_t next_n, int32_t H, const uint8_t* kcache,
                                 int64_t num_blocks, int32_t page_size,
                                 const int32_t* block_table, int32_t max_blocks,
                                 const int32_t* context_lens, const float* weights, int32_t k,
                                 int32_t* out_idx, void* workspace, size_t workspace_bytes,
                                 idx_device_errors* errors, idx_stream_t stream) {
  idx_status s = check_paged_common(q_vals, q_scales, B, next_n, H, kcache, num_blocks, page_size,
                                    block_table, max_blocks, context_lens, weights);
  if (s != IDX_OK) return s;
  if (k < 1 || k > 2048) return fail(IDX_ERR_INVALID_ARG, "k=%d outside [1, 2048]", k);
  s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (B == 0) return ok();
  if (!out_idx) return fail(IDX_ERR_INVALID_ARG, "null out_idx");
  if ((int64_t)B * next_n > 65535)
    return fail(IDX_ERR_INVALID_ARG, "B*next_n=%d above 65535", B * next_n);
  int sms = 0;
  if ((s = idx::current_device_ok(&sms)) != IDX_OK) return s;
  const size_t need = idx::paged_topk_workspace_bytes(B, next_n, max_blocks, k);
  if (workspace_bytes < need || workspace == nullptr)
    return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(IDX_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  idx::PagedArgs a{};
  a.kcache = kcache;
  a.q_vals = q_vals;
  a.q_scales = q_scales;
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.weights = weights;
  a.logits = nullptr;
  a.ld = 0;
  a.num_blocks = num_blocks;
  a.B = B;
  a.max_blocks = max_blocks;
  a.clean = 0;
  const int32_t item_tiles = idx::paged_topk_item_tiles(
      B, max_blocks, (int64_t)sms * idx::paged_ctas_per_sm(H * next_n));
  set_paged_chunking(a, (int64_t)max_blocks * 64, sms, H * next_n, item_tiles);
  if (a.chunks <= 0) return fail(IDX_ERR_INVALID_ARG, "max_blocks too large");
  // every claim of the call (items, plus one failing and one stale claim per
  // CTA) must fit the counter's item field
  if ((int64_t)B * a.chunks + 2 * (int64_t)a.grid >= (int64_t(1) << idx::kItemBits) - 1)
    return fail(IDX_ERR_INVALID_ARG, "B * work items per sequence = %lld too large",
                (long long)B * a.chunks);
  a.item_gen = next_item_generation();
  a.topk = k;
  a.out_idx = out_idx;
  a.workspace = workspace;
  a.errors = errors;
  return from_cuda(idx::launch_paged_logits_topk(H, next_n, a, (cudaStream_t)stream),
                   "paged_logits_topk launch");
}

size_t idx_paged_decode_step_workspace_bytes(int32_t B, int32_t next_n, int32_t H,
                                             int32_t max_blocks, int32_t page_size, int32_t k) {
  (void)page_size;
  return idx::paged_step_workspace_bytes(B, next_n, H, max_blocks, k);
}

idx_status idx_paged_decode_step(const void* k_new_bf16, const void* q_bf16, int32_t B,
                                 int32_t next_n, int32_t H, uint8_t* kcache, int64_t num_blocks,
                                 int32_t page_size, const int32_t* block_table,
                                 int32_t max_blocks, const int32_t* context_lens,
                                 const float* weights, int32_t k, int32_t* out_idx,
                                 void* workspace, size_t workspace_bytes,
                                 idx_device_errors* errors, idx_stream_t stream) {
  // the checks of the fused call, on a placeholder for the quantised query
  // (the step writes it into the workspace)
  idx_status s = check_paged_common(reinterpret_cast<const uint8_t*>(q_bf16),
                                    reinterpret_cast<const uint8_t*>(q_bf16), B, next_n, H, kcache,
                                    num_blocks, page_size, block_table, max_blocks, context_lens,
                                    weights);
  if (s != IDX_OK) return s;
  if (k < 1 || k > 2048) return fail(IDX_ERR_INVALID_ARG, "k=%d outside [1, 2048]", k);
  int sms = 0;
  if ((s = idx::current_device_ok(&sms)) != IDX_OK) return s;
  if (B == 0) return ok();
  if (!out_idx || !k_new_bf16) return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k_new_bf16, 16)) return fail(IDX_ERR_INVALID_ARG, "k_new not 16-byte aligned");
  if ((int64_t)B * next_n > 65535)
    return fail(IDX_ERR_INVALID_ARG, "B*next_n=%d above 65535", B * next_n);
  const size_t need = idx::paged_step_workspace_bytes(B, next_n, H, max_blocks, k);
  if (workspace_bytes < need || workspace == nullptr)
    return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(IDX_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  idx::PagedArgs a{};
  a.kcache = kcache;
  a.kcache_w = kcache;
  a.q_bf16 = static_cast<const uint16_t*>(q_bf16);
  a.k_new = static_cast<const uint16_t*>(k_new_bf16);
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.weights = weights;
  a.num_blocks = num_blocks;
  a.B = B;
  a.max_blocks = max_blocks;
  const int32_t item_tiles = idx::paged_topk_item_tiles(
      B, max_blocks, (int64_t)sms * idx::paged_ctas_per_sm(H * next_n));
  set_paged_chunking(a, (int64_t)max_blocks * 64, sms, H * next_n, item_tiles);
  if (a.chunks <= 0) return fail(IDX_ERR_INVALID_ARG, "max_blocks too large");
  if ((int64_t)B * a.chunks + 2 * (int64_t)a.grid >= (int64_t(1) << idx::kItemBits) - 1)
    return fail(IDX_ERR_INVALID_ARG, "B * work items per sequence = %lld too large",
                (long long)B * a.chunks);
  a.item_gen = next_item_generation();
  a.topk = k;
  a.out_idx = out_idx;
  a.workspace = workspace;
  a.errors = errors;
  return from_cuda(idx::launch_paged_decode_step(H, next_n, a, (cudaStream_t)stream),
                   "paged_decode_step launch");
}

idx_status idx_gather_k(const uint8_t* kcache, int64_t num_blocks, int32_t page_size,
                        const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                        const int64_t* out_offsets, int32_t B, uint8_t* k_vals,
                        uint8_t* k_scales, int64_t out_rows, idx_device_errors* errors,
                        idx_stream_t stream) {
  if (B < 0 || B > 65535) return fail(IDX_ERR_INVALID_ARG, "B=%d outside [0, 65535]", B);
  if (page_size != 64) return fail(IDX_ERR_INVALID_ARG, "page_size=%d (only 64)", page_size);
  if (max_blocks <= 0) return fail(IDX_ERR_INVALID_ARG, "max_blocks=%d", max_blocks);
  if (num_blocks <= 0) return fail(IDX_ERR_INVALID_ARG, "num_blocks=%lld", (long long)num_blocks);
  if (out_rows < 0) return fail(IDX_ERR_INVALID_ARG, "out_rows=%lld", (long long)out_rows);
  idx_status s = idx::current_device_ok(nullptr);
  if (s != IDX_OK) return s;
  if (B == 0) return ok();
  if (!kcache || !block_table || !seq_lens || !out_offsets || !k_vals || !k_scales)
    return fail(IDX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(kcache, 16) || !aligned(k_vals, 16) || !aligned(k_scales, 4))
    return fail(IDX_ERR_INVALID_ARG, "alignment: kcache/k_vals 16 bytes, k_scales 4");
  return from_cuda(idx::launch_gather_k(kcache, num_blocks, block_table, max_blocks, seq_lens,
                                        out_offsets, B, k_vals, k_scales, out_rows, errors,
                                        (cudaStream_t)stream),
                   "gather_k launch");
}

}  // extern "C"
