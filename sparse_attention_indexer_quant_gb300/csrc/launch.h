// Internal launchers behind the C ABI (argument checking happens in api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "idx.h"

namespace idx {

// Records a detail message for idx_last_error_detail() (this host thread) and
// returns s; ok() clears it and returns IDX_OK.
idx_status fail(idx_status s, const char* fmt, ...);
idx_status ok();
// The fail-closed device gate of every entry point, applied to the current
// device (cached per device); *sms_out gets its SM count.
idx_status current_device_ok(int* sms_out);

cudaError_t launch_quant_insert(const void* k, int64_t n_tokens, int64_t row_stride,
                                const int64_t* slots, uint8_t* cache, int64_t num_blocks,
                                idx_device_errors* errors, cudaStream_t stream);

cudaError_t launch_quant_q(const void* q, int64_t rows, uint8_t* vals, uint8_t* scales,
                           cudaStream_t stream);

cudaError_t launch_rope_quant_q(const void* q, int64_t T, int32_t H, const int32_t* positions,
                                const float* cs, const float* sn, int32_t num_pos,
                                int32_t rot_dim, uint8_t* vals, uint8_t* scales,
                                idx_device_errors* errors, cudaStream_t stream);

cudaError_t launch_kpool_insert(const void* k, const float* gate, const float* ape,
                                const int64_t* slots, int64_t n, int32_t kpool, uint8_t* cache,
                                int64_t num_blocks, float* pooled, idx_device_errors* errors,
                                cudaStream_t stream);

// Paged decode (persistent kernels reading the cache with cp.async).
struct PagedArgs {
  const uint8_t* kcache;
  const uint8_t* q_vals;
  const uint8_t* q_scales;
  const int32_t* block_table;
  const int32_t* context_lens;
  const float* weights;
  float* logits;          // unfused: [rows, ld]
  int64_t ld;
  int64_t num_blocks;
  int32_t B;
  int32_t max_blocks;
  int32_t clean;
  int32_t tiles_per_cta;  // keys per work item = 128 * tiles_per_cta
  int32_t chunks;         // work items per sequence
  int32_t grid;           // persistent CTAs
  int32_t sms;            // SMs of the device
  int32_t topk;           // fused only
  int32_t* out_idx;       // fused only: [rows, topk]
  void* workspace;        // fused only
  unsigned long long* item_counter;  // generation-tagged work-item counter: dynamic
                                     // scheduling; null: static
  unsigned long long item_gen;       // this call's generation (nonzero, < 2^40)
  int32_t wait_first;                // wait for the previous kernel before letting the
                                     // next one start (its early code may read the inputs)
  idx_device_errors* errors;
  // decode step only (the scoring pass quantises each sequence's query heads
  // and inserts its new keys before any of its items is scored)
  const uint16_t* q_bf16;            // [rows, H, 128] bf16
  const uint16_t* k_new;             // [rows, 128] bf16: row b*next_n + j at position
                                     // L_b - next_n + j of sequence b
  uint8_t* q_vals_w;                 // == q_vals, written by the scoring pass
  uint8_t* q_scales_w;               // == q_scales
  uint8_t* kcache_w;                 // == kcache
  unsigned long long* seq_state;     // [B] generation-tagged count of a sequence's
                                     // preparation chunks done; non-null selects the
                                     // decode step
  unsigned long long* prep_counter;  // generation-tagged claim counter of the chunks
};

cudaError_t launch_paged_logits(int H, int next_n, const PagedArgs& a, cudaStream_t stream);

// Launches kern<<<grid, block, smem, stream>>>(args...) with programmatic stream
// serialization: the kernel may be scheduled while the previous kernel in the
// stream is finishing, and must call pdl_wait() before reading its inputs.
template <class... KArgs, class... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// launch_dependent with thread-block clusters of cluster_x CTAs along x.
template <class... KArgs, class... Args>
cudaError_t launch_dependent_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

cudaError_t launch_paged_logits_topk(int H, int next_n, const PagedArgs& a, cudaStream_t stream);
size_t paged_topk_workspace_bytes(int32_t B, int32_t next_n, int32_t max_blocks, int32_t k);
// the decode step: the fused call's workspace plus the quantised query heads
size_t paged_step_workspace_bytes(int32_t B, int32_t next_n, int32_t H, int32_t max_blocks,
                                  int32_t k);
cudaError_t launch_paged_decode_step(int H, int next_n, const PagedArgs& a, cudaStream_t stream);
// 128-key tiles per work item of the fused scoring pass
int32_t paged_topk_item_tiles(int32_t B, int32_t max_blocks, int64_t ctas);

// Prefill: tensor maps over contiguous keys (values 2-D: 64 B x S, 64-byte
// swizzle; scales 2-D: 512 B x ceil(S/128) tiles).
struct MqaArgs {
  const uint8_t* q_vals;
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const float* weights;
  const int32_t* row_start;
  const int32_t* row_end;
  float* logits;
  int64_t T;
  int64_t S;
  int64_t ld;
  int32_t clean;
  idx_device_errors* errors;
  // logits + top-k: candidate lists instead of logits rows
  int32_t topk;
  float* cand_vals;       // [T][cand_ld] admitted logits
  int32_t* cand_idx;      // [T][cand_ld] their positions in the row's window
  uint32_t* cand_cnt;     // [T] list lengths
  int64_t cand_ld;
};
cudaError_t launch_mqa_logits(const CUtensorMap& tm_kvals, int H, const MqaArgs& a,
                              cudaStream_t stream);

// top-k of every row's candidate list (the second launch of mqa_logits + top-k)
cudaError_t launch_cand_topk(const float* cand_vals, const int32_t* cand_idx,
                             const uint32_t* cand_cnt, int64_t cand_ld, int64_t rows, int32_t k,
                             int32_t* out, cudaStream_t stream);

cudaError_t launch_topk_rows(const float* logits, int64_t rows, int64_t ld,
                             const int32_t* row_start, const int32_t* row_end, int32_t k,
                             int32_t* out, int sms, cudaStream_t stream);

cudaError_t launch_gather_k(const uint8_t* cache, int64_t num_blocks, const int32_t* block_table,
                            int32_t max_blocks, const int32_t* seq_lens,
                            const int64_t* out_offsets, int32_t B, uint8_t* k_vals,
                            uint8_t* k_scales, int64_t out_rows, idx_device_errors* errors,
                            cudaStream_t stream);

}  // namespace idx
