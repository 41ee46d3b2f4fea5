/*
 * idx.h -- C ABI of libidx, the GB300 (sm_103a) MXFP4 lightning-indexer path.
 *
 * The operations are those of the DSA lightning indexer with an MXFP4 K-cache as
 * described by:
 *   - vLLM PR #48558 "[Kernel] MXFP4 indexer cache for GLM-5.2 / DSA" (sections
 *     "What", "Changes", "Benefit", "Notes", and the "Live validation" comment);
 *   - Whamp/vllm PR #14 "Enable SM86 MXFP4 sparse-indexer cache" (sections
 *     "Summary", "Validation");
 *   - vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer",
 *     class SparseAttnIndexerKpool (mqa_logits, paged_mqa_logits,
 *     top_k_per_row, forward_cuda).
 *
 * Formats (fixed by this library; the pages give the sizes, not the rounding):
 *   - An indexer key or query head is 128 values.  MXFP4 stores it as 64 bytes
 *     of E2M1 codes (element 2i in the low nibble of byte i, element 2i+1 in the
 *     high nibble) and 4 UE8M0 scale bytes, one per block of 32 elements, in
 *     block order: 68 bytes instead of FP8's 132 (PR #48558, "Benefit").
 *   - Scale of a block: byte e+127 for the smallest integer e with
 *     max|x| <= 6 * 2^e, clamped to [0, 254]; an all-zero block gets byte 0.
 *   - Code of x: x / 2^e rounded to the nearest of {0,0.5,1,1.5,2,3,4,6}, ties to
 *     the even code, magnitudes above 6 saturate to 6; bit 3 is the sign of x
 *     (also when the magnitude rounds to 0).  Inf/NaN inputs are outside the
 *     contract.
 *   - Paged cache: pages of page_size = 64 tokens, 4352 bytes each: the 64x64
 *     value bytes of the page's tokens (token-major), then their 64x4 scale
 *     bytes ("block-split" layout, PR #48558 "Live validation").  Token slot
 *     s = page * 64 + offset.
 *   - logit[r, s] = sum_h w[r, h] * max(0, sum_d q^[r, h, d] * k^[s, d]) on
 *     dequantised operands, fp32 accumulation.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory and never synchronises; work is enqueued on
 *     `stream` (NULL = the legacy default stream) and the call returns at once.
 *     So every call other than idx_paged_logits_topk_noalloc can be captured
 *     in a CUDA graph; a replay reads its buffers afresh (the fused call's
 *     work-item counter starts over on every replay).
 *   - Argument and device errors are returned synchronously, before anything is
 *     enqueued.  IDX_ERR_CUDA reports a launch failure (the CUDA error string
 *     is available from idx_last_error_detail()).
 *   - Contract violations that only the device can see (a slot or block id out
 *     of range, a context longer than the block table or the logits row) are
 *     skipped by the kernels and counted in the optional `errors` struct.  The
 *     kernels never trap.  A pipeline wait that exceeds its limit (a library
 *     bug, not an input error) sets a bit in errors->timeouts and the kernel
 *     returns early.
 *   - Supported shapes: head_dim 128, page_size 64, H in {32, 64},
 *     next_n in {1, 2}, 1 <= k <= 2048.  Others give IDX_ERR_INVALID_ARG.
 *   - Only sm_103 devices are accepted (IDX_ERR_UNSUPPORTED_DEVICE otherwise).
 */
#ifndef IDX_H_
#define IDX_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define IDX_API __attribute__((visibility("default")))
#else
#define IDX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* idx_stream_t;

typedef enum {
  IDX_OK = 0,
  IDX_ERR_INVALID_ARG = 1,
  IDX_ERR_UNSUPPORTED_DEVICE = 2,
  IDX_ERR_WORKSPACE_TOO_SMALL = 3,
  IDX_ERR_CUDA = 4
} idx_status;

/* Device-side error counters (device memory, zeroed by the caller). */
typedef struct {
  int32_t bad_inputs; /* skipped slots / block ids / over-long contexts */
  int32_t timeouts;   /* bit mask of pipeline waits that gave up */
} idx_device_errors;

/* Library version, major * 10000 + minor * 100 + patch. */
IDX_API int idx_version(void);

/* Static description of a status code. */
IDX_API const char* idx_status_string(idx_status status);

/* Detail of the last failing call on this host thread ("" if none). */
IDX_API const char* idx_last_error_detail(void);

/* Fail-closed architecture gate (Whamp/vllm PR #14, "Summary": fail-closed
 * capability gates).  Pure host logic: IDX_OK only for compute capability
 * 10.3 (sm_103, GB300). */
IDX_API idx_status idx_arch_supported(int major, int minor);

/* Applies idx_arch_supported to `device`.  IDX_ERR_CUDA if the device cannot be
 * queried. */
IDX_API idx_status idx_check_device(int device);

/* ---------------------------------------------------------------------------
 * idx_quant_insert -- quantise indexer keys to MXFP4 and scatter them into the
 * paged cache (PR #48558, "Changes": indexer_k_quant_and_cache with scale_fmt
 * "mxfp4"; "Live validation": block-split value/scale layout).
 *   k_bf16        [n_tokens, k_row_stride] bf16; the first 128 values of each row
 *                 are the key.  Base 16-byte aligned, k_row_stride a multiple of 8.
 *   slot_mapping  [n_tokens] int64 slots; -1 = padding, skipped; any other value
 *                 outside [0, num_blocks*page_size) is skipped and counted.
 *   kcache        [num_blocks, page_size*68] bytes, 16-byte aligned.  Only the 68
 *                 bytes of each inserted token are written.
 * n_tokens == 0 is a no-op.  Slots must be distinct (duplicates race).
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_quant_insert(const void* k_bf16, int64_t n_tokens, int64_t k_row_stride,
                            const int64_t* slot_mapping, uint8_t* kcache, int64_t num_blocks,
                            int32_t page_size, idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_quant_q -- quantise query heads with the same rule (PR #48558, "Notes":
 * MXFP4 q-quant; sparse_indexer forward_cuda: FP4 q is a (values, scales) pair).
 *   q_bf16    [rows, 128] bf16, contiguous, 16-byte aligned (rows = T * H).
 *   q_vals    [rows, 64] bytes out;  q_scales [rows, 4] bytes out.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_quant_q(const void* q_bf16, int64_t rows, uint8_t* q_vals, uint8_t* q_scales,
                       idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_rope_quant_q -- rotary position embedding of the query heads fused with
 * their MXFP4 quantisation (PR #48558, "Notes": a fused q-rope + MXFP4 q-quant
 * kernel could follow the PyTorch q-quant).  The pages give no rotary
 * parameters; the caller passes the table.
 *   q_bf16     [T, H, 128] bf16, contiguous, 16-byte aligned.
 *   positions  [T] int32: the table row of token t.  When rot_dim > 0, a token
 *              whose position is outside [0, num_pos) is skipped (its rows are
 *              not written) and counted in errors->bad_inputs; with rot_dim = 0
 *              positions are not read (may be any pointer, even NULL).
 *   cos_table, sin_table [num_pos, rot_dim / 2] fp32: cosine and sine of the
 *              angle of pair i at each position (may be NULL when rot_dim = 0).
 *   rot_dim    even, 0..128: dimensions [0, rot_dim) turn in pairs (2i, 2i+1):
 *              x' = x cos - y sin, y' = x sin + y cos, in fp32 with the products
 *              y sin and y cos rounded first and one fused multiply-add each;
 *              the other dimensions pass through.
 *   q_vals / q_scales [T*H, 64] / [T*H, 4] out, as idx_quant_q (row t*H + h).
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_rope_quant_q(const void* q_bf16, int64_t T, int32_t H,
                            const int32_t* positions, const float* cos_table,
                            const float* sin_table, int32_t num_pos, int32_t rot_dim,
                            uint8_t* q_vals, uint8_t* q_scales, idx_device_errors* errors,
                            idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_kpool_insert -- K-pool compressed insert (sparse_indexer docs,
 * _kpool_compress_insert): pools of kpool consecutive keys become one MXFP4
 * key, written at pool-granular slots, masked in the kernel (no compaction,
 * no synchronisation).
 *   k_bf16        [n, 128] bf16 keys of the batch in token order, contiguous.
 *   gate          [n, 128] fp32 gate scores; ape [kpool, 128] fp32 position terms.
 *   slot_mapping  [n] int64, pool-granular: row p completes a pool, and is
 *                 written, iff slot[p] >= 0 and p >= kpool - 1 (a valid slot
 *                 earlier belongs to a pool that began before the batch); a
 *                 batch with n < kpool writes nothing.  Slots past the cache are
 *                 skipped and counted.  Pool chunks start pool-aligned.
 *   Written row p: kc[d] = sum_j softmax_j(gate[p-kpool+1+j, d] + ape[j, d])
 *                 * k[p-kpool+1+j, d] over j < kpool (fp32; the pages fix the
 *                 masking, this library reads the pooling as a softmax of gate
 *                 plus position term), quantised as a key and stored at slot[p].
 *   kcache        paged cache as for idx_quant_insert.
 *   pooled        [n, 128] fp32 out, optional (NULL): kc of the written rows;
 *                 other rows are not touched.
 *   1 <= kpool <= 128.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_kpool_insert(const void* k_bf16, const float* gate, const float* ape,
                            const int64_t* slot_mapping, int64_t n, int32_t kpool,
                            uint8_t* kcache, int64_t num_blocks, int32_t page_size,
                            float* pooled, idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_paged_mqa_logits -- decode logits through block tables (sparse_indexer
 * docs: paged_mqa_logits; PR #48558 "Notes": the paged MQA-logits reader).
 *   q_vals/q_scales  [B*next_n*H, 64] / [B*next_n*H, 4]: query row r = b*next_n + j,
 *                    head h at row r*H + h.
 *   kcache           paged cache as for idx_quant_insert, num_blocks pages.
 *   block_table      [B, max_blocks] int32 page ids.
 *   context_lens     [B] int32: L_b, tokens of sequence b including its next_n
 *                    new ones.  Row (b, j) sees positions [0, L_b - next_n + j].
 *   weights          [B*next_n, H] fp32.
 *   logits           [B*next_n, ld] fp32 out.  Column s < window length gets the
 *                    logit.  With clean != 0 every other column in [0, ld) gets
 *                    -inf; with clean == 0 those columns are not written.
 * A context longer than min(max_blocks*page_size, ld) is clamped and counted.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_paged_mqa_logits(const uint8_t* q_vals, const uint8_t* q_scales, int32_t B,
                                int32_t next_n, int32_t H, const uint8_t* kcache,
                                int64_t num_blocks, int32_t page_size,
                                const int32_t* block_table, int32_t max_blocks,
                                const int32_t* context_lens, const float* weights,
                                float* logits, int64_t ld, int clean,
                                idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_mqa_logits -- prefill logits over contiguous keys (sparse_indexer docs:
 * mqa_logits).
 *   q_vals/q_scales  [T*H, 64] / [T*H, 4]: query t, head h at row t*H + h.
 *   k_vals/k_scales  [S, 64] / [S, 4] (e.g. from idx_gather_k), 16-byte aligned.
 *   weights          [T, H] fp32.
 *   row_start/row_end [T] int32: query t sees keys [row_start[t], row_end[t]),
 *                    0 <= start <= end <= S (windows outside are clamped and
 *                    counted in errors->bad_inputs).
 *   logits           [T, ld] fp32 out, ld >= S.  Columns in the window get the
 *                    logit; with clean != 0 the other columns of [0, S) get
 *                    -inf, otherwise they are not written.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_mqa_logits(const uint8_t* q_vals, const uint8_t* q_scales, int64_t T, int32_t H,
                          const uint8_t* k_vals, const uint8_t* k_scales, int64_t S,
                          const float* weights, const int32_t* row_start,
                          const int32_t* row_end, float* logits, int64_t ld, int clean,
                          idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_mqa_logits_topk -- idx_mqa_logits followed by top-k of every row
 * (sparse_indexer docs: mqa_logits then top_k_per_row) without a logits
 * tensor: the scoring kernel keeps, per row, a threshold that only grows (the
 * k-th largest of the logits admitted so far, to within a histogram bin) and
 * appends only the logits that reach it, with their positions, to the row's
 * candidate list; a second kernel selects the k largest of each list.
 *   Arguments as for idx_mqa_logits (without logits/ld/clean) and
 *   idx_topk_rows: out_idx [T, k] int32 holds positions relative to
 *   row_start[t], in no particular order, -1 after the last valid one.
 *   workspace  at least idx_mqa_logits_topk_workspace_bytes(T, S, k) bytes,
 *              256-byte aligned, no initialisation: per row a list of up to S
 *              candidates (8 bytes each: every position of a row whose logits
 *              rise with the position is a candidate), of which typically a
 *              small part is written.  Calls that share it must not overlap.
 * ------------------------------------------------------------------------ */
IDX_API size_t idx_mqa_logits_topk_workspace_bytes(int64_t T, int64_t S, int32_t k);

IDX_API idx_status idx_mqa_logits_topk(const uint8_t* q_vals, const uint8_t* q_scales, int64_t T,
                               int32_t H, const uint8_t* k_vals, const uint8_t* k_scales,
                               int64_t S, const float* weights, const int32_t* row_start,
                               const int32_t* row_end, int32_t k, int32_t* out_idx,
                               void* workspace, size_t workspace_bytes,
                               idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_topk_rows -- top-k per logits row (sparse_indexer docs: top_k_per_row
 * into topk_indices_buffer).
 *   logits           [rows, ld] fp32; only columns [row_start[r], row_end[r]) are
 *                    read (NULL row_start means 0 for every row).
 *   out_idx          [rows, k] int32 out: the columns of the k largest values,
 *                    each minus row_start[r], in no particular order.  A row
 *                    with fewer than k columns lists all of them, then -1.
 *                    Equal values may be taken in any order.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_topk_rows(const float* logits, int64_t rows, int64_t ld,
                         const int32_t* row_start, const int32_t* row_end, int32_t k,
                         int32_t* out_idx, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_paged_logits_topk -- idx_paged_mqa_logits followed by top-k of every row,
 * without writing the logits to memory.  Arguments as for those two entries;
 * out_idx [B*next_n, k] int32 holds positions in the sequence (-1 padded).
 *   workspace        device scratch of at least
 *                    idx_paged_logits_topk_workspace_bytes(...) bytes, 256-byte
 *                    aligned; its contents need no initialisation and are
 *                    meaningless after the call.  Calls that share a workspace
 *                    must not overlap on the GPU.
 *   A batch of more than about 16 million work items (B times the items per
 *   sequence, up to 16 pages each) is rejected with IDX_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
IDX_API size_t idx_paged_logits_topk_workspace_bytes(int32_t B, int32_t next_n, int32_t max_blocks,
                                             int32_t page_size, int32_t k);

IDX_API idx_status idx_paged_logits_topk(const uint8_t* q_vals, const uint8_t* q_scales, int32_t B,
                                 int32_t next_n, int32_t H, const uint8_t* kcache,
                                 int64_t num_blocks, int32_t page_size,
                                 const int32_t* block_table, int32_t max_blocks,
                                 const int32_t* context_lens, const float* weights, int32_t k,
                                 int32_t* out_idx, void* workspace, size_t workspace_bytes,
                                 idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_paged_logits_topk_noalloc -- idx_paged_logits_topk for callers that
 * cannot allocate device memory: an engine whose allocator is frozen after
 * start-up, a plugin host that passes raw buffers but offers no allocator, or a
 * latency-critical step that must not pay for cudaMalloc (it can block on the
 * device).  The pages have no counterpart for this entry; it only changes where
 * the scratch comes from.
 *   Arguments as for idx_paged_logits_topk, without workspace/workspace_bytes.
 *   The scratch is a 32 MiB array inside the library: every GPU that loads the
 *   library reserves it until the process exits.  Its device address is looked
 *   up on the first call in each CUDA context (the calling thread's current
 *   one) and kept for later calls in that context; a device reset ends the
 *   context, and the next call looks the address up again.
 *   A batch whose idx_paged_logits_topk_workspace_bytes exceeds 32 MiB is
 *   rejected with IDX_ERR_INVALID_ARG (the reason is in
 *   idx_last_error_detail()); use idx_paged_logits_topk with a caller
 *   workspace for it.
 *   All calls share the one scratch array: calls that overlap on the GPU race.
 *   Nothing in the scratch needs clearing between calls: the work-item counter
 *   at its start carries each call's generation and is reset by the call's
 *   select pass; the logits rows behind it are rewritten before being read.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_paged_logits_topk_noalloc(
    const uint8_t* q_vals, const uint8_t* q_scales, int32_t B, int32_t next_n, int32_t H,
    const uint8_t* kcache, int64_t num_blocks, int32_t page_size, const int32_t* block_table,
    int32_t max_blocks, const int32_t* context_lens, const float* weights, int32_t k,
    int32_t* out_idx, idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_paged_decode_step -- one decode step of the indexer in two launches:
 * the step's insert (PR #48558, "Changes": indexer_k_quant_and_cache ahead of
 * the paged reader) and query quantisation ("Notes") done by the scoring
 * launch of idx_paged_logits_topk, before it scores, then its select.
 *   k_new_bf16   [B*next_n, 128] bf16, contiguous, 16-byte aligned: the step's
 *                new keys; row b*next_n + j is position L_b - next_n + j of
 *                sequence b and is written to that position's page (through
 *                the block table) and offset, as idx_quant_insert would.  A
 *                position outside the block table, or a page id outside the
 *                cache, is skipped and counted.
 *   q_bf16       [B*next_n, H, 128] bf16, contiguous, 16-byte aligned: the
 *                step's query heads, quantised as idx_quant_q would (into the
 *                workspace; nothing else of the caller's is written).
 *   The other arguments are those of idx_paged_logits_topk; context_lens
 *   count the new tokens.  out_idx [B*next_n, k] as there.
 *   workspace    at least idx_paged_decode_step_workspace_bytes(...) bytes,
 *                256-byte aligned, no initialisation, not shared by calls that
 *                overlap on the GPU.  Besides the fused call's contents it
 *                holds the quantised query heads, a chunk counter and one
 *                count per sequence (generation-tagged; the select resets
 *                them to the call's generation with no claims).
 *   The scoring launch does the step's quantisation and insert first, in
 *   small chunks that its CTAs claim from a counter in the workspace; a CTA
 *   waits for a sequence's chunks to be done before it reads any of the
 *   sequence's keys (a bounded wait; a wait that gives up sets the timeout
 *   bit).  The launch needs no co-residency of its CTAs.
 * ------------------------------------------------------------------------ */
IDX_API size_t idx_paged_decode_step_workspace_bytes(int32_t B, int32_t next_n, int32_t H,
                                             int32_t max_blocks, int32_t page_size, int32_t k);

IDX_API idx_status idx_paged_decode_step(const void* k_new_bf16, const void* q_bf16, int32_t B,
                                 int32_t next_n, int32_t H, uint8_t* kcache, int64_t num_blocks,
                                 int32_t page_size, const int32_t* block_table,
                                 int32_t max_blocks, const int32_t* context_lens,
                                 const float* weights, int32_t k, int32_t* out_idx,
                                 void* workspace, size_t workspace_bytes,
                                 idx_device_errors* errors, idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_gather_k -- copy sequences' cached tokens into contiguous value/scale
 * arrays (PR #48558 "Live validation": the shared cp_gather reader).
 *   seq_lens     [B] int32 tokens to copy per sequence (<= max_blocks*page_size).
 *   out_offsets  [B] int64 first output row of each sequence.
 *   k_vals/k_scales [out_rows, 64] / [out_rows, 4] out; rows beyond out_rows are
 *                skipped and counted.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_gather_k(const uint8_t* kcache, int64_t num_blocks, int32_t page_size,
                        const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                        const int64_t* out_offsets, int32_t B, uint8_t* k_vals,
                        uint8_t* k_scales, int64_t out_rows, idx_device_errors* errors,
                        idx_stream_t stream);

/* ---------------------------------------------------------------------------
 * idx_copy_async -- copy `bytes` bytes from src to dst with the GPU's SMs, for
 * the small host<->device transfers of a decode step (its inputs in, its top-k
 * indices out).  The pages have no counterpart for this entry.  On GB300 the
 * SMs reach page-locked host memory over NVLink-C2C, so for a few hundred KB
 * this costs about a kernel launch and one memory round trip, less than a
 * copy-engine transfer.
 *   dst, src   each either device memory of the current device, managed
 *              memory, or page-locked host memory mapped into the device's
 *              address space (as pinned allocations are under unified
 *              addressing), each covering `bytes` bytes of one allocation;
 *              the two ranges must not overlap.  Owned by the caller.
 *   Enqueued on `stream` in stream order (the copy reads src after the
 *   stream's previous work and later work sees dst); bytes == 0 does nothing.
 *   A pointer whose first or last byte the device cannot reach is refused
 *   with IDX_ERR_INVALID_ARG before anything is enqueued.
 * ------------------------------------------------------------------------ */
IDX_API idx_status idx_copy_async(void* dst, const void* src, size_t bytes, idx_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H_ */
