/*
 * CPU oracle for the MXFP4 lightning-indexer path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the indexer path computes.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load it.  The CUDA
 * library shares no code, header, table or constant with it, and the product
 * path never calls it.
 *
 * Sources (web pages on the subject):
 *   [PR-48558]  vLLM PR #48558 "[Kernel] MXFP4 indexer cache for GLM-5.2 / DSA"
 *               sections "What", "Changes", "Benefit", "Notes" and the
 *               "Live validation" comment (block-split value/scale layout,
 *               132 -> 68 B per token per head, E2M1 values + UE8M0 block-32
 *               scales, slot_mapping of int64).
 *   [PR-14]     Whamp/vllm PR #14 "Enable SM86 MXFP4 sparse-indexer cache",
 *               sections "Summary" and "Validation" (software E2M1/UE8M0
 *               writers, exact top-k-set and poisoned-tail checks).
 *   [SPARSE-IDX] vLLM API docs "vllm.models.glm5next.nvidia.sparse_indexer",
 *               class SparseAttnIndexerKpool (mqa_logits, paged_mqa_logits,
 *               top_k_per_row; FP4 q arrives as a (values, scales) pair).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - UE8M0 scale of a 32-element block: the smallest integer e with
 *     amax <= 6 * 2^e, stored as e + 127 clamped to [0, 254]; amax == 0 gives
 *     byte 0 (the minimum exponent).
 *   - E2M1: round to nearest, ties to the even code, over
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}; magnitudes above 6 saturate to 6; the sign
 *     bit (0x8) follows the sign of the input, also when the magnitude rounds
 *     to zero.
 *   - Packing: byte i of a token holds element 2i in the low nibble and
 *     element 2i+1 in the high nibble; the 4 scale bytes are in block order.
 *   - Page of P tokens: P*64 value bytes, then P*4 scale bytes.
 *   - logit[r,s] = sum_h w[r,h] * max(0, sum_d q^[r,h,d] * k^[s,d]), computed
 *     here in fp64 on exactly dequantised operands; beside each logit the
 *     oracle returns mag[r,s] = sum_h |w[r,h]| * sum_d |q^[r,h,d] * k^[s,d]|,
 *     the scale that the comparison tolerance multiplies.
 *   - Top-k: rank by (logit descending, index ascending); fewer than k valid
 *     keys give all of them followed by -1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D_HEAD 128          /* indexer head_dim */
#define BLOCK 32            /* MX block size */
#define VAL_BYTES 64        /* 128 E2M1 nibbles */
#define SCALE_BYTES 4       /* one UE8M0 byte per block of 32 */

/* The eight E2M1 magnitudes, indexed by the 3 low bits of a code. */
static const double E2M1_GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* bf16 bit pattern -> its exact value. */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* UE8M0 scale byte of one block: smallest integer e with amax <= 6 * 2^e,
 * found by walking e upward and comparing against ldexp(6, e) in fp64, so no
 * rounded log2 is involved.  amax == 0 -> byte 0. */
uint8_t oracle_ue8m0_scale(const double* x, int n) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) {
    double a = fabs(x[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0) return 0;
  for (int e = -127; e <= 127; ++e) {
    if (amax <= ldexp(6.0, e)) return (uint8_t)(e + 127);
  }
  return 254; /* clamp to the largest finite E8M0 value */
}

/* E2M1 code of y (already divided by the block scale). */
uint8_t oracle_e2m1_code(double y) {
  uint8_t sign = signbit(y) ? 0x8 : 0x0;
  double a = fabs(y);
  if (a > 6.0) return (uint8_t)(sign | 7);
  int best = 0;
  double best_dist = fabs(a - E2M1_GRID[0]);
  for (int c = 1; c < 8; ++c) {
    double dist = fabs(a - E2M1_GRID[c]);
    /* strictly nearer wins; an exact tie goes to the even code */
    if (dist < best_dist || (dist == best_dist && (c % 2 == 0) && (best % 2 != 0))) {
      best = c;
      best_dist = dist;
    }
  }
  return (uint8_t)(sign | best);
}

/* Value of a 4-bit E2M1 code. */
double oracle_e2m1_value(uint8_t code) {
  double v = E2M1_GRID[code & 7];
  return (code & 8) ? -v : v;
}

/* Quantise one 128-element bf16 vector to 64 packed value bytes and 4 scale
 * bytes ([PR-48558] "Changes": E2M1 values + UE8M0 block-32 scales). */
void oracle_quant_vec128(const uint16_t* x_bf16, uint8_t* vals, uint8_t* scales) {
  double x[D_HEAD];
  for (int d = 0; d < D_HEAD; ++d) x[d] = oracle_bf16_to_double(x_bf16[d]);
  uint8_t codes[D_HEAD];
  for (int b = 0; b < D_HEAD / BLOCK; ++b) {
    uint8_t s = oracle_ue8m0_scale(x + b * BLOCK, BLOCK);
    scales[b] = s;
    for (int i = 0; i < BLOCK; ++i) {
      double y = ldexp(x[b * BLOCK + i], 127 - (int)s); /* exact power-of-2 divide */
      codes[b * BLOCK + i] = oracle_e2m1_code(y);
    }
  }
  for (int i = 0; i < VAL_BYTES; ++i)
    vals[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
}

/* Inverse of the above: 128 exact values. */
void oracle_dequant_vec128(const uint8_t* vals, const uint8_t* scales, double* out) {
  for (int d = 0; d < D_HEAD; ++d) {
    uint8_t byte = vals[d / 2];
    uint8_t code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    int e = (int)scales[d / BLOCK] - 127;
    out[d] = ldexp(oracle_e2m1_value(code), e);
  }
}

/* Quantise-and-insert ([PR-48558] "Changes", indexer_k_quant_and_cache with
 * scale_fmt "mxfp4"; "Live validation": block-split value/scale layout).
 * Token i goes to slot slots[i] = page * P + offset.  Slot -1 is padding and is
 * skipped; any other slot outside [0, num_blocks * P) is skipped and counted.
 * Returns the number of such bad slots.  Bytes not written keep their value. */
int64_t oracle_quant_insert(const uint16_t* k, int64_t n_tokens, int64_t row_stride,
                            const int64_t* slots, uint8_t* cache, int64_t num_blocks,
                            int32_t page_size) {
  int64_t bad = 0;
  const int64_t page_bytes = (int64_t)page_size * (VAL_BYTES + SCALE_BYTES);
  for (int64_t i = 0; i < n_tokens; ++i) {
    int64_t slot = slots[i];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_blocks * (int64_t)page_size) { ++bad; continue; }
    int64_t page = slot / page_size, off = slot % page_size;
    uint8_t* vdst = cache + page * page_bytes + off * VAL_BYTES;
    uint8_t* sdst = cache + page * page_bytes + (int64_t)page_size * VAL_BYTES + off * SCALE_BYTES;
    oracle_quant_vec128(k + i * row_stride, vdst, sdst);
  }
  return bad;
}

/* Query quantisation: each of `rows` 128-element vectors (rows = T * H) to
 * vals[rows, 64] and scales[rows, 4] ([PR-48558] "Notes": MXFP4 q-quant;
 * [SPARSE-IDX] forward_cuda: FP4 q is a (values, scales) pair). */
void oracle_quant_q(const uint16_t* q, int64_t rows, uint8_t* vals, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r)
    oracle_quant_vec128(q + r * D_HEAD, vals + r * VAL_BYTES, scales + r * SCALE_BYTES);
}

/* One logit and its tolerance scale, from dequantised q (H x 128) and k. */
static void logit_one(const double* qhat, const double* khat, const float* w, int32_t H,
                      double* logit, double* mag) {
  double acc = 0.0, m = 0.0;
  for (int32_t h = 0; h < H; ++h) {
    double dot = 0.0, adot = 0.0;
    for (int d = 0; d < D_HEAD; ++d) {
      double p = qhat[h * D_HEAD + d] * khat[d];
      dot += p;
      adot += fabs(p);
    }
    double relu = dot > 0.0 ? dot : 0.0;
    acc += (double)w[h] * relu;
    m += fabs((double)w[h]) * adot;
  }
  *logit = acc;
  *mag = m;
}

/* Prefill logits over contiguous keys ([SPARSE-IDX] mqa_logits).
 * Row t sees keys [row_start[t], row_end[t]); only those columns of logits/mag
 * (row stride ld) are written. */
void oracle_mqa_logits(const uint8_t* q_vals, const uint8_t* q_scales, int64_t T, int32_t H,
                       const uint8_t* k_vals, const uint8_t* k_scales, int64_t S,
                       const float* weights, const int32_t* row_start, const int32_t* row_end,
                       double* logits, double* mag, int64_t ld) {
  (void)S;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double* qhat = (double*)malloc(sizeof(double) * (size_t)H * D_HEAD);
    double khat[D_HEAD];
    for (int32_t h = 0; h < H; ++h)
      oracle_dequant_vec128(q_vals + (t * H + h) * VAL_BYTES, q_scales + (t * H + h) * SCALE_BYTES,
                            qhat + h * D_HEAD);
    for (int64_t s = row_start[t]; s < row_end[t]; ++s) {
      oracle_dequant_vec128(k_vals + s * VAL_BYTES, k_scales + s * SCALE_BYTES, khat);
      logit_one(qhat, khat, weights + t * H, H, logits + t * ld + s, mag + t * ld + s);
    }
    free(qhat);
  }
}

/* Decode logits through a block table ([SPARSE-IDX] paged_mqa_logits;
 * [PR-48558] "Notes": the paged MQA-logits reader).
 * Row r = b * next_n + j is query token j of sequence b, whose context (new
 * tokens included) has L_b = context_lens[b] tokens; it sees positions
 * [0, L_b - next_n + j].  Position s lives in page block_table[b][s / P] at
 * offset s % P.  Columns [0, len_r) of logits/mag are written. */
void oracle_paged_mqa_logits(const uint8_t* q_vals, const uint8_t* q_scales, int32_t B,
                             int32_t next_n, int32_t H, const uint8_t* cache, int32_t page_size,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* context_lens, const float* weights, double* logits,
                             double* mag, int64_t ld) {
  const int64_t page_bytes = (int64_t)page_size * (VAL_BYTES + SCALE_BYTES);
  const int64_t rows = (int64_t)B * next_n;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t b = r / next_n, j = r % next_n;
    int64_t len = (int64_t)context_lens[b] - next_n + j + 1;
    double* qhat = (double*)malloc(sizeof(double) * (size_t)H * D_HEAD);
    double khat[D_HEAD];
    for (int32_t h = 0; h < H; ++h)
      oracle_dequant_vec128(q_vals + (r * H + h) * VAL_BYTES, q_scales + (r * H + h) * SCALE_BYTES,
                            qhat + h * D_HEAD);
    for (int64_t s = 0; s < len; ++s) {
      int64_t page = block_table[b * max_blocks + s / page_size];
      int64_t off = s % page_size;
      const uint8_t* kv = cache + page * page_bytes + off * VAL_BYTES;
      const uint8_t* ks = cache + page * page_bytes + (int64_t)page_size * VAL_BYTES + off * SCALE_BYTES;
      oracle_dequant_vec128(kv, ks, khat);
      logit_one(qhat, khat, weights + r * H, H, logits + r * ld + s, mag + r * ld + s);
    }
    free(qhat);
  }
}

typedef struct { double v; int64_t i; } ranked_t;

static int rank_cmp(const void* a, const void* b) {
  const ranked_t* x = (const ranked_t*)a;
  const ranked_t* y = (const ranked_t*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i < y->i) ? -1 : (x->i > y->i);
}

/* Top-k of each row ([SPARSE-IDX] top_k_per_row into topk_indices_buffer).
 * Row r ranks columns [row_start[r], row_end[r]) of logits (stride ld) by
 * (value desc, index asc) and writes the first min(k, len) indices, each as
 * column - row_start[r], then -1 up to k. */
void oracle_topk_rows(const double* logits, int64_t rows, int64_t ld, const int32_t* row_start,
                      const int32_t* row_end, int32_t k, int32_t* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t st = row_start[r], len = (int64_t)row_end[r] - st;
    if (len < 0) len = 0;
    ranked_t* tmp = (ranked_t*)malloc(sizeof(ranked_t) * (size_t)(len > 0 ? len : 1));
    for (int64_t i = 0; i < len; ++i) { tmp[i].v = logits[r * ld + st + i]; tmp[i].i = i; }
    qsort(tmp, (size_t)len, sizeof(ranked_t), rank_cmp);
    for (int32_t i = 0; i < k; ++i) out[r * (int64_t)k + i] = (i < len) ? (int32_t)tmp[i].i : -1;
    free(tmp);
  }
}

/* Gather a sequence's cached tokens into contiguous value/scale arrays
 * ([PR-48558] "Live validation": the shared cp_gather over the block-split
 * layout).  Sequence b's tokens [0, seq_lens[b]) go to rows
 * out_offsets[b] + s of k_vals[., 64] and k_scales[., 4]. */
void oracle_gather_k(const uint8_t* cache, int32_t page_size, const int32_t* block_table,
                     int32_t max_blocks, const int32_t* seq_lens, const int64_t* out_offsets,
                     int32_t B, uint8_t* k_vals, uint8_t* k_scales) {
  const int64_t page_bytes = (int64_t)page_size * (VAL_BYTES + SCALE_BYTES);
  for (int32_t b = 0; b < B; ++b) {
    for (int64_t s = 0; s < seq_lens[b]; ++s) {
      int64_t page = block_table[(int64_t)b * max_blocks + s / page_size];
      int64_t off = s % page_size;
      int64_t dst = out_offsets[b] + s;
      memcpy(k_vals + dst * VAL_BYTES, cache + page * page_bytes + off * VAL_BYTES, VAL_BYTES);
      memcpy(k_scales + dst * SCALE_BYTES,
             cache + page * page_bytes + (int64_t)page_size * VAL_BYTES + off * SCALE_BYTES,
             SCALE_BYTES);
    }
  }
}

/* ------------------------------------------------------------------------
 * Quantisation of an fp32 vector of 128 (the rounded result of an fp32
 * computation, e.g. a rotated query or a pooled key): the same scale, code and
 * packing rules as oracle_quant_vec128, applied to the exact fp32 values. */
void oracle_quant_vec128_f32(const float* xf, uint8_t* vals, uint8_t* scales) {
  double x[D_HEAD];
  for (int d = 0; d < D_HEAD; ++d) x[d] = (double)xf[d];
  uint8_t codes[D_HEAD];
  for (int b = 0; b < D_HEAD / BLOCK; ++b) {
    uint8_t s = oracle_ue8m0_scale(x + b * BLOCK, BLOCK);
    scales[b] = s;
    for (int i = 0; i < BLOCK; ++i)
      codes[b * BLOCK + i] = oracle_e2m1_code(ldexp(x[b * BLOCK + i], 127 - (int)s));
  }
  for (int i = 0; i < VAL_BYTES; ++i)
    vals[i] = (uint8_t)((codes[2 * i + 1] << 4) | codes[2 * i]); /* element 2i low */
}

/* ------------------------------------------------------------------------
 * Rotary position embedding of query heads, then MXFP4 quantisation
 * ([PR-48558] "Notes": a fused q-rope + MXFP4 q-quant).  The pages give no
 * rotary parameters, so the caller passes the table:
 *   q      [T, H, 128] bf16; pos [T] row of the table for token t;
 *   cs, sn [num_pos, rot_dim / 2] fp32 cosines and sines.
 * Reading: the first rot_dim dimensions (even, <= 128) are rotated in
 * interleaved pairs (2i, 2i+1) by the angle of table column i; the other
 * dimensions pass through.  The rotation is an fp32 computation whose result
 * is then quantised, so the rounding that decides the codes is fixed here in
 * fp32 with one stated order:
 *   x' = fmaf(x, c, -(y * s)),  y' = fmaf(x, s, y * c)
 * (each product y*s, y*c rounded to fp32 first, then one fused multiply-add).
 * out_f32 (optional) receives the rotated values. */
void oracle_rope_quant_q(const uint16_t* q, const int32_t* pos, int64_t T, int32_t H,
                         const float* cs, const float* sn, int32_t rot_dim, uint8_t* vals,
                         uint8_t* scales, float* out_f32) {
  const int32_t half = rot_dim / 2;
  for (int64_t t = 0; t < T; ++t) {
    const float* c_row = cs + (int64_t)pos[t] * half;
    const float* s_row = sn + (int64_t)pos[t] * half;
    for (int32_t h = 0; h < H; ++h) {
      const int64_t r = t * H + h;
      float x[D_HEAD];
      for (int d = 0; d < D_HEAD; ++d) x[d] = (float)oracle_bf16_to_double(q[r * D_HEAD + d]);
      for (int32_t i = 0; i < half; ++i) {
        const float a = x[2 * i], b = x[2 * i + 1], c = c_row[i], s = s_row[i];
        const float bs = b * s, bc = b * c;
        x[2 * i] = fmaf(a, c, -bs);
        x[2 * i + 1] = fmaf(a, s, bc);
      }
      if (out_f32) memcpy(out_f32 + r * D_HEAD, x, sizeof x);
      oracle_quant_vec128_f32(x, vals + r * VAL_BYTES, scales + r * SCALE_BYTES);
    }
  }
}

/* ------------------------------------------------------------------------
 * K-pool compressed insert ([SPARSE-IDX] _kpool_compress_insert).
 * The masking rule is the page's: with n rows and pool size P, row p is a
 * pool-completion candidate; it is written iff slot[p] >= 0 and p >= P - 1
 * (a valid slot at p < P - 1 belongs to a pool that started before the batch
 * and is dropped); nothing is written when n < P.  Pool p covers rows
 * p - P + 1 .. p.
 * The pooling arithmetic is not given by the pages; reading: per dimension d,
 * the pool's rows are weighted by a softmax over the pool of
 * gate[row, d] + ape[j, d] (j = position of the row within the pool) and
 * summed:  kc[d] = sum_j softmax_j(gate + ape) * k[row_j, d].
 *
 * oracle_kpool_compress: kc for every candidate row in fp64 (rows that are not
 * written get NaN), and beside it mag[p, d] = sum_j w_j |k[row_j, d]| (the
 * scale of the comparison tolerance).  gate [n, 128] fp32, ape [P, 128] fp32,
 * k [n, 128] bf16. */
void oracle_kpool_compress(const uint16_t* k, const float* gate, const float* ape,
                           const int64_t* slots, int64_t n, int32_t P, double* kc, double* mag) {
  double* z = (double*)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1));
  for (int64_t p = 0; p < n; ++p) {
    const int write = (n >= P) && slots[p] >= 0 && p >= P - 1;
    const int64_t r0 = p - P + 1; /* the pool's first row */
    for (int d = 0; d < D_HEAD; ++d) {
      if (!write) {
        kc[p * D_HEAD + d] = NAN;
        mag[p * D_HEAD + d] = NAN;
        continue;
      }
      double m = -INFINITY;
      for (int32_t j = 0; j < P; ++j) {
        z[j] = (double)gate[(r0 + j) * D_HEAD + d] + (double)ape[(int64_t)j * D_HEAD + d];
        if (z[j] > m) m = z[j];
      }
      double den = 0.0, num = 0.0, am = 0.0;
      for (int32_t j = 0; j < P; ++j) {
        const double e = exp(z[j] - m);
        const double kv = oracle_bf16_to_double(k[(r0 + j) * D_HEAD + d]);
        den += e;
        num += e * kv;
        am += e * fabs(kv);
      }
      kc[p * D_HEAD + d] = num / den;
      mag[p * D_HEAD + d] = am / den;
    }
  }
  free(z);
}

/* The write step of the K-pool insert: the pooled vector of every written row
 * p (kc32 [n, 128], the fp32 values that are quantised; other rows are not
 * read) is quantised like a key and stored at slot[p] of the paged cache.
 * Slots outside [0, num_blocks * page_size) are skipped and counted. */
int64_t oracle_kpool_insert(const float* kc32, const int64_t* slots, int64_t n, int32_t P,
                            uint8_t* cache, int64_t num_blocks, int32_t page_size) {
  int64_t bad = 0;
  if (n < P) return 0;
  const int64_t page_bytes = (int64_t)page_size * (VAL_BYTES + SCALE_BYTES);
  for (int64_t p = P - 1; p < n; ++p) {
    const int64_t slot = slots[p];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)page_size) { ++bad; continue; }
    const int64_t page = slot / page_size, off = slot % page_size;
    oracle_quant_vec128_f32(kc32 + p * D_HEAD, cache + page * page_bytes + off * VAL_BYTES,
                            cache + page * page_bytes + (int64_t)page_size * VAL_BYTES +
                                off * SCALE_BYTES);
  }
  return bad;
}
