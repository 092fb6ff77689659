/*
 * sga_oracle.c -- plain CPU oracle for vocab-sharded greedy token selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the package smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library: every type and helper below is defined here again on purpose.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] vLLM PR #34049, "[Spec Decode] Reduce TP communication for
 *        speculative decoding draft token generation" -- Solution: local
 *        argmax on each vocab shard, gather (max_value, global_index),
 *        reduce across ranks to the global argmax.
 *   [P2] vLLM PR #39419, "[SpecDecode] Reduce TP communication for
 *        large-vocab draft models speculative decoding" -- review thread
 *        "Refactor local argmax code": local argmax first, then the
 *        draft-to-target id map target_id = k + d2t[k].
 *   [P4] vLLM PR #62604, sharded greedy verification -- Purpose item 1
 *        (per-shard statistics, all-gather on dim 0, one kernel for global
 *        argmax + acceptance + bonus + sampled/rejected counts) and item 2
 *        (fused get_top_tokens: padding mask, lowest id on ties, NaN wins,
 *        as torch.argmax); Test Plan (all -inf rows, NaN rows staying
 *        in-vocabulary, unaligned padding, empty batch).
 *
 * Readings of points the pages leave open (all listed in the design notes):
 *   - ids at or past org_vocab are padding; their value is replaced by -inf
 *     before any comparison ([P4] item 2, "padding mask").
 *   - "NaN wins": the first (lowest-id) NaN among non-padding ids wins and
 *     keeps its own bits.  "Lowest id on ties": equal values (including
 *     +0 and -0) resolve to the lower global id.
 *   - The reported value is the winning element widened to fp32 exactly
 *     (bf16 bits shifted left by 16), or -inf when the winner is padding.
 *   - A row whose every non-padding value is -inf (or that has no
 *     non-padding id at all) reports id = its first id, value -inf.
 *   - Greedy acceptance: drafts are accepted while they equal the target
 *     argmax of the same position; a = accepted count; the emitted tokens
 *     are the target argmaxes of positions 0..a; num_sampled = a + 1,
 *     num_rejected = K - a; "bonus" = the last emitted token.
 *
 * Everything is a plain loop in the order the definitions state.  OpenMP
 * only splits independent rows (or independent dot products); it never
 * changes the order of any comparison or sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

typedef struct {
  float v;
  int32_t id;
} oracle_stat;

/* Widen element idx of a logits buffer to fp32 without rounding. */
static float widen(const void *x, int dtype, int64_t idx) {
  float f;
  if (dtype == ORACLE_F32) {
    memcpy(&f, (const char *)x + 4 * idx, 4);
  } else {
    uint16_t b;
    uint32_t u;
    memcpy(&b, (const char *)x + 2 * idx, 2);
    u = ((uint32_t)b) << 16;
    memcpy(&f, &u, 4);
  }
  return f;
}

/* The padding mask of [P4] item 2: ids >= org_vocab count as -inf. */
static float masked(const void *row, int dtype, int64_t local_j, int64_t global_id,
                    int64_t org_vocab) {
  if (global_id >= org_vocab) return -INFINITY;
  return widen(row, dtype, local_j);
}

/* torch.argmax order: a candidate replaces the running best when the best is
 * not NaN and the candidate is NaN or strictly greater.  Scanning ids in
 * ascending order, this keeps the first NaN and the lowest id among ties. */
static int better(float cand, float best) {
  return !isnan(best) && (isnan(cand) || cand > best);
}

/* Argmax of one row over global ids [first, first + width), where element
 * local j of `row` is global id first + j.  Returns the winning global id and
 * writes the winner's value (its own bits, or -inf if padding). */
static int32_t scan_row(const void *row, int dtype, int64_t first, int64_t width,
                        int64_t org_vocab, float *value_out) {
  int64_t best_j = 0;
  float best = masked(row, dtype, 0, first, org_vocab);
  for (int64_t j = 1; j < width; ++j) {
    float c = masked(row, dtype, j, first + j, org_vocab);
    if (better(c, best)) {
      best = c;
      best_j = j;
    }
  }
  *value_out = masked(row, dtype, best_j, first + best_j, org_vocab);
  return (int32_t)(first + best_j);
}

static int64_t elt_size(int dtype) { return dtype == ORACLE_F32 ? 4 : 2; }

/* Definition: argmax of the whole (unsharded) masked row, as torch.argmax
 * would give on the full logits ([P4] item 2, "same result as torch.argmax"). */
void oracle_full_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                        int64_t vocab, int64_t org_vocab, float *out_vals,
                        int32_t *out_ids) {
  int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
  for (r = 0; r < rows; ++r) {
    const char *row = (const char *)logits + r * ld * elt_size(dtype);
    out_ids[r] = scan_row(row, dtype, 0, vocab, org_vocab, &out_vals[r]);
  }
}

/* Local argmax of one vocab shard ([P1] Solution step 1; [P4] item 1):
 * `logits` points at element (0, shard_start) of rows with stride ld, and
 * the shard covers global ids [shard_start, shard_start + shard_width).  The
 * stat of row r goes to out[r] (the caller passes its shard's block of the
 * dim-0 gathered buffer). */
void oracle_shard_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                         int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                         oracle_stat *out) {
  int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
  for (r = 0; r < rows; ++r) {
    const char *row = (const char *)logits + r * ld * elt_size(dtype);
    float v;
    int32_t id = scan_row(row, dtype, shard_start, shard_width, org_vocab, &v);
    out[r].v = v;
    out[r].id = id;
  }
}

/* Cross-shard reduction of the gathered stats ([P1] Solution step 3): the
 * buffer is shard-major, stats[s * rows + r], shards in ascending id order,
 * exactly as all_gather(dim=0) lays it out ([P4] Test Plan).  The same
 * torch.argmax order over shards: the first NaN sticks, ties keep the lower
 * shard (hence the lower id). */
void oracle_shard_reduce(const oracle_stat *stats, int num_shards, int64_t rows,
                         float *out_vals, int32_t *out_ids) {
  int64_t r;
  for (r = 0; r < rows; ++r) {
    oracle_stat best = stats[r];
    for (int s = 1; s < num_shards; ++s) {
      oracle_stat c = stats[(int64_t)s * rows + r];
      if (better(c.v, best.v)) best = c;
    }
    out_vals[r] = best.v;
    out_ids[r] = best.id;
  }
}

/* Greedy verification of [P4] item 1, from the gathered stats.
 * Request i has K_i = cu_num_draft[i+1] - cu_num_draft[i] drafts
 * draft_tokens[cu_num_draft[i] + j] and K_i + 1 target rows starting at row
 * b_i = cu_num_draft[i] + i (its K_i draft positions, then the bonus row).
 * Outputs: out_sampled[i * (max_k + 1) + j] = target argmax of row b_i + j
 * for j <= a_i, else -1; num_sampled = a_i + 1; num_rejected = K_i - a_i;
 * bonus = target argmax of row b_i + a_i.  target_ids (nullable) gets the
 * per-row global argmax ids.  in_prefill (nullable) marks the requests
 * still in prefill ([P4] Test Plan names "prefilling requests"; reading:
 * such a request emits nothing this step): sampled all -1, num_sampled =
 * num_rejected = 0, bonus = -1; its rows' target ids are still reported.
 * Returns 0; -1 if some K_i is outside [0, max_k] (nothing is written for
 * that request); -2 if out of memory. */
int oracle_greedy_verify(const oracle_stat *stats, int num_shards, int num_reqs,
                         const int32_t *cu_num_draft, const int32_t *draft_tokens,
                         int max_k, const uint8_t *in_prefill, int32_t *out_sampled,
                         int32_t *out_num_sampled, int32_t *out_num_rejected,
                         int32_t *out_bonus, int32_t *out_target_ids) {
  int status = 0;
  int64_t total_rows = (int64_t)cu_num_draft[num_reqs] + num_reqs;
  if (total_rows <= 0) return 0;
  /* step 1: the global argmax of every target row (the cross-shard reduce) */
  float *t_val = (float *)malloc((size_t)total_rows * sizeof(float));
  int32_t *t = (int32_t *)malloc((size_t)total_rows * sizeof(int32_t));
  if (!t_val || !t) {
    free(t_val);
    free(t);
    return -2;
  }
  oracle_shard_reduce(stats, num_shards, total_rows, t_val, t);
  if (out_target_ids) memcpy(out_target_ids, t, (size_t)total_rows * sizeof(int32_t));
  /* step 2: per request, accept while the draft equals the target argmax of
   * its position; emit the target argmaxes of positions 0..a */
  for (int i = 0; i < num_reqs; ++i) {
    int32_t c = cu_num_draft[i];
    int32_t k = cu_num_draft[i + 1] - c;
    int64_t b = (int64_t)c + i;
    if (k < 0 || k > max_k) {
      status = -1;
      continue;
    }
    if (in_prefill && in_prefill[i]) {
      for (int j = 0; j <= max_k; ++j) out_sampled[(int64_t)i * (max_k + 1) + j] = -1;
      out_num_sampled[i] = 0;
      out_num_rejected[i] = 0;
      out_bonus[i] = -1;
      continue;
    }
    int a = 0;
    while (a < k && draft_tokens[c + a] == t[b + a]) ++a;
    for (int j = 0; j <= max_k; ++j)
      out_sampled[(int64_t)i * (max_k + 1) + j] = (j <= a) ? t[b + j] : -1;
    out_num_sampled[i] = a + 1;
    out_num_rejected[i] = k - a;
    out_bonus[i] = t[b + a];
  }
  free(t_val);
  free(t);
  return status;
}

/* Draft-to-target id map of [P2] ("Refactor local argmax code"): after the
 * local argmax and the cross-shard reduce, a draft id k becomes
 * k + d2t[k].  Returns -1 if some id is outside [0, d2t_len). */
int oracle_d2t_map(const int32_t *draft_ids, int64_t n, const int64_t *d2t,
                   int64_t d2t_len, int32_t *out_target_ids) {
  int status = 0;
  for (int64_t r = 0; r < n; ++r) {
    int32_t k = draft_ids[r];
    if (k < 0 || k >= d2t_len) {
      status = -1;
      out_target_ids[r] = k;
      continue;
    }
    out_target_ids[r] = (int32_t)(k + d2t[k]);
  }
  return status;
}

/* Logits of the fused LM-head variant ([P4] Purpose, vocab-parallel LM head;
 * item 2 fused get_top_tokens): logit[r][j] = sum_k hidden[r][k] * weight[j][k]
 * for the ids of one shard, bf16 inputs widened exactly, accumulated in fp64
 * in k order.  out_logits is [n_sel][shard_width]. */
void oracle_lmhead_logits(const uint16_t *hidden, int64_t H, const uint16_t *weight,
                          int64_t shard_width, const int64_t *rows_sel, int64_t n_sel,
                          double *out_logits) {
  for (int64_t q = 0; q < n_sel; ++q) {
    const uint16_t *h = hidden + rows_sel[q] * H;
    double *out = out_logits + q * shard_width;
    int64_t j;
#pragma omp parallel for schedule(static)
    for (j = 0; j < shard_width; ++j) {
      const uint16_t *w = weight + j * H;
      double acc = 0.0;
      for (int64_t k = 0; k < H; ++k) {
        double a = (double)widen(h, ORACLE_BF16, k);
        double b = (double)widen(w, ORACLE_BF16, k);
        acc += a * b;
      }
      out[j] = acc;
    }
  }
}

/* Argmax over fp64 logits rows (from oracle_lmhead_logits) with the padding
 * mask and torch.argmax order, plus the largest value at any other id (top2)
 * for the tolerance gate.  Column j of a row is global id first + j. */
void oracle_argmax_f64(const double *logits, int64_t n_rows, int64_t width,
                       int64_t first, int64_t org_vocab, double *out_top1,
                       double *out_top2, int32_t *out_ids) {
  for (int64_t q = 0; q < n_rows; ++q) {
    const double *row = logits + q * width;
    int64_t best_j = 0;
    double best = (first >= org_vocab) ? -INFINITY : row[0];
    for (int64_t j = 1; j < width; ++j) {
      double c = (first + j >= org_vocab) ? -INFINITY : row[j];
      if (!isnan(best) && (isnan(c) || c > best)) {
        best = c;
        best_j = j;
      }
    }
    double second = -INFINITY;
    for (int64_t j = 0; j < width; ++j) {
      double c = (first + j >= org_vocab) ? -INFINITY : row[j];
      if (j != best_j && c > second) second = c;
    }
    out_top1[q] = best;
    out_top2[q] = second;
    out_ids[q] = (int32_t)(first + best_j);
  }
}

/* Number of threads the OpenMP loops above use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* OCP FP8 E4M3 (the "e4m3fn" variant) decoded exactly: sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6);
 * S.1111.111 is NaN; there is no infinity.  Every value is exact in double. */
static double e4m3_value(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 0xF, m = c & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

double oracle_e4m3_value(uint8_t c) { return e4m3_value(c); }

/* Logits of the fp8 LM-head variant: hidden and weight stored as E4M3 codes
 * with positive scales (one per hidden row, one per weight tensor):
 * logit[r][j] = hidden_scale[r] * weight_scale * sum_k dec(h[r][k]) * dec(w[j][k]),
 * products and the sum in fp64 in k order.  Positive scales do not change
 * which id is the argmax of a row, only the value. */
void oracle_lmhead_logits_fp8(const uint8_t *hidden, const float *hidden_scale, int64_t H,
                              const uint8_t *weight, double weight_scale, int64_t shard_width,
                              const int64_t *rows_sel, int64_t n_sel, double *out_logits) {
  double value[256]; /* e4m3_value of every code, looked up in the loops */
  for (int c = 0; c < 256; ++c) value[c] = e4m3_value((uint8_t)c);
  for (int64_t q = 0; q < n_sel; ++q) {
    const uint8_t *h = hidden + rows_sel[q] * H;
    const double scale = (double)hidden_scale[rows_sel[q]] * weight_scale;
    double *out = out_logits + q * shard_width;
    int64_t j;
#pragma omp parallel for schedule(static)
    for (j = 0; j < shard_width; ++j) {
      const uint8_t *w = weight + j * H;
      double acc = 0.0;
      for (int64_t k = 0; k < H; ++k) acc += value[h[k]] * value[w[k]];
      out[j] = scale * acc;
    }
  }
}

/* Number of fixed global blocks [b * block, (b + 1) * block) that meet the
 * shard [shard_start, shard_start + shard_width). */
int64_t oracle_block_count(int64_t shard_start, int64_t shard_width, int64_t block) {
  return (shard_start + shard_width - 1) / block - shard_start / block + 1;
}

/* Block-granular statistics of one shard ([P4] item 1: each rank reduces its
 * shard to per-block (max, id) statistics; the blocks keep the global
 * boundaries of the unsharded kernels, 8192 ids for draft positions and 1024
 * for the bonus position, also where a block straddles a shard edge).
 *
 * Row r uses block size B = draft_block, except the bonus row of a request
 * (row b_i + K_i with b_i = cu_num_draft[i] + i), which uses bonus_block;
 * cu_num_draft may be NULL, and then every row uses draft_block.  With
 * b0 = floor(shard_start / B), piece p of row r is the argmax (scan_row, the
 * same rule as a whole shard) over global ids
 *   [max(shard_start, (b0 + p) * B), min(shard_start + shard_width, (b0 + p + 1) * B)).
 * Every row has n_pieces slots, the larger of the two block counts
 * oracle_block_count(shard_start, shard_width, B), written to
 * out[p * rows + r]; the slots past the row's own piece count hold value
 * -inf with the shard's last id, which never wins the reduction because a
 * real piece precedes it.  (When one size divides the other the smaller
 * block has the larger count; 3 and 2 over ids [2, 4) show that it need not.)
 * Returns n_pieces, or -1 if a block size is not positive or cu_num_draft
 * does not describe `rows` rows. */
int64_t oracle_block_stats(const void *logits, int dtype, int64_t rows, int64_t ld,
                           int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                           int64_t draft_block, int64_t bonus_block, int num_reqs,
                           const int32_t *cu_num_draft, oracle_stat *out) {
  if (draft_block <= 0 || bonus_block <= 0) return -1;
  const int64_t n_draft = oracle_block_count(shard_start, shard_width, draft_block);
  const int64_t n_bonus = oracle_block_count(shard_start, shard_width, bonus_block);
  const int64_t n_pieces = n_draft > n_bonus ? n_draft : n_bonus;
  const int64_t shard_end = shard_start + shard_width;
  char *is_bonus = (char *)calloc((size_t)(rows > 0 ? rows : 1), 1);
  if (!is_bonus) return -1;
  if (cu_num_draft) {
    if ((int64_t)cu_num_draft[num_reqs] + num_reqs != rows) {
      free(is_bonus);
      return -1;
    }
    for (int i = 0; i < num_reqs; ++i) is_bonus[(int64_t)cu_num_draft[i + 1] + i] = 1;
  }
  int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
  for (r = 0; r < rows; ++r) {
    const char *row = (const char *)logits + r * ld * elt_size(dtype);
    const int64_t B = is_bonus[r] ? bonus_block : draft_block;
    const int64_t b0 = shard_start / B;
    const int64_t own = oracle_block_count(shard_start, shard_width, B);
    for (int64_t p = 0; p < n_pieces; ++p) {
      oracle_stat st;
      if (p < own) {
        int64_t lo = (b0 + p) * B, hi = (b0 + p + 1) * B;
        if (lo < shard_start) lo = shard_start;
        if (hi > shard_end) hi = shard_end;
        st.id = scan_row(row + (lo - shard_start) * elt_size(dtype), dtype, lo, hi - lo,
                         org_vocab, &st.v);
      } else {
        st.v = -INFINITY;
        st.id = (int32_t)(shard_end - 1);
      }
      out[p * rows + r] = st;
    }
  }
  free(is_bonus);
  return n_pieces;
}
