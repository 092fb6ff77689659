/*
 * sga.h -- C ABI of libsga.so: vocab-sharded greedy token selection for
 * speculative decoding, hand-written CUDA kernels for GB300 (sm_103a).
 *
 * The method (web pages, cited by title and section):
 *   vLLM PR #34049 "[Spec Decode] Reduce TP communication for speculative
 *     decoding draft token generation", Solution: each tensor-parallel rank
 *     takes the argmax of its own vocab shard, only (max_value, global_index)
 *     pairs are gathered, and a reduction across ranks gives the global
 *     argmax.
 *   vLLM PR #39419 "[SpecDecode] Reduce TP communication for large-vocab
 *     draft models speculative decoding", review "Refactor local argmax code":
 *     the draft-to-target id map target_id = k + d2t[k] is applied after the
 *     local argmax.
 *   vLLM PR #62604 (sharded greedy verification), Purpose item 1: per-shard
 *     statistics, all-gathered on dim 0, then ONE kernel for the global
 *     argmax, the acceptance, the bonus token and the sampled/rejected
 *     counts; item 2: the padding mask, "lowest id on ties, NaN wins, as
 *     torch.argmax"; vocabulary < 2^24.
 *
 * Tensor-parallel ranks are emulated on one GPU: shard s writes its stats to
 * rows [s*R, (s+1)*R) of one buffer, which is byte-for-byte what
 * all_gather(dim=0) of the per-rank [R] stats would produce.
 *
 * Conventions for every entry point:
 *   - Every pointer is a DEVICE pointer unless stated otherwise; the caller
 *     owns every buffer.  The library allocates no memory and keeps no state
 *     besides per-device cached kernel attributes, a device error word, and
 *     the merge slots of the decode-size LM head (see sga_lmhead_argmax).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.
 *   - Arguments are validated on the host BEFORE anything is launched; a
 *     negative SGA_ERR_* means nothing was enqueued.  SGA_ERR_CUDA means a
 *     launch failed (cudaGetLastError); the CUDA error is left for the caller
 *     to inspect through cudaGetLastError/cudaPeekAtLastError semantics.
 *   - Inputs are never written.  Outputs are fully written on success.
 *   - Comparison order ("argmax order"): NaN beats every number and the
 *     lowest-id NaN wins; among numbers the larger wins (+0 and -0 are equal);
 *     equal values resolve to the lower global id.  Ids at or past org_vocab
 *     are padding and count as -inf.  A row (or shard) with no value above
 *     -inf reports its first id with value -inf.  The reported value is the
 *     winning element widened exactly to fp32 (its own bits, NaN payload
 *     kept), or -inf for a padded winner.
 */
#ifndef SGA_H
#define SGA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SGA_VERSION 100 /* 1.0.0 */

/* One per-row statistic of one shard: 8 bytes, {fp32 value bits, int32 id}. */
typedef struct sga_stat {
  float v;
  int32_t id;
} sga_stat;

/* Logits element types. */
enum sga_dtype { SGA_F32 = 0, SGA_BF16 = 1 };

/* A cudaStream_t passed as an opaque pointer. */
typedef void *sga_stream;

/* Status codes (0 = success). */
enum sga_status {
  SGA_OK = 0,
  SGA_ERR_NULL = -1,        /* a required pointer is NULL */
  SGA_ERR_SIZE = -2,        /* a size or count is negative / out of range */
  SGA_ERR_SHARD = -3,       /* shard outside the vocab or wider than the row stride */
  SGA_ERR_VOCAB = -4,       /* org_vocab <= 0, or an id would reach 2^24 */
  SGA_ERR_DTYPE = -5,       /* unknown dtype */
  SGA_ERR_ALIGN = -6,       /* pointer not aligned as the entry point requires */
  SGA_ERR_WORKSPACE = -7,   /* workspace smaller than the *_workspace() size */
  SGA_ERR_MAXK = -8,        /* max_k outside [1, SGA_MAX_K] */
  SGA_ERR_CUDA = -9,        /* a CUDA runtime call or launch failed */
  SGA_ERR_DEVICE = -10,     /* the device has no sm_103 kernels (not a GB300) */
  SGA_ERR_UNSUPPORTED = -11 /* shape outside what the kernel supports */
};

/* Largest number of drafts per request the verify kernel handles. */
#define SGA_MAX_K 15

/* Largest id + 1 any entry point accepts (the pages' vocabulary bound). */
#define SGA_MAX_VOCAB (1 << 24)

/* Library version, SGA_VERSION of the build. */
int sga_version(void);

/* Static English text for a status code; never NULL. */
const char *sga_status_string(int status);

/*
 * sga_local_argmax -- per-shard argmax with the padding mask.
 * Page: vLLM PR #34049, Solution step 1 (local argmax on each TP rank's vocab
 * shard, index made global); vLLM PR #62604, Purpose item 2 (padding mask,
 * torch.argmax order) and item 1 (per-shard statistics).
 *
 *   logits       device, rows x (>= shard_width) elements of `dtype`, row
 *                stride `ld` ELEMENTS; points at the shard's first column,
 *                i.e. element (0, shard_start) of the full matrix, or at
 *                element 0 of a separate per-rank [rows, shard_width] buffer.
 *                Must be aligned to the element size.  Any row stride and
 *                any 16-byte misalignment of the rows is handled.
 *   dtype        SGA_F32 or SGA_BF16.
 *   rows         >= 0; 0 enqueues nothing and returns SGA_OK.
 *   ld           >= shard_width.
 *   shard_start  global id of column 0 of the shard (>= 0).
 *   shard_width  > 0; shard_start + shard_width <= SGA_MAX_VOCAB.
 *   org_vocab    1 .. SGA_MAX_VOCAB; global ids >= org_vocab are padding.
 *   out_stats    device, `rows` entries, 8-byte aligned: out_stats[r] =
 *                argmax (value, GLOBAL id) of row r over the shard.  To
 *                emulate the dim-0 all-gather pass stats + s*rows.
 * Reads each non-padding logit of the shard once; padding ids are not read.
 */
int sga_local_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                     int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                     sga_stat *out_stats, sga_stream stream);

/*
 * sga_local_argmax_shards -- sga_local_argmax for several shards of one
 * logits buffer in a single launch (one GPU holding the vocab slices of
 * several tensor-parallel ranks).  Same statistics, same layout: shard s of
 * row r goes to out_stats[s*rows + r], exactly the dim-0 all-gather order.
 * Page: as sga_local_argmax (vLLM PR #34049, Solution; vLLM PR #62604,
 * Purpose items 1-2 and Test Plan: TP ranks emulated in one process with the
 * per-shard statistics concatenated in rank order).
 *
 *   logits        device; element (r, 0) holds global id shard_starts[0] of
 *                 row r; global id g sits at column g - shard_starts[0].
 *   num_shards    1 .. 64.
 *   shard_starts, shard_widths   HOST arrays of num_shards entries; shards
 *                 ascending and non-overlapping (shard_starts[s] >=
 *                 shard_starts[s-1] + shard_widths[s-1]); every width > 0;
 *                 the last shard must end at or before column ld.
 *   rows          0 .. 2^28 / num_shards.
 *   out_stats     device, num_shards * rows entries, 8-byte aligned.
 * Other arguments and the errors as sga_local_argmax.
 */
int sga_local_argmax_shards(const void *logits, int dtype, int64_t rows, int64_t ld,
                            int num_shards, const int64_t *shard_starts,
                            const int64_t *shard_widths, int64_t org_vocab,
                            sga_stat *out_stats, sga_stream stream);

/*
 * sga_block_slots -- statistics per row that sga_local_argmax_blocks writes
 * for one shard: the larger of the numbers of fixed global blocks of
 * draft_block and of bonus_block ids that meet [shard_start, shard_start +
 * shard_width).  Returns that count (>= 1), or a negative SGA_ERR_* for an
 * invalid shard or block size.  Pure host arithmetic, no CUDA call.
 */
int64_t sga_block_slots(int64_t shard_start, int64_t shard_width, int64_t draft_block,
                        int64_t bonus_block);

/*
 * sga_local_argmax_blocks -- block-granular statistics of one shard: for
 * every row, the argmax (value, GLOBAL id) of each fixed global block of ids
 * [b*B, (b+1)*B) that meets the shard, clipped to the shard; a block that
 * straddles a shard edge gives one piece on each side.
 * Page: vLLM PR #62604, Purpose item 1 (each rank reduces its shard to
 * per-block (max, token id) statistics; the blocks keep the unsharded
 * kernels' global boundaries, 8192 ids for draft positions and 1024 for the
 * bonus position, also across shard edges, so ties resolve as on the full
 * logits).
 *
 *   logits, dtype, rows, ld, shard_start, shard_width, org_vocab
 *                 as sga_local_argmax (rows <= 2^28 / slots).
 *   draft_block   block size B of the draft rows, 1 .. SGA_MAX_VOCAB.
 *   bonus_block   block size of the bonus rows, 1 .. SGA_MAX_VOCAB.
 *   num_reqs, cu_num_draft   the request layout of sga_greedy_verify
 *                 (device int32 [num_reqs + 1]; rows == cu_num_draft[num_reqs]
 *                 + num_reqs is a precondition).  Row cu_num_draft[i+1] + i
 *                 is the bonus row of request i.  cu_num_draft may be NULL:
 *                 then every row is a draft row and num_reqs is ignored.
 *   out_stats     device, slots * rows entries, 8-byte aligned, with slots =
 *                 sga_block_slots(shard_start, shard_width, draft_block,
 *                 bonus_block).  Piece p of row r (ascending ids) goes to
 *                 out_stats[p*rows + r]; a row with fewer pieces than slots
 *                 (the rows whose block size gives the smaller count) gets
 *                 (-inf, shard_start + shard_width - 1) in its remaining
 *                 slots, which never wins a reduction.  An all-padding piece
 *                 reports (-inf, its first id).
 * The stats of all shards, concatenated in shard order, go to
 * sga_shard_reduce or sga_greedy_verify with num_shards = the sum of the
 * shards' slots (at most 4096) and give the same ids as per-shard stats.
 * Errors as sga_local_argmax, plus SGA_ERR_SIZE for a block size out of range.
 */
int sga_local_argmax_blocks(const void *logits, int dtype, int64_t rows, int64_t ld,
                            int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                            int64_t draft_block, int64_t bonus_block, int num_reqs,
                            const int32_t *cu_num_draft, sga_stat *out_stats,
                            sga_stream stream);

/*
 * sga_local_argmax_blocks_shards -- sga_local_argmax_blocks for several
 * shards of one logits buffer in a single launch (one GPU holding the vocab
 * slices of several tensor-parallel ranks), as sga_local_argmax_shards is
 * for per-shard statistics.  Shard s's slots follow shard s-1's: with
 * slots_s = sga_block_slots(starts[s], widths[s], draft_block, bonus_block),
 * piece p of row r of shard s goes to out_stats[(slots_0 + ... + slots_{s-1}
 * + p) * rows + r], exactly what concatenating the per-shard calls' outputs
 * in shard order gives.
 * Page: as sga_local_argmax_blocks (vLLM PR #62604, Purpose item 1).
 *
 *   logits        device; element (r, 0) holds global id shard_starts[0] of
 *                 row r; global id g sits at column g - shard_starts[0].
 *   num_shards    1 .. 64.
 *   shard_starts, shard_widths   HOST arrays, shards ascending and
 *                 non-overlapping; the last shard ends at or before column ld.
 *   rows          0 .. 2^28 / (total slots).
 *   out_stats     device, (total slots) * rows entries, 8-byte aligned.
 * Other arguments and the errors as sga_local_argmax_blocks.
 */
int sga_local_argmax_blocks_shards(const void *logits, int dtype, int64_t rows, int64_t ld,
                                   int num_shards, const int64_t *shard_starts,
                                   const int64_t *shard_widths, int64_t org_vocab,
                                   int64_t draft_block, int64_t bonus_block, int num_reqs,
                                   const int32_t *cu_num_draft, sga_stat *out_stats,
                                   sga_stream stream);

/*
 * sga_shard_reduce -- global argmax from the gathered shard statistics,
 * optionally mapped from draft ids to target ids.
 * Page: vLLM PR #34049, Solution step 3 (reduce across ranks to the global
 * argmax); vLLM PR #62604, Purpose item 2 (dim-0 all-gather layout, same
 * result as torch.argmax); vLLM PR #39419, "Refactor local argmax code"
 * (target_id = k + draft_id_to_target_id[k], after the local argmax).
 *
 *   stats       device, num_shards * rows entries, shard-major
 *               (stats[s*rows + r]); shards in ascending id order.
 *   num_shards  1 .. 4096.
 *   rows        >= 0 (0: nothing enqueued).
 *   out_vals    device fp32 [rows] (nullable): value of the winner.
 *   out_ids     device int32 [rows]: global id of the winner, after d2t.
 *   d2t         device int64 [d2t_len] or NULL.  When given, out_ids[r] =
 *               k + d2t[k] for the winning id k; an id outside [0, d2t_len)
 *               is left unmapped and sets the device error word (see
 *               sga_device_error).
 */
int sga_shard_reduce(const sga_stat *stats, int num_shards, int64_t rows, float *out_vals,
                     int32_t *out_ids, const int64_t *d2t, int64_t d2t_len,
                     sga_stream stream);

/*
 * sga_greedy_verify -- one fused kernel: cross-shard reduce of every target
 * row, greedy acceptance, bonus token and sampled/rejected counts.
 * Page: vLLM PR #62604, Purpose item 1 (one kernel finishes the global
 * argmax, acceptance, bonus token and sampled/rejected counts) and Test Plan
 * (compared with rejection_sample + get_num_sampled_and_rejected on the full
 * logits; placeholder drafts).
 *
 *   stats          device, num_shards * R_tot entries, shard-major, where
 *                  R_tot = cu_num_draft[num_reqs] + num_reqs.
 *   num_shards     1 .. 4096.
 *   num_reqs       >= 0 (0: nothing enqueued).
 *   cu_num_draft   device int32 [num_reqs + 1], cu[0] = 0, non-decreasing:
 *                  request i has K_i = cu[i+1] - cu[i] drafts and owns target
 *                  rows b_i .. b_i + K_i with b_i = cu[i] + i (K_i draft
 *                  positions, then its bonus row).  K_i must lie in
 *                  [0, max_k]; a request that breaks this gets num_sampled =
 *                  num_rejected = 0, bonus = -1, sampled all -1, and the
 *                  device error word is set.
 *   draft_tokens   device int32 [cu[num_reqs]] (may be NULL when every K_i is
 *                  0).  A negative id is a placeholder and never matches.
 *   max_k          1 .. SGA_MAX_K: row length - 1 of out_sampled.
 *   out_sampled    device int32 [num_reqs, max_k + 1]: with a_i = number of
 *                  leading drafts equal to the target argmax of their row,
 *                  entries 0..a_i are the target argmaxes of rows
 *                  b_i .. b_i + a_i, the rest -1.
 *   out_num_sampled, out_num_rejected   device int32 [num_reqs]: a_i + 1 and
 *                  K_i - a_i.
 *   out_bonus      device int32 [num_reqs]: the last emitted token, the target
 *                  argmax of row b_i + a_i.
 *   out_target_ids device int32 [R_tot] or NULL: every row's global argmax.
 * All int32 pointers must be 4-byte aligned, stats 8-byte aligned.
 */
int sga_greedy_verify(const sga_stat *stats, int num_shards, int num_reqs,
                      const int32_t *cu_num_draft, const int32_t *draft_tokens, int max_k,
                      int32_t *out_sampled, int32_t *out_num_sampled,
                      int32_t *out_num_rejected, int32_t *out_bonus,
                      int32_t *out_target_ids, sga_stream stream);

/*
 * sga_greedy_verify_prefill -- sga_greedy_verify for a batch that mixes
 * decoding requests with requests still in prefill.
 * Page: vLLM PR #62604, Test Plan (the sharded verifier handles "prefilling
 * requests").  The pages do not say what such a request yields; this library
 * reads it as: a request still in prefill emits nothing this step.
 *
 *   in_prefill     device uint8 [num_reqs] or NULL (NULL = sga_greedy_verify):
 *                  nonzero marks request i as still in prefill.  Such a
 *                  request gets out_sampled row all -1, out_num_sampled =
 *                  out_num_rejected = 0 and out_bonus = -1; the target
 *                  argmaxes of its rows still go to out_target_ids.  Its
 *                  K_i must still lie in [0, max_k] (else the K_i error
 *                  result of sga_greedy_verify applies).
 * Other arguments, results and errors as sga_greedy_verify.
 */
int sga_greedy_verify_prefill(const sga_stat *stats, int num_shards, int num_reqs,
                              const int32_t *cu_num_draft, const int32_t *draft_tokens,
                              const uint8_t *in_prefill, int max_k, int32_t *out_sampled,
                              int32_t *out_num_sampled, int32_t *out_num_rejected,
                              int32_t *out_bonus, int32_t *out_target_ids, sga_stream stream);

/*
 * sga_lmhead_argmax -- fused LM-head GEMM + per-shard argmax: the shard's
 * logits hidden . weight_shard^T are computed on the tensor cores (tcgen05,
 * fp32 accumulation in tensor memory) and reduced to per-row statistics in
 * the epilogue; the logits are never written to global memory.
 * Page: vLLM PR #62604, Purpose (vocab-parallel LM head: each rank holds a
 * vocab slice of the weight) and item 2 (fused get_top_tokens); vLLM PR
 * #39419, Changes (get_top_tokens on the model: lm_head applied to the hidden
 * states, then the local argmax).
 *
 *   hidden        device bf16 [M, H] row-major (row stride H), 16-byte aligned.
 *   M             0 .. 1048576 (0: nothing enqueued).
 *   H             hidden size: a positive multiple of 64.
 *   weight_shard  device bf16 [shard_width, H] row-major, 16-byte aligned; row j
 *                 holds global id shard_start + j.
 *   shard_start, shard_width, org_vocab   as for sga_local_argmax.
 *   out_stats     device [M], 8-byte aligned: argmax (value, global id) of
 *                 each row's logits over the shard.  The value is the fp32
 *                 accumulator of the winning logit; accumulation order is
 *                 the kernel's, so values match an exact dot product only to
 *                 fp32 rounding and near-ties may resolve to either id.
 *   workspace     device, >= sga_lmhead_argmax_workspace(M, shard_width)
 *                 bytes, 8-byte aligned; holds partial statistics.
 *                 Contents on entry are ignored; the caller must not use it
 *                 concurrently from two calls.  Unused for M <= 128.
 * Decode sizes (M <= 128; one CTA per SM up to M = 64, CTA pairs above):
 * one kernel launch, whose CTAs merge their per-row
 * winners in library-owned device memory (32 merge slots per device, one
 * taken per call in turn; the last CTA writes out_stats and clears the
 * slot).  Calls whose kernels overlap on the GPU must not share a slot: at
 * most 32 decode-size LM-head calls (of any LM-head entry point) may be in
 * flight on one device at once, and a captured graph that holds such a call
 * must not be replayed concurrently with itself.
 * Requires a GPU of compute capability 10.3 (SGA_ERR_DEVICE otherwise).
 */
size_t sga_lmhead_argmax_workspace(int64_t M, int64_t shard_width);
int sga_lmhead_argmax(const void *hidden, int64_t M, int64_t H, const void *weight_shard,
                      int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                      sga_stat *out_stats, void *workspace, size_t workspace_bytes,
                      sga_stream stream);

/*
 * sga_lmhead_argmax_fp8 -- sga_lmhead_argmax with FP8 (OCP E4M3, "e4m3fn")
 * operands: hidden states and the weight shard stored as E4M3 codes (one byte
 * each) with a positive scale per hidden row and one positive weight scale.
 * logit[r][j] = hidden_scale[r] * weight_scale * sum_k h[r][k] * w[j][k].
 * Positive scales cannot change which id is the argmax of a row, so the
 * tensor cores (tcgen05 kind::f8f6f4, fp32 accumulation) work on the raw
 * codes and only the reported value is scaled.
 * Page: as sga_lmhead_argmax (vLLM PR #62604, Purpose; PR #39419, Changes);
 * FP8 models are the pages' workloads (vLLM PR #34049, Test Plan:
 * Llama 4 Maverick FP8), an fp8 LM head is this library's extension.
 *
 *   hidden_q      device uint8 [M, H] E4M3 codes, 16-byte aligned.
 *   hidden_scale  device fp32 [M] (nullable: all 1), 4-byte aligned; each
 *                 scale must be positive and finite (not checked).
 *   H             a positive multiple of 128.
 *   weight_q      device uint8 [shard_width, H] E4M3 codes, 16-byte aligned.
 *   weight_scale  host value, positive and finite (SGA_ERR_SIZE otherwise).
 *   workspace     as sga_lmhead_argmax (same size function).
 * The reported value is fp32(acc) * (hidden_scale[r] * weight_scale).
 */
int sga_lmhead_argmax_fp8(const void *hidden_q, const float *hidden_scale, int64_t M, int64_t H,
                          const void *weight_q, float weight_scale, int64_t shard_start,
                          int64_t shard_width, int64_t org_vocab, sga_stat *out_stats,
                          void *workspace, size_t workspace_bytes, sga_stream stream);

/*
 * sga_lmhead_argmax_shards -- sga_lmhead_argmax for several vocab shards of
 * one weight buffer in a single call (one GPU holding the vocab slices of
 * several tensor-parallel ranks), as sga_local_argmax_shards is for the
 * per-shard argmax.  At decode sizes (M <= 128) every shard runs in one
 * launch of a decode-size kernel, whose CTAs merge in library-owned memory
 * as in sga_lmhead_argmax (same 32-call limit); from M = 129 every shard
 * runs in one GEMM launch followed by one finalize launch.  The statistics
 * are identical to num_shards sga_lmhead_argmax calls.
 * Page: as sga_lmhead_argmax (vLLM PR #62604, Purpose; PR #39419, Changes).
 *
 *   weight        device [rows, H] (bf16), 16-byte aligned; row g -
 *                 shard_starts[0] holds global id g (the buffer spans every
 *                 shard, and any gap between them).
 *   num_shards    1 .. 64.
 *   shard_starts, shard_widths   HOST arrays, shards ascending and
 *                 non-overlapping, each as sga_lmhead_argmax's.
 *   out_stats     device, num_shards * M entries, 8-byte aligned: shard s's
 *                 stats at out_stats[s * M + r] (the gathered layout).
 *   workspace     device, >= sga_lmhead_argmax_shards_workspace(M,
 *                 num_shards, shard_widths) bytes, 8-byte aligned, as
 *                 sga_lmhead_argmax's.
 * Other arguments and the errors as sga_lmhead_argmax.
 */
size_t sga_lmhead_argmax_shards_workspace(int64_t M, int num_shards, const int64_t *shard_widths);
int sga_lmhead_argmax_shards(const void *hidden, int64_t M, int64_t H, const void *weight,
                             int num_shards, const int64_t *shard_starts,
                             const int64_t *shard_widths, int64_t org_vocab,
                             sga_stat *out_stats, void *workspace, size_t workspace_bytes,
                             sga_stream stream);

/*
 * sga_lmhead_argmax_shards_fp8 -- sga_lmhead_argmax_shards with the E4M3
 * operands of sga_lmhead_argmax_fp8: one weight_scale for the whole weight
 * buffer; otherwise as sga_lmhead_argmax_fp8 and sga_lmhead_argmax_shards.
 */
int sga_lmhead_argmax_shards_fp8(const void *hidden_q, const float *hidden_scale, int64_t M,
                                 int64_t H, const void *weight_q, float weight_scale,
                                 int num_shards, const int64_t *shard_starts,
                                 const int64_t *shard_widths, int64_t org_vocab,
                                 sga_stat *out_stats, void *workspace, size_t workspace_bytes,
                                 sga_stream stream);

/*
 * sga_lmhead_argmax_noalloc -- sga_lmhead_argmax for callers that must not
 * allocate device memory.  The pages have no counterpart to this entry point.
 *
 * Some callers of this code cannot call cudaMalloc on their decode path: an
 * inference server or framework plugin that owns a device memory pool sized
 * at start-up and forbids allocations outside it, or a latency-critical loop
 * where cudaMalloc/cudaFree would synchronise the device.  Such a caller may
 * have no way to provide the workspace that sga_lmhead_argmax needs.  This
 * entry point takes the same inputs and outputs but keeps its per-tile
 * partial statistics in a fixed scratch array inside the library's device
 * image (SGA_LMHEAD_NOALLOC_SCRATCH_BYTES = 4 MiB, held on every GPU that
 * loads the library until the process exits).  It calls no allocating
 * routine.
 *
 *   Arguments and results: as sga_lmhead_argmax, without workspace.
 *   Limit: sga_lmhead_argmax_workspace(M, shard_width) must not exceed
 *          SGA_LMHEAD_NOALLOC_SCRATCH_BYTES (M * P * 8 bytes, P partials per
 *          row: for M >= 129 P = min(ceil(shard_width / 256), 128); for
 *          M <= 128, where the scratch is not used, P =
 *          max(ceil(shard_width / 256), min(ceil(shard_width / 128), 256)));
 *          larger calls return SGA_ERR_WORKSPACE and enqueue nothing.
 *   Set-up: the first call on a device looks up the device address of the
 *          scratch array for that device (with that device current), so make
 *          the first call on each device before any stream capture.  The
 *          address is looked up again when the device's current context has
 *          changed (after cudaDeviceReset, for instance); make the first call
 *          after such a change outside any stream capture as well.
 *   Sharing: every call on a device uses the same scratch array, which keeps
 *          the last call's contents; each call writes every scratch entry it
 *          reads, so nothing has to start at zero.  Calls whose kernels
 *          overlap on the GPU (different streams, no ordering between them)
 *          race on the scratch array and may return wrong results.
 */
#define SGA_LMHEAD_NOALLOC_SCRATCH_BYTES (4u << 20)
int sga_lmhead_argmax_noalloc(const void *hidden, int64_t M, int64_t H,
                              const void *weight_shard, int64_t shard_start,
                              int64_t shard_width, int64_t org_vocab, sga_stat *out_stats,
                              sga_stream stream);

/*
 * Device error word of the current device.  Kernels OR bits into it instead
 * of trapping: SGA_DEVERR_K_RANGE (a request's K_i outside [0, max_k]),
 * SGA_DEVERR_D2T_RANGE (a winning id outside the d2t table),
 * SGA_DEVERR_TIMEOUT (a bounded wait inside a pipelined kernel gave up; its
 * outputs are not valid), SGA_DEVERR_LAYOUT (sga_local_argmax_blocks[_shards]:
 * a request of cu_num_draft names rows outside [0, rows) or ends before it
 * starts; that request's statistics are not written, and with a decreasing
 * cu_num_draft the other requests' statistics are not valid either).  sga_device_error synchronises the current device
 * and copies the word to *out_word (host pointer); sga_clear_device_error
 * synchronises and zeroes it.  Both return SGA_OK or SGA_ERR_CUDA.
 */
#define SGA_DEVERR_K_RANGE 1u
#define SGA_DEVERR_D2T_RANGE 2u
#define SGA_DEVERR_TIMEOUT 4u
#define SGA_DEVERR_LAYOUT 8u
int sga_device_error(uint32_t *out_word);
int sga_clear_device_error(void);

/*
 * sga_selftest_wait_timeout -- exercises the bounded-wait path that every
 * pipelined kernel of this library uses (the pages have no counterpart): one
 * thread waits on a shared-memory mbarrier that nothing arrives at; after
 * limit_ns (1 us .. 1 s) the wait gives up, SGA_DEVERR_TIMEOUT is OR-ed into
 * the device error word and the kernel returns normally.  waited_ns (device,
 * nullable, 8-byte aligned) receives the time the wait took.  The context stays
 * usable: no trap, no fault.
 */
int sga_selftest_wait_timeout(uint64_t limit_ns, uint64_t *waited_ns, sga_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* SGA_H */
