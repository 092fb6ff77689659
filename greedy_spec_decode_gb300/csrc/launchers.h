// launchers.h -- host-side launchers of the sga kernels (one per .cu file),
// called by sga_abi.cu after it has validated the arguments.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sga.h"

namespace sga {

// Key of the CUDA context current on the calling thread (0 while none is
// current).  What the library caches per device -- symbol addresses, function
// attributes -- belongs to one context; an entry whose key differs from the
// current one is looked up again, so a device reset (which destroys the
// context and reloads the module) or a different context never meets a
// stale address.
uintptr_t current_context_key();

// ---------------------------------------------------------------------------
// Launchers (host).  Arguments are already validated by sga_abi.cu.
// ---------------------------------------------------------------------------
cudaError_t launch_local_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                                int64_t shard_start, int64_t width, int64_t valid,
                                sga_stat *out, int num_sms, uint32_t *err, cudaStream_t stream);

// Several shards of one logits buffer in one launch: shard s covers global
// ids [starts[s], starts[s] + ...) held at column cols[s] of `logits`, with
// valids[s] non-padding ids; its stats go to out[s * rows + r].
constexpr int kMaxShardsPerLaunch = 64;
cudaError_t launch_local_argmax_table(const void *logits, int dtype, int64_t rows, int64_t ld,
                                      int num_shards, const int64_t *starts,
                                      const int64_t *cols, const int64_t *valids, sga_stat *out,
                                      int num_sms, uint32_t *err, cudaStream_t stream);

// Block-granular statistics of one shard (blocks.cu).
int64_t block_count(int64_t shard_start, int64_t shard_width, int64_t block);
int64_t block_slots(int64_t shard_start, int64_t shard_width, int64_t draft_block,
                    int64_t bonus_block);
constexpr int kMaxBlockShards = 64;
// Several shards of one logits buffer in one launch: shard s covers global
// ids [starts[s], starts[s] + widths[s]) held at column cols[s] of `logits`;
// its slots follow the previous shards' slots in the gathered statistics.
cudaError_t launch_block_argmax_table(const void *logits, int dtype, int64_t rows, int64_t ld,
                                      int num_shards, const int64_t *starts, const int64_t *cols,
                                      const int64_t *widths, int64_t org_vocab,
                                      int64_t draft_block, int64_t bonus_block, int num_reqs,
                                      const int32_t *cu_num_draft, sga_stat *out, int num_sms,
                                      uint32_t *err, cudaStream_t stream);
cudaError_t launch_block_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                                int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                                int64_t draft_block, int64_t bonus_block, int num_reqs,
                                const int32_t *cu_num_draft, sga_stat *out, int num_sms,
                                uint32_t *err, cudaStream_t stream);

cudaError_t launch_shard_reduce(const sga_stat *stats, int num_shards, int64_t rows,
                                float *out_vals, int32_t *out_ids, const int64_t *d2t,
                                int64_t d2t_len, uint32_t *err, cudaStream_t stream);

cudaError_t launch_greedy_verify(const sga_stat *stats, int num_shards, int num_reqs,
                                 const int32_t *cu_num_draft, const int32_t *draft_tokens,
                                 int max_k, int32_t *out_sampled, int32_t *out_num_sampled,
                                 int32_t *out_num_rejected, int32_t *out_bonus,
                                 int32_t *out_target_ids, uint32_t *err, cudaStream_t stream,
                                 const uint8_t *in_prefill = nullptr);

size_t lmhead_workspace_bytes(int64_t M, int64_t width);
// fp8 = false: bf16 hidden/weight (row_scale, w_scale unused).  fp8 = true:
// E4M3 codes; the reported values are scaled by row_scale[r] (nullable: 1)
// times w_scale.
cudaError_t launch_lmhead_argmax(const void *hidden, int64_t M, int64_t H, const void *weight,
                                 int64_t shard_start, int64_t width, int64_t valid,
                                 sga_stat *out, void *workspace, int num_sms, uint32_t *err,
                                 cudaStream_t stream, bool fp8 = false,
                                 const float *row_scale = nullptr, float w_scale = 1.0f);


// Shards of one LM-head launch, at most.
constexpr int kMaxLmShards = 64;

// Fused LM head + argmax of several shards of one weight buffer (row 0 =
// global id starts[0]; shards ascending): stats of shard s to out[s * M ..];
// one decode launch for M <= 128 (the CTAs merge in-kernel), else one GEMM
// launch and one finalize for every shard.  Workspace:
// lmhead_shards_workspace_bytes.
cudaError_t launch_lmhead_argmax_shards(const void *hidden, int64_t M, int64_t H,
                                        const void *weight, int num_shards,
                                        const int64_t *starts, const int64_t *widths,
                                        const int64_t *valids, sga_stat *out, void *workspace,
                                        int num_sms, uint32_t *err, cudaStream_t stream,
                                        bool fp8 = false, const float *row_scale = nullptr,
                                        float w_scale = 1.0f);
size_t lmhead_shards_workspace_bytes(int64_t M, int num_shards, const int64_t *widths);

// Decode-size LM head (lmhead_decode.cu), M <= 128, over num_shards shards in
// one launch: shard s covers global ids [starts[s], starts[s] + valids[s])
// at weight rows row0s[s] .. (ascending shards).  The CTAs merge their
// winners in library-owned memory and the last one writes the statistics of
// shard s, row r to out[s * M + r] (values scaled by row_scale[r] * w_scale
// when fp8).  *launched is false when no shard has a valid id (nothing is
// launched and out is not written).
cudaError_t launch_lmhead_decode(bool fp8, const void *hidden, int64_t M, int64_t H,
                                 const void *weight, int num_shards, const int64_t *starts,
                                 const int64_t *row0s, const int64_t *valids, sga_stat *out,
                                 const float *row_scale, float w_scale, int num_sms,
                                 uint32_t *err, cudaStream_t stream, bool *launched);

// Bounded-wait self-test (lmhead.cu).
cudaError_t launch_selftest_timeout(unsigned long long limit_ns, uint32_t *err,
                                    unsigned long long *waited_ns, cudaStream_t stream);

// Scratch of the no-allocation LM-head entry point (lmhead.cu): its size and
// the device address of the array on the current device.
size_t lmhead_noalloc_scratch_bytes();
cudaError_t lmhead_noalloc_scratch(sga_stat **out);

}  // namespace sga
