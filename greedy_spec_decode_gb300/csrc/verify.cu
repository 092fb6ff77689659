// verify.cu -- fused cross-shard reduce + greedy verification.
//
// vLLM PR #62604, Purpose item 1: the gathered per-shard statistics go into
// one kernel that finishes the global argmax, the acceptance, the bonus token
// and the sampled/rejected counts.  Readings (the pages name these outputs but
// do not define them): a draft is accepted while it equals the target argmax
// of its own row; with a accepted drafts the request emits the target
// argmaxes of rows 0..a, num_sampled = a + 1, num_rejected = K - a, and the
// bonus token is the last emitted one.
//
// Layout: 16 lanes per request (K <= 15, so K + 1 <= 16 rows), two requests
// per warp.  Lane j reduces row j of its request over the shards, compares
// with draft j, and one ballot gives the first mismatch.  The work is a few
// bytes per row, so the kernel is latency-bound; it exists to keep the whole
// verify step in one launch.
#include "common.cuh"

namespace sga {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    greedy_verify_kernel(const sga_stat *__restrict__ stats, int num_shards, int num_reqs,
                         const int32_t *__restrict__ cu_num_draft,
                         const int32_t *__restrict__ draft_tokens, int max_k,
                         int32_t *__restrict__ out_sampled, int32_t *__restrict__ out_num_sampled,
                         int32_t *__restrict__ out_num_rejected, int32_t *__restrict__ out_bonus,
                         int32_t *__restrict__ out_target_ids, uint32_t *err) {
  pdl_wait();  // the stats of the previous kernels in the stream are visible
  const int lane = threadIdx.x & 31;
  const int group = lane >> 4;  // request slot within the warp
  const int j = lane & 15;      // row (draft position) within the request
  const int64_t req = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 4;
  const bool live = req < num_reqs;
  const int64_t total_rows = static_cast<int64_t>(cu_num_draft[num_reqs]) + num_reqs;

  int32_t c = 0, k = 0;
  if (live) {
    c = cu_num_draft[req];
    k = cu_num_draft[req + 1] - c;
  }
  const bool bad = live && (k < 0 || k > max_k);
  const bool has_row = live && !bad && j <= k;

  int32_t t = -1;
  bool mismatch = false;
  if (has_row) {
    const int64_t row = static_cast<int64_t>(c) + req + j;
    sga_stat b = stats[row];
    for (int s = 1; s < num_shards; ++s) {
      const sga_stat cand = stats[static_cast<int64_t>(s) * total_rows + row];
      if (scan_better(cand.v, b.v)) b = cand;
    }
    t = b.id;
    if (out_target_ids) out_target_ids[row] = t;
    if (j < k) mismatch = draft_tokens[c + j] != t;
  }
  const uint32_t ballot = __ballot_sync(0xffffffffu, mismatch);
  const uint32_t mine = (ballot >> (group * 16)) & 0xffffu;
  const int a = mine ? __ffs(mine) - 1 : k;  // accepted drafts

  if (!live) return;
  int32_t *sampled_row = out_sampled + req * (max_k + 1);
  if (bad) {
    if (j <= max_k) sampled_row[j] = -1;
    if (j == 0) {
      out_num_sampled[req] = 0;
      out_num_rejected[req] = 0;
      out_bonus[req] = -1;
      atomicOr(err, SGA_DEVERR_K_RANGE);
    }
    return;
  }
  if (j <= max_k) sampled_row[j] = j <= a ? t : -1;
  if (j == a) out_bonus[req] = t;
  if (j == 0) {
    out_num_sampled[req] = a + 1;
    out_num_rejected[req] = k - a;
  }
}

}  // namespace

cudaError_t launch_greedy_verify(const sga_stat *stats, int num_shards, int num_reqs,
                                 const int32_t *cu_num_draft, const int32_t *draft_tokens,
                                 int max_k, int32_t *out_sampled, int32_t *out_num_sampled,
                                 int32_t *out_num_rejected, int32_t *out_bonus,
                                 int32_t *out_target_ids, uint32_t *err, cudaStream_t stream) {
  const int64_t threads_needed = static_cast<int64_t>(num_reqs) * 16;
  const unsigned blocks = static_cast<unsigned>((threads_needed + kThreads - 1) / kThreads);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, greedy_verify_kernel, stats, num_shards, num_reqs, cu_num_draft,
                            draft_tokens, max_k, out_sampled, out_num_sampled, out_num_rejected,
                            out_bonus, out_target_ids, err);
}

}  // namespace sga
