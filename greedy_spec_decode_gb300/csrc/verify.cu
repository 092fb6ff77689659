// verify.cu -- fused cross-shard reduce + greedy verification.
//
// vLLM PR #62604, Purpose item 1: the gathered per-shard statistics go into
// one kernel that finishes the global argmax, the acceptance, the bonus token
// and the sampled/rejected counts.  Readings (the pages name these outputs but
// do not define them): a draft is accepted while it equals the target argmax
// of its own row; with a accepted drafts the request emits the target
// argmaxes of rows 0..a, num_sampled = a + 1, num_rejected = K - a, and the
// bonus token is the last emitted one.  A request flagged as still in prefill
// (Test Plan: "prefilling requests") emits nothing: sampled all -1, both
// counts 0, bonus -1; its rows' target ids are still reported.
//
// Layout: 16 lanes per request (K <= 15, so K + 1 <= 16 rows), two requests
// per warp.  Lane j reduces row j of its request over the gathered statistics
// (one entry per shard, or per block piece of block-granular statistics), compares
// with draft j, and one ballot gives the first mismatch.  The work is a few
// bytes per row, so the kernel is latency-bound; it exists to keep the whole
// verify step in one launch.
#include "common.cuh"
#include "scan.cuh"

namespace sga {
namespace {

constexpr int kThreads = 256;
// Above this many statistics per row the wide kernel (a warp per row) is used.
#ifndef SGA_VERIFY_WIDE_ENTRIES
#define SGA_VERIFY_WIDE_ENTRIES 16
#endif
constexpr int kWideEntries = SGA_VERIFY_WIDE_ENTRIES;

__global__ void __launch_bounds__(kThreads)
    greedy_verify_kernel(const sga_stat *__restrict__ stats, int num_shards, int num_reqs,
                         const int32_t *__restrict__ cu_num_draft,
                         const int32_t *__restrict__ draft_tokens,
                         const uint8_t *__restrict__ in_prefill, int max_k,
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
  bool prefill = false;
  if (live) {
    c = cu_num_draft[req];
    k = cu_num_draft[req + 1] - c;
    prefill = in_prefill != nullptr && in_prefill[req] != 0;
  }
  const bool bad = live && (k < 0 || k > max_k);
  const bool has_row = live && !bad && j <= k;

  int32_t t = -1;
  bool mismatch = false;
  if (has_row) {
    const int64_t row = static_cast<int64_t>(c) + req + j;
    // the draft is loaded before the statistics so that both loads overlap
    const int32_t draft = j < k ? draft_tokens[c + j] : 0;
    t = reduce_stats(stats, num_shards, total_rows, row).id;
    if (out_target_ids) out_target_ids[row] = t;
    mismatch = j < k && draft != t;
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
  if (prefill) {
    // a request still in prefill emits nothing this step
    if (j <= max_k) sampled_row[j] = -1;
    if (j == 0) {
      out_num_sampled[req] = 0;
      out_num_rejected[req] = 0;
      out_bonus[req] = -1;
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

// Many statistics per row (block-granular statistics: hundreds per row): one
// CTA per request, 512 threads.  Thread (stream k = tid / 16, row j = tid % 16)
// scans entries k, k + 32, ... of row j in ascending order with the scan rule,
// so the 16 threads of a half-warp read 16 consecutive rows of one entry
// (128 contiguous bytes per load).  The 32 streams of a row are then merged in
// shared memory on (value, entry position): NaN first, larger value, then the
// EARLIER position, which is exactly the sequential scan over all entries
// (the first NaN, else the first maximum).  Lanes 0..15 of warp 0 finish the
// request as in the narrow kernel.
constexpr int kWideThreads = 512;
constexpr int kStreams = kWideThreads / 16;

__global__ void __launch_bounds__(kWideThreads)
    greedy_verify_wide_kernel(const sga_stat *__restrict__ stats, int num_entries, int num_reqs,
                              const int32_t *__restrict__ cu_num_draft,
                              const int32_t *__restrict__ draft_tokens,
                              const uint8_t *__restrict__ in_prefill, int max_k,
                              int32_t *__restrict__ out_sampled,
                              int32_t *__restrict__ out_num_sampled,
                              int32_t *__restrict__ out_num_rejected,
                              int32_t *__restrict__ out_bonus, int32_t *__restrict__ out_target_ids,
                              uint32_t *err) {
  __shared__ float part_v[kStreams][16];
  __shared__ int32_t part_pos[kStreams][16];
  __shared__ int32_t part_id[kStreams][16];
  __shared__ int32_t t_row[16];
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int j = threadIdx.x & 15;       // row within the request
  const int stream = threadIdx.x >> 4;  // entries stream, stream + 32, ...
  const int64_t req = blockIdx.x;
  const int64_t total_rows = static_cast<int64_t>(cu_num_draft[num_reqs]) + num_reqs;
  const int32_t c = cu_num_draft[req];
  const int32_t k = cu_num_draft[req + 1] - c;
  const bool bad = k < 0 || k > max_k;
  const bool has_row = !bad && j <= k;
  const int64_t row = static_cast<int64_t>(c) + req + j;

  // lanes 0..15 load their draft now so that it overlaps the statistics
  const int32_t draft = threadIdx.x < 16 && !bad && j < k ? draft_tokens[c + j] : 0;
  const bool prefill = threadIdx.x < 16 && in_prefill != nullptr && in_prefill[req] != 0;
  float bv = __int_as_float(0xff800000);
  int32_t bpos = kNoId, bid = 0;
  if (has_row) {
    // batches of eight loads (bounds-predicated) issued before their
    // comparisons; entries in ascending order per thread
    for (int e0 = stream; e0 < num_entries; e0 += 8 * kStreams) {
      sga_stat x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u * kStreams < num_entries)
          x[u] = stats[static_cast<int64_t>(e0 + u * kStreams) * total_rows + row];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u * kStreams < num_entries && (bpos == kNoId || scan_better(x[u].v, bv))) {
          bv = x[u].v;
          bpos = e0 + u * kStreams;
          bid = x[u].id;
        }
    }
  }
  part_v[stream][j] = bv;
  part_pos[stream][j] = bpos;
  part_id[stream][j] = bid;
  __syncthreads();
  if (threadIdx.x < 16 && has_row) {
    float v = part_v[0][j];
    int32_t pos = part_pos[0][j], id = part_id[0][j];
    for (int q = 1; q < kStreams; ++q) {
      const int32_t qp = part_pos[q][j];
      if (qp != kNoId && (pos == kNoId || pair_beats(part_v[q][j], qp, v, pos))) {
        v = part_v[q][j];
        pos = qp;
        id = part_id[q][j];
      }
    }
    t_row[j] = id;
    if (out_target_ids) out_target_ids[row] = id;
  }
  __syncthreads();
  if (threadIdx.x >= 16) return;
  int32_t *sampled_row = out_sampled + req * (max_k + 1);
  if (bad) {
    if (lane <= max_k) sampled_row[lane] = -1;
    if (lane == 0) {
      out_num_sampled[req] = 0;
      out_num_rejected[req] = 0;
      out_bonus[req] = -1;
      atomicOr(err, SGA_DEVERR_K_RANGE);
    }
    return;
  }
  if (prefill) {
    // a request still in prefill emits nothing this step
    if (lane <= max_k) sampled_row[lane] = -1;
    if (lane == 0) {
      out_num_sampled[req] = 0;
      out_num_rejected[req] = 0;
      out_bonus[req] = -1;
    }
    return;
  }
  const int32_t t = lane <= k ? t_row[lane] : -1;
  const bool mismatch = lane < k && draft != t;
  const uint32_t mine = __ballot_sync(0x0000ffffu, mismatch);
  const int a = mine ? __ffs(mine) - 1 : k;  // accepted drafts
  if (lane <= max_k) sampled_row[lane] = lane <= a ? t : -1;
  if (lane == a) out_bonus[req] = t;
  if (lane == 0) {
    out_num_sampled[req] = a + 1;
    out_num_rejected[req] = k - a;
  }
}

}  // namespace

cudaError_t launch_greedy_verify(const sga_stat *stats, int num_shards, int num_reqs,
                                 const int32_t *cu_num_draft, const int32_t *draft_tokens,
                                 int max_k, int32_t *out_sampled, int32_t *out_num_sampled,
                                 int32_t *out_num_rejected, int32_t *out_bonus,
                                 int32_t *out_target_ids, uint32_t *err, cudaStream_t stream,
                                 const uint8_t *in_prefill) {
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (num_shards > kWideEntries) {
    cfg.gridDim = dim3(static_cast<unsigned>(num_reqs));
    cfg.blockDim = dim3(kWideThreads);
    return cudaLaunchKernelEx(&cfg, greedy_verify_wide_kernel, stats, num_shards, num_reqs,
                              cu_num_draft, draft_tokens, in_prefill, max_k, out_sampled,
                              out_num_sampled, out_num_rejected, out_bonus, out_target_ids, err);
  }
  const int64_t threads_needed = static_cast<int64_t>(num_reqs) * 16;
  cfg.gridDim = dim3(static_cast<unsigned>((threads_needed + kThreads - 1) / kThreads));
  cfg.blockDim = dim3(kThreads);
  return cudaLaunchKernelEx(&cfg, greedy_verify_kernel, stats, num_shards, num_reqs, cu_num_draft,
                            draft_tokens, in_prefill, max_k, out_sampled, out_num_sampled,
                            out_num_rejected, out_bonus, out_target_ids, err);
}

}  // namespace sga
