// reduce.cu -- the cross-shard reduce of gathered statistics: per row the
// argmax, in the scan order (first NaN, else the first maximum), of its
// entries stats[s * rows + r], s = 0 .. num_shards - 1, optionally mapped from
// draft-vocabulary ids to target ids.
//
// vLLM PR #34049, Solution step 3: each rank reduces the gathered (max_value,
// global_index) pairs to the global argmax.  vLLM PR #39419, "Refactor local
// argmax code": a draft model with its own vocabulary maps the winning id k to
// k + draft_id_to_target_id[k] after the argmax.
//
// Two kernels: with up to kWideEntries entries per row (one per shard) a
// thread reduces one row with its loads in batches of eight
// (reduce_stats); with more (block-granular statistics: 200 per row at the
// large-verify shape) a CTA of 512 threads reduces 16 rows, 32 threads per
// row each scanning every 32nd entry, and the 32 partial winners of a row
// merge in shared memory on (value, entry position), which is exactly the
// sequential scan.
#include "common.cuh"
#include "scan.cuh"

namespace sga {
namespace {

#ifndef SGA_REDUCE_WIDE_ENTRIES
#define SGA_REDUCE_WIDE_ENTRIES 16
#endif
constexpr int kWideEntries = SGA_REDUCE_WIDE_ENTRIES;
constexpr int kWideThreads = 512;
constexpr int kWideRows = 16;
constexpr int kStreams = kWideThreads / kWideRows;

// The optional draft-to-target map and the stores of one row's result.
__device__ __forceinline__ void store_row(const sga_stat b, int64_t r, float *__restrict__ out_vals,
                                          int32_t *__restrict__ out_ids,
                                          const int64_t *__restrict__ d2t, int64_t d2t_len,
                                          uint32_t *err) {
  int32_t id = b.id;
  if (d2t != nullptr) {
    if (id >= 0 && id < d2t_len)
      id = static_cast<int32_t>(id + d2t[id]);
    else
      atomicOr(err, SGA_DEVERR_D2T_RANGE);
  }
  if (out_vals) out_vals[r] = b.v;
  out_ids[r] = id;
}

__global__ void shard_reduce_kernel(const sga_stat *__restrict__ stats, int num_shards, int64_t rows,
                                    float *__restrict__ out_vals, int32_t *__restrict__ out_ids,
                                    const int64_t *__restrict__ d2t, int64_t d2t_len,
                                    uint32_t *err) {
  pdl_wait();
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < rows;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x)
    store_row(reduce_stats(stats, num_shards, rows, r), r, out_vals, out_ids, d2t, d2t_len, err);
}

// Groups of 16 rows, CTA b taking groups b, b + gridDim.x, ...; thread
// (stream k = tid / 16, row j = tid % 16) scans entries k, k + 32, ... of its
// row, so a half-warp reads 16 consecutive rows of one entry (128 contiguous
// bytes).
__global__ void __launch_bounds__(kWideThreads)
    shard_reduce_wide_kernel(const sga_stat *__restrict__ stats, int num_entries, int64_t rows,
                             float *__restrict__ out_vals, int32_t *__restrict__ out_ids,
                             const int64_t *__restrict__ d2t, int64_t d2t_len, uint32_t *err) {
  __shared__ float part_v[kStreams][kWideRows];
  __shared__ int32_t part_pos[kStreams][kWideRows];
  __shared__ int32_t part_id[kStreams][kWideRows];
  pdl_wait();
  const int j = threadIdx.x % kWideRows;
  const int stream = threadIdx.x / kWideRows;
  const int64_t n_groups = (rows + kWideRows - 1) / kWideRows;
  for (int64_t grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {  // CTA-uniform
    const int64_t r = grp * kWideRows + j;
    float bv = __int_as_float(0xff800000);
    int32_t bpos = kNoId, bid = 0;
    if (r < rows) {
      // batches of eight loads (bounds-predicated) issued before their
      // comparisons; entries in ascending order per thread
      for (int e0 = stream; e0 < num_entries; e0 += 8 * kStreams) {
        sga_stat x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (e0 + u * kStreams < num_entries)
            x[u] = stats[static_cast<int64_t>(e0 + u * kStreams) * rows + r];
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
    if (threadIdx.x < kWideRows && r < rows) {
      // stream 0 holds entry 0 (num_entries >= 1), so pos starts valid
      sga_stat b;
      b.v = part_v[0][j];
      b.id = part_id[0][j];
      int32_t pos = part_pos[0][j];
      for (int q = 1; q < kStreams; ++q) {
        const int32_t qp = part_pos[q][j];
        if (qp != kNoId && pair_beats(part_v[q][j], qp, b.v, pos)) {
          b.v = part_v[q][j];
          b.id = part_id[q][j];
          pos = qp;
        }
      }
      store_row(b, r, out_vals, out_ids, d2t, d2t_len, err);
    }
    __syncthreads();  // the partials are rewritten by the next group
  }
}

}  // namespace

cudaError_t launch_shard_reduce(const sga_stat *stats, int num_shards, int64_t rows,
                                float *out_vals, int32_t *out_ids, const int64_t *d2t,
                                int64_t d2t_len, uint32_t *err, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (num_shards > kWideEntries) {
    int64_t groups = (rows + kWideRows - 1) / kWideRows;
    if (groups > (int64_t(1) << 20)) groups = int64_t(1) << 20;
    cfg.gridDim = dim3(static_cast<unsigned>(groups));
    cfg.blockDim = dim3(kWideThreads);
    return cudaLaunchKernelEx(&cfg, shard_reduce_wide_kernel, stats, num_shards, rows, out_vals,
                              out_ids, d2t, d2t_len, err);
  }
  const int threads = 256;
  int64_t blocks = (rows + threads - 1) / threads;
  if (blocks > 65535) blocks = 65535;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  return cudaLaunchKernelEx(&cfg, shard_reduce_kernel, stats, num_shards, rows, out_vals, out_ids,
                            d2t, d2t_len, err);
}

}  // namespace sga
