// argmax.cu -- per-shard argmax (with the padding mask) and the cross-shard
// reduce of the gathered statistics.
//
// vLLM PR #34049, Solution: local argmax on each vocab shard with the index
// made global, gather of (max_value, global_index), reduction across ranks.
// vLLM PR #62604, Purpose item 2: padding mask, lowest id on ties, NaN wins.
//
// The local argmax streams R x w logits once, so it is HBM-bound.  Each row of
// the shard is split into `chunks` contiguous pieces, one CTA each; the CTAs
// of a row form a thread-block cluster and merge their partial winners through
// distributed shared memory, so no workspace and no second pass are needed.
// Loads are 16-byte, L1-bypassing, four in flight per thread; the unaligned
// head and the tail of a row are read element by element.  Ids ascend within
// each thread's sequence, so the per-element test is the cheap scan rule, and
// a vector is inspected element-wise only when its NaN-propagating max could
// replace the running best.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace sga {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kMaxChunks = 8;

template <bool kBf16>
__device__ __forceinline__ float load_elem(const char *p, int64_t j) {
  if (kBf16) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p) + j);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  } else {
    return __ldg(reinterpret_cast<const float *>(p) + j);
  }
}

// Consume one 16-byte vector whose first element has global id `id`.
template <bool kBf16>
__device__ __forceinline__ void consume(const uint4 a, int32_t id, float &best, int32_t &best_id) {
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
  if (kBf16) {
    const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(w[0], w[1]), max_nan_bf16x2(w[2], w[3]));
    const float vmax = max_nan(bf16_lo(m), bf16_hi(m));
    if (scan_better(vmax, best)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = bf16_lo(w[k]);
        if (scan_better(lo, best)) {
          best = lo;
          best_id = id + 2 * k;
        }
        const float hi = bf16_hi(w[k]);
        if (scan_better(hi, best)) {
          best = hi;
          best_id = id + 2 * k + 1;
        }
      }
    }
  } else {
    const float vmax = max_nan(max_nan(__uint_as_float(w[0]), __uint_as_float(w[1])),
                               max_nan(__uint_as_float(w[2]), __uint_as_float(w[3])));
    if (scan_better(vmax, best)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x = __uint_as_float(w[k]);
        if (scan_better(x, best)) {
          best = x;
          best_id = id + k;
        }
      }
    }
  }
}

// grid.x = rows * chunks; the `chunks` CTAs of one row form one cluster.
// `valid` = number of non-padding ids of the shard (the rest is never read).
template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
    local_argmax_kernel(const char *__restrict__ logits, int64_t ld_bytes, int64_t shard_start,
                        int64_t valid, sga_stat *__restrict__ out, int chunks) {
  constexpr int kElt = kBf16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;
  __shared__ float warp_v[kThreads / 32];
  __shared__ int32_t warp_i[kThreads / 32];
  __shared__ float cta_v;
  __shared__ int32_t cta_i;

  const int64_t row = blockIdx.x / chunks;
  const int chunk = static_cast<int>(blockIdx.x % chunks);
  const int tid = threadIdx.x;
  const char *p = logits + row * ld_bytes;
  const int32_t id0 = static_cast<int32_t>(shard_start);

  float best = __int_as_float(0xff800000);  // -inf
  int32_t best_id = kNoId;

  // Split the row into an element-wise head up to the first 16-byte boundary,
  // whole 16-byte vectors, and an element-wise tail.
  int64_t head = static_cast<int64_t>(((16u - (reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / kElt);
  if (head > valid) head = valid;
  const int64_t nvec = (valid - head) / kVec;
  const int64_t tail = valid - head - nvec * kVec;
  const int64_t v0 = nvec * chunk / chunks;
  const int64_t v1 = nvec * (chunk + 1) / chunks;

  if (chunk == 0 && tid < head) {
    const float x = load_elem<kBf16>(p, tid);
    if (scan_better(x, best)) {
      best = x;
      best_id = id0 + tid;
    }
  }

  const uint4 *vp = reinterpret_cast<const uint4 *>(p + head * kElt);
  const int32_t body_id = id0 + static_cast<int32_t>(head);
  int64_t v = v0 + tid;
  for (; v + (kUnroll - 1) * kThreads < v1; v += kUnroll * kThreads) {
    uint4 a[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) a[u] = ld_stream_v4(vp + v + u * kThreads);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      consume<kBf16>(a[u], body_id + static_cast<int32_t>((v + u * kThreads) * kVec), best, best_id);
  }
  for (; v < v1; v += kThreads)
    consume<kBf16>(ld_stream_v4(vp + v), body_id + static_cast<int32_t>(v * kVec), best, best_id);

  if (chunk == chunks - 1 && tid < tail) {
    const int64_t j = head + nvec * kVec + tid;
    const float x = load_elem<kBf16>(p, j);
    if (scan_better(x, best)) {
      best = x;
      best_id = id0 + static_cast<int32_t>(j);
    }
  }

  // CTA reduction with the full (value, id) order.
  warp_argmax(best, best_id);
  if ((tid & 31) == 0) {
    warp_v[tid >> 5] = best;
    warp_i[tid >> 5] = best_id;
  }
  __syncthreads();
  if (tid < 32) {
    best = tid < kThreads / 32 ? warp_v[tid] : __int_as_float(0xff800000);
    best_id = tid < kThreads / 32 ? warp_i[tid] : kNoId;
    warp_argmax(best, best_id);
    if (tid == 0) {
      cta_v = best;
      cta_i = best_id;
    }
  }

  if (chunks > 1) {
    // Merge the partial winners of the row's CTAs through distributed shared
    // memory; the second cluster barrier keeps every CTA's shared memory alive
    // until rank 0 has read it.
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (cluster.block_rank() == 0 && tid < 32) {
      best = __int_as_float(0xff800000);
      best_id = kNoId;
      if (tid < chunks) {
        best = *cluster.map_shared_rank(&cta_v, tid);
        best_id = *cluster.map_shared_rank(&cta_i, tid);
      }
      warp_argmax(best, best_id);
    }
    cluster.sync();
    if (cluster.block_rank() != 0) return;
  }
  if (tid == 0) {
    sga_stat s;
    s.v = best;  // -inf when nothing beat -inf
    s.id = best_id == kNoId ? id0 : best_id;
    out[row] = s;
  }
}

__global__ void shard_reduce_kernel(const sga_stat *__restrict__ stats, int num_shards, int64_t rows,
                                    float *__restrict__ out_vals, int32_t *__restrict__ out_ids,
                                    const int64_t *__restrict__ d2t, int64_t d2t_len,
                                    uint32_t *err) {
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < rows;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    sga_stat b = stats[r];
    for (int s = 1; s < num_shards; ++s) {
      const sga_stat c = stats[static_cast<int64_t>(s) * rows + r];
      if (scan_better(c.v, b.v)) b = c;
    }
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
}

}  // namespace

cudaError_t launch_local_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                                int64_t shard_start, int64_t width, int64_t valid,
                                sga_stat *out, int num_sms, cudaStream_t stream) {
  (void)width;
  const int elt = dtype == SGA_BF16 ? 2 : 4;
  const int64_t nvec = valid * elt / 16;
  const int64_t target_ctas = static_cast<int64_t>(num_sms) * 4;
  int chunks = 1;
  while (chunks < kMaxChunks && rows * chunks < target_ctas &&
         nvec / (2 * chunks) >= kThreads * kUnroll)
    chunks *= 2;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows * chunks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = chunks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const char *base = static_cast<const char *>(logits);
  const int64_t ld_bytes = ld * elt;
  if (dtype == SGA_BF16)
    return cudaLaunchKernelEx(&cfg, local_argmax_kernel<true>, base, ld_bytes, shard_start, valid,
                              out, chunks);
  return cudaLaunchKernelEx(&cfg, local_argmax_kernel<false>, base, ld_bytes, shard_start, valid,
                            out, chunks);
}

cudaError_t launch_shard_reduce(const sga_stat *stats, int num_shards, int64_t rows,
                                float *out_vals, int32_t *out_ids, const int64_t *d2t,
                                int64_t d2t_len, uint32_t *err, cudaStream_t stream) {
  const int threads = 256;
  int64_t blocks = (rows + threads - 1) / threads;
  if (blocks > 65535) blocks = 65535;
  shard_reduce_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      stats, num_shards, rows, out_vals, out_ids, d2t, d2t_len, err);
  return cudaGetLastError();
}

}  // namespace sga
