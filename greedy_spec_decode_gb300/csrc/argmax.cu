// argmax.cu -- per-shard argmax (with the padding mask); the cross-shard
// reduce of the gathered statistics is in reduce.cu.
//
// vLLM PR #34049, Solution: local argmax on each vocab shard with the index
// made global, gather of (max_value, global_index), reduction across ranks.
// vLLM PR #62604, Purpose item 2: padding mask, lowest id on ties, NaN wins.
//
// The local argmax streams R x w logits once, so it is HBM-bound; the design
// keeps the instruction count per 16-byte vector small so that the load
// stream, not the issue slots, sets the pace:
//   * each (row, shard) is split into `chunks` contiguous pieces, one CTA
//     each; the CTAs of a (row, shard) form a thread-block cluster and merge
//     their partial winners through distributed shared memory (no workspace,
//     no second pass).  One launch may cover several shards (all the shards a
//     GPU holds): grid = rows x shards x chunks.
//   * the 16-byte-aligned body of a row is copied into a shared-memory ring by
//     cp.async.bulk (a dedicated copy warp, mbarrier completion, 4 x 8 KB in
//     flight per CTA, about 190 KB per SM); consumer threads read 16-byte
//     vectors from shared memory.  The unaligned head and the tail of a row are
//     read element by element.
//   * in the body a thread keeps only the NaN-propagating maximum of the best
//     vector it has seen and that vector's index (strictly greater replaces,
//     so ties keep the earliest vector) together with that vector's 16 bytes;
//     after the loop it picks the vector's first element equal to the maximum
//     (or its first NaN).  Ids ascend along each thread's sequence, so this is
//     exactly the scan rule of the oracle.
#include <cooperative_groups.h>

#include "common.cuh"
#include "scan.cuh"

namespace cg = cooperative_groups;

namespace sga {
namespace {

// Tuning knobs (compile-time).  Measured on GB300 with the large-verify shape
// (4096 x 202048 bf16, 3 shards in one launch): the cp.async.bulk ring (128
// consumer threads + 1 copy warp, 4 stages of 8 KB) streams at 7.0 TB/s; the
// plain 16-byte-load body peaks at 6.0 TB/s (256 threads, 8 loads in flight).
// SGA_ARGMAX_THREADS: consumer threads per CTA; SGA_ARGMAX_UNROLL applies to
// the plain-load body only (SGA_ARGMAX_BULK=0).
#ifndef SGA_ARGMAX_THREADS
#define SGA_ARGMAX_THREADS 128
#endif
#ifndef SGA_ARGMAX_UNROLL
#define SGA_ARGMAX_UNROLL 8
#endif
constexpr int kThreads = SGA_ARGMAX_THREADS;
constexpr int kUnroll = SGA_ARGMAX_UNROLL;
constexpr int kMinBlocks = 2048 / kThreads;
constexpr int kMaxChunks = 8;

struct ShardTable {
  int n;
  int32_t start[kMaxShardsPerLaunch];  // global id of the shard's first column
  int32_t col[kMaxShardsPerLaunch];    // column of that id relative to `logits`
  int32_t valid[kMaxShardsPerLaunch];  // non-padding ids of the shard
};

#ifndef SGA_ARGMAX_BULK
#define SGA_ARGMAX_BULK 1
#endif
#ifndef SGA_ARGMAX_PREFETCH
// L2 prefetch of the first ring stages before the PDL wait.  Measured on the
// large-verify step: one launch for all shards 231.8 -> 229.9 us, one launch
// per shard 252.9 -> 244.0 us per step; the small workloads unchanged.
#define SGA_ARGMAX_PREFETCH 1
#endif
#ifndef SGA_ARGMAX_STAGES
#define SGA_ARGMAX_STAGES 4
#endif
#ifndef SGA_ARGMAX_STAGE_BYTES
#define SGA_ARGMAX_STAGE_BYTES 8192
#endif
constexpr int kStages = SGA_ARGMAX_STAGES;
constexpr int kStageVec = SGA_ARGMAX_STAGE_BYTES / 16;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; false after kWaitLimitNs or on abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int *abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// grid.x = rows * shards * chunks, CTA b: chunk = b % chunks, then (row,
// shard) in row-major order so consecutive CTAs stream consecutive memory.
// The `chunks` CTAs of one (row, shard) form one cluster.
//
// kBulk = false: every thread streams its vectors with 16-byte loads.
// kBulk = true: one extra warp copies the body into a shared-memory ring with
// cp.async.bulk (kStages x SGA_ARGMAX_STAGE_BYTES, mbarrier completion) and
// the kThreads consumer threads read it from shared memory.
template <bool kBf16, bool kBulk>
__global__ void __launch_bounds__(kThreads + (kBulk ? 32 : 0), kBulk ? 2048 / (kThreads + 32) : kMinBlocks)
    local_argmax_kernel(const char *__restrict__ logits, int64_t ld_bytes,
                        const __grid_constant__ ShardTable tab, sga_stat *__restrict__ out,
                        int rows, int chunks, uint32_t *err) {
  constexpr int kElt = kBf16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;
  constexpr int kWarps = (kThreads + (kBulk ? 32 : 0)) / 32;
  __shared__ float warp_v[kWarps];
  __shared__ int32_t warp_i[kWarps];
  __shared__ float cta_v;
  __shared__ int32_t cta_i;

  const int chunk = static_cast<int>(blockIdx.x % chunks);
  const int rs = static_cast<int>(blockIdx.x / chunks);
  const int row = rs / tab.n;
  const int s = rs - row * tab.n;
  const int32_t id0 = tab.start[s];
  const int valid = tab.valid[s];
  const char *p = logits + row * ld_bytes + static_cast<int64_t>(tab.col[s]) * kElt;
  const int tid = threadIdx.x;

  float best = __int_as_float(0xff800000);  // -inf
  int32_t best_id = kNoId;

  // Element-wise head up to the first 16-byte boundary, whole vectors, tail.
  int head = static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / kElt);
  if (head > valid) head = valid;
  const int nvec = (valid - head) / kVec;
  const int tail = valid - head - nvec * kVec;
  const int v0 = static_cast<int>(static_cast<int64_t>(nvec) * chunk / chunks);
  const int v1 = static_cast<int>(static_cast<int64_t>(nvec) * (chunk + 1) / chunks);

  if (kBulk && SGA_ARGMAX_PREFETCH && tid == kThreads && v1 > v0) {
    // Warm L2 with what the ring loads first while the previous kernel
    // drains: the addresses come from the parameters alone, and a prefetch
    // only fills L2, which stays coherent with any later write, so it may
    // precede the dependency wait.
    const int n = min(v1 - v0, kStages * kStageVec);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                     reinterpret_cast<const uint4 *>(p + head * kElt) + v0),
                 "r"(n * 16)
                 : "memory");
  }
  pdl_wait();  // inputs written by the previous kernel in the stream are visible

  if (chunk == 0 && tid < head) {
    const float x = load_elem<kBf16>(p, tid);
    if (scan_better(x, best)) {
      best = x;
      best_id = id0 + tid;
    }
  }

  const uint4 *vp = reinterpret_cast<const uint4 *>(p + head * kElt);
  float vbest = __int_as_float(0xff800000);
  int vbest_idx = -1;
  uint4 vraw = make_uint4(0u, 0u, 0u, 0u);  // the best vector itself
  if (!kBulk) {
    int v = v0 + tid;
    for (; v + (kUnroll - 1) * kThreads < v1; v += kUnroll * kThreads) {
      uint4 a[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) a[u] = ld_stream_v4(vp + v + u * kThreads);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const float m = vec_max<kBf16>(a[u]);
        if (scan_better(m, vbest)) {
          vbest = m;
          vbest_idx = v + u * kThreads;
          vraw = a[u];
        }
      }
    }
    for (; v < v1; v += kThreads) {
      const uint4 a = ld_stream_v4(vp + v);
      const float m = vec_max<kBf16>(a);
      if (scan_better(m, vbest)) {
        vbest = m;
        vbest_idx = v;
        vraw = a;
      }
    }
  } else {
    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t empty[kStages];
    __shared__ int abort_flag;
    const int nbody = v1 - v0;
    const int nst = (nbody + kStageVec - 1) / kStageVec;
    if (tid == 0) {
      for (int k = 0; k < kStages; ++k) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
            static_cast<uint32_t>(__cvta_generic_to_shared(&full[k]))));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(&empty[k]))),
                     "r"(kThreads / 32));
      }
      abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const volatile int *abort_v = &abort_flag;
    int issued = 0;
    if (tid == kThreads) {
      // producer: one lane of the extra warp
      for (int j = 0; j < nst; ++j) {
        const int slot = j % kStages;
        const uint32_t e = static_cast<uint32_t>(__cvta_generic_to_shared(&empty[slot]));
        if (j >= kStages && !mbar_wait_bounded(e, ((j / kStages) - 1) & 1, abort_v)) {
          abort_flag = 1;
          atomicOr(err, SGA_DEVERR_TIMEOUT);
          break;
        }
        const int n = min(kStageVec, nbody - j * kStageVec);
        const uint32_t f = static_cast<uint32_t>(__cvta_generic_to_shared(&full[slot]));
        const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(ring + slot * kStageVec));
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(f), "r"(n * 16)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            ::"r"(dst), "l"(vp + v0 + j * kStageVec), "r"(n * 16), "r"(f)
            : "memory");
        issued = j + 1;
      }
    } else if (tid < kThreads) {
      const int lane = tid & 31;
      for (int j = 0; j < nst; ++j) {
        const int slot = j % kStages;
        const uint32_t f = static_cast<uint32_t>(__cvta_generic_to_shared(&full[slot]));
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(f, (j / kStages) & 1, abort_v));
        if (!ok) {
          if (lane == 0) {
            abort_flag = 1;
            atomicOr(err, SGA_DEVERR_TIMEOUT);
          }
          break;
        }
        const int n = min(kStageVec, nbody - j * kStageVec);
        const uint4 *st = ring + slot * kStageVec;
        for (int i = tid; i < n; i += kThreads) {
          const uint4 a = st[i];
          const float m = vec_max<kBf16>(a);
          if (scan_better(m, vbest)) {
            vbest = m;
            vbest_idx = v0 + j * kStageVec + i;
            vraw = a;
          }
        }
        __syncwarp();
        if (lane == 0)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                           static_cast<uint32_t>(__cvta_generic_to_shared(&empty[slot])))
                       : "memory");
      }
    }
    __syncthreads();
    if (abort_flag && tid == kThreads) {
      // let this CTA's own copies land before its shared memory is released
      const int zero = 0;
      for (int j = issued - 1; j >= 0 && j >= issued - kStages; --j)
        mbar_wait_bounded(static_cast<uint32_t>(__cvta_generic_to_shared(&full[j % kStages])),
                          (j / kStages) & 1, &zero);
    }
  }
  pdl_launch_dependents();
  if (vbest_idx >= 0) scan_vec<kBf16>(vraw, id0 + head + vbest_idx * kVec, best, best_id);

  if (chunk == chunks - 1 && tid < tail) {
    const int j = head + nvec * kVec + tid;
    const float x = load_elem<kBf16>(p, j);
    if (scan_better(x, best)) {
      best = x;
      best_id = id0 + j;
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
    best = tid < kWarps ? warp_v[tid] : __int_as_float(0xff800000);
    best_id = tid < kWarps ? warp_i[tid] : kNoId;
    warp_argmax(best, best_id);
    if (tid == 0) {
      cta_v = best;
      cta_i = best_id;
    }
  }

  if (chunks > 1) {
    // Merge the partial winners of the (row, shard)'s CTAs through distributed
    // shared memory; the second cluster barrier keeps every CTA's shared
    // memory alive until rank 0 has read it.
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
    sga_stat st;
    st.v = best;  // -inf when nothing beat -inf
    st.id = best_id == kNoId ? id0 : best_id;
    out[static_cast<int64_t>(s) * rows + row] = st;
  }
}

// Pieces per (row, shard).  Splitting a row costs two cluster barriers and a
// shorter-lived CTA (its reduction tail is not streaming), so a row is split
// (in powers of two) only while the grid stays within half of the resident
// CTA slots.  Measured on GB300 after an L2 flush (one step, argmax + reduce
// or verify): 32 rows x 2 shards of 76032 bf16 ids: 1 / 2 / 4 / 8 pieces per
// row 15.5 / 13.1 / 12.8 / 13.0 us (the rule picks 4); 96 rows x 4 shards of
// 50016: 19.1 / 20.0 / 23.5 / 23.5 us (the rule picks 1; a one-wave target
// picked 4).
#ifndef SGA_ARGMAX_WAVES
#define SGA_ARGMAX_WAVES 1
#endif
int pick_chunks(int64_t rs_count, int64_t max_valid, int elt, int num_sms) {
  const int64_t nvec = max_valid * elt / 16;
  // resident CTAs per SM: bounded by threads, and for the ring by shared memory
  int64_t per_sm = kMinBlocks;
  if (SGA_ARGMAX_BULK) {
    const int64_t by_threads = 2048 / (kThreads + 32);
    const int64_t by_smem = (227 * 1024) / (kStages * kStageVec * 16 + 1024 + 256);
    per_sm = by_threads < by_smem ? by_threads : by_smem;
  }
  const int64_t want_ctas = static_cast<int64_t>(num_sms) * per_sm * SGA_ARGMAX_WAVES;
  int chunks = 1;
  while (chunks < kMaxChunks && nvec / (2 * chunks) >= kThreads &&
         rs_count * chunks * 4 <= want_ctas)
    chunks *= 2;
  return chunks;
}

}  // namespace

cudaError_t launch_local_argmax_table(const void *logits, int dtype, int64_t rows, int64_t ld,
                                      int num_shards, const int64_t *starts,
                                      const int64_t *cols, const int64_t *valids, sga_stat *out,
                                      int num_sms, uint32_t *err, cudaStream_t stream) {
  ShardTable tab;
  tab.n = num_shards;
  int64_t max_valid = 0;
  for (int s = 0; s < num_shards; ++s) {
    tab.start[s] = static_cast<int32_t>(starts[s]);
    tab.col[s] = static_cast<int32_t>(cols[s]);
    tab.valid[s] = static_cast<int32_t>(valids[s]);
    if (valids[s] > max_valid) max_valid = valids[s];
  }
  const int elt = dtype == SGA_BF16 ? 2 : 4;
  const int chunks = pick_chunks(rows * num_shards, max_valid, elt, num_sms);
  constexpr bool kBulk = SGA_ARGMAX_BULK != 0;
  const size_t smem = kBulk ? static_cast<size_t>(kStages) * kStageVec * 16 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows * num_shards * chunks));
  cfg.blockDim = dim3(kThreads + (kBulk ? 32 : 0));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = chunks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const char *base = static_cast<const char *>(logits);
  const int64_t ld_bytes = ld * elt;
  const int rows_i = static_cast<int>(rows);
  if (dtype == SGA_BF16) {
    auto kern = local_argmax_kernel<true, kBulk>;
    if (smem > 48 * 1024) {
      const cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, kern, base, ld_bytes, tab, out, rows_i, chunks, err);
  }
  auto kern = local_argmax_kernel<false, kBulk>;
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, kern, base, ld_bytes, tab, out, rows_i, chunks, err);
}

cudaError_t launch_local_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                                int64_t shard_start, int64_t width, int64_t valid,
                                sga_stat *out, int num_sms, uint32_t *err, cudaStream_t stream) {
  (void)width;
  const int64_t col = 0;
  return launch_local_argmax_table(logits, dtype, rows, ld, 1, &shard_start, &col, &valid, out,
                                   num_sms, err, stream);
}

}  // namespace sga
