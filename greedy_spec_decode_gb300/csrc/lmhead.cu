// lmhead.cu -- fused LM-head GEMM + per-shard argmax on the 5th-generation
// tensor cores (tcgen05), operands staged by TMA, accumulators in TMEM.
//
// vLLM PR #62604, Purpose: with a vocab-parallel LM head each rank holds a
// vocab slice of the weight; item 2 fuses get_top_tokens.  vLLM PR #39419,
// Changes: get_top_tokens applies lm_head to the hidden states and keeps only
// the local argmax.  Here the logits hidden . W_shard^T never reach global
// memory: each 128 x 256 logits tile is accumulated in tensor memory and the
// epilogue keeps a running (max, id) per row.
//
// Kernel structure (CTA pairs, persistent, warp-specialised; M > 128 rows):
//   warp 0      TMA producer (both CTAs): its 128 hidden rows and 128 weight
//               rows of the pair's 256 x 256 tile, 128-byte K blocks,
//               128-byte swizzle, into a 6-stage shared ring.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators
//               per CTA); the leader's lane issues tcgen05.mma.cta_group::2
//               (M = 256, N = 256, K = 16 bf16 / 32 fp8).
//   warps 2..5  epilogue (both CTAs): tcgen05.ld of each accumulator row (one
//               TMEM lane per thread), argmax over the tile's valid columns,
//               then release the accumulator so the MMA of the next tile
//               overlaps this epilogue; one partial per (shard, row, chunk)
//               to the workspace.
// A small second kernel reduces each row's partials (one warp per row).
//
// The decode-size kernels (M <= 128, weight as the MMA's 128-row operand) are
// in lmhead_decode.cu; the PTX and host helpers all use are in tcgen05.cuh.
//
// Every mbarrier wait is bounded in time; on expiry the CTA records
// SGA_DEVERR_TIMEOUT, stops issuing work, waits (bounded) for its own copies
// and MMAs in flight, frees its TMEM and exits.
#include "tcgen05.cuh"

namespace sga {
namespace {

constexpr int TMEM_COLS = 2 * BN;      // double-buffered accumulator

// ---------------------------------------------------------------------------
// 2-SM kernel (tcgen05 cta_group::2): a cluster of two CTAs computes a
// 256-row x 256-id tile.  Each CTA stages its own 128 rows of hidden and its
// own 128 weight rows (half of the tile's ids), so per SM the shared-memory
// stage is 32 KB instead of the 48 KB a one-CTA 128 x 256 tile needs and the
// L2 traffic per MMA is 2/3 of it; six stages fit.  The even CTA (leader) issues every MMA; the
// tile's rows 0..127 accumulate in the leader's TMEM and rows 128..255 in the
// follower's, all 256 ids in both.
//   full[s]       leader only: 1 arrival (the leader's expect_tx of the
//                 pair's 64 KB); both CTAs' TMA copies complete their bytes
//                 on it (cta_group::2 copies may signal the peer's barrier).
//   empty[s]      1 arrival in each CTA, from the leader's multicast commit.
//   tmem_full[b]  1 arrival in each CTA, from the leader's multicast commit.
//   tmem_empty[b] leader only: 8 arrivals, one per epilogue warp of the pair.
// ---------------------------------------------------------------------------
#ifndef SGA_LMHEAD_STAGES2
#define SGA_LMHEAD_STAGES2 6
#endif
constexpr int STAGES2 = SGA_LMHEAD_STAGES2;
constexpr int A2_BYTES = 128 * ROW_BYTES;  // 16 KB
constexpr int B2_BYTES = 128 * ROW_BYTES;  // 16 KB (half of the 256-id tile)
constexpr int STAGE2_BYTES = A2_BYTES + B2_BYTES;
constexpr int SMEM2_BYTES = 1024 + STAGES2 * STAGE2_BYTES + 256;

struct Shared2 {
  uint64_t full[STAGES2];
  uint64_t empty[STAGES2];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort2(Shared2 *sh, uint32_t *err) {
  *reinterpret_cast<volatile int *>(&sh->abort) = 1;
  atomicOr(err, SGA_DEVERR_TIMEOUT);
}

// The shards of one GEMM launch (one, or every shard a GPU holds): shard s
// covers global ids [start, start + valid) (its non-padding ids) at rows
// row0 .. row0 + valid - 1 of the launch's weight map, and its 256-id tiles
// are numbers tile0[s] .. tile0[s + 1] - 1 of the launch (a shard without
// valid ids has none).
// Partial slots per (shard, row) of the 2-SM kernel, at most: the chunks a
// launch cuts its tiles into (one per CTA pair of a row block).
constexpr int kMaxChunks = 128;

struct GemmShardTable {
  int n;
  int32_t start[kMaxLmShards];
  int32_t row0[kMaxLmShards];
  int32_t valid[kMaxLmShards];
  int32_t tile0[kMaxLmShards + 1];
};

// First tile of chunk c when T tiles are cut into C contiguous chunks, and
// the chunk that holds tile t (the inverse); C <= T, so no chunk is empty.
__host__ __device__ __forceinline__ int chunk_first_tile(int c, int T, int C) {
  return static_cast<int>(static_cast<int64_t>(c) * T / C);
}
__host__ __device__ __forceinline__ int chunk_of_tile(int t, int T, int C) {
  return static_cast<int>((static_cast<int64_t>(t + 1) * C - 1) / T);
}

// Scan of 32 accumulator columns (ids id0 .. id0 + 31, all valid) in id
// order with the scan rule.  A NaN-propagating max of the 32 values goes
// first: when it cannot beat `best` (the common case once a tile is under
// way) no element can, and the ordered scan is skipped.
__device__ __forceinline__ void scan32(const uint32_t (&r)[32], int32_t id0, float &best,
                                       int32_t &best_id) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = max_nan(__uint_as_float(r[i]), __uint_as_float(r[i + 16]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = max_nan(m[i], m[i + w]);
  }
  if (scan_better(m[0], best)) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float x = __uint_as_float(r[i]);
      if (scan_better(x, best)) {
        best = x;
        best_id = id0 + i;
      }
    }
  }
}

// Work: the launch's T tiles (all shards, in id order) are cut into C
// contiguous chunks; a unit is (chunk c, 256-row block mp), numbered u = c *
// m_pairs + mp so that the pairs of one chunk, which stream the same weight
// tiles, run side by side and share them through L2.  Pair p takes units
// p, p + pairs, ...  Each epilogue thread keeps one hidden row's running
// (max, id) over all tiles of its unit and writes one partial per (shard,
// row, chunk) -- at the unit's end and at each shard edge inside it -- to
// ws[(s * M + row) * C + c]; the finalize kernel merges the chunks that meet
// shard s.
template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    lmhead_argmax_2sm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                             const __grid_constant__ CUtensorMap tmap_b, int M, int num_kb,
                             int m_pairs, int num_chunks,
                             const __grid_constant__ GemmShardTable tab,
                             sga_stat *__restrict__ ws, uint32_t *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *a_tiles = base;
  uint8_t *b_tiles = base + STAGES2 * A2_BYTES;
  Shared2 *sh = reinterpret_cast<Shared2 *>(base + STAGES2 * STAGE2_BYTES);
  const volatile int *abort_flag = &sh->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh->tmem_full[b]), 1);
      mbar_init(smem_u32(&sh->tmem_empty[b]), 8);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  // launched with programmatic stream serialisation: everything above (barrier
  // set-up, TMEM allocation) overlaps the previous kernel's tail; inputs and
  // the workspace are touched only after that kernel has completed
  pdl_wait();
  const int T = tab.tile0[tab.n];
  const int total = m_pairs * num_chunks;

  int prod_stage = 0;
  uint32_t prod_phase = 0;
  long long issued = 0;

  if (warp == 0 && lane == 0) {
    // -------------------------------------------------------------- producer
    for (int u = pair; u < total && !*abort_flag; u += num_pairs) {
      const int c = u / m_pairs, mp = u % m_pairs;
      const int t1 = chunk_first_tile(c + 1, T, num_chunks);
      int s = 0;
      for (int t = chunk_first_tile(c, T, num_chunks); t < t1 && !*abort_flag; ++t) {
        while (t >= tab.tile0[s + 1]) ++s;
        const int wrow = tab.row0[s] + (t - tab.tile0[s]) * BN + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(smem_u32(&sh->empty[prod_stage]), prod_phase ^ 1, abort_flag)) {
            raise_abort2(sh, err);
            break;
          }
          const uint32_t full_leader = map_to_rank(smem_u32(&sh->full[prod_stage]), 0);
          if (leader) mbar_expect_tx(smem_u32(&sh->full[prod_stage]), 2 * STAGE2_BYTES);
          tma_load_2d_pair(smem_u32(a_tiles + prod_stage * A2_BYTES), &tmap_a, kb * kBk<kFp8>,
                           mp * 256 + static_cast<int>(rank) * 128, full_leader);
          tma_load_2d_pair(smem_u32(b_tiles + prod_stage * B2_BYTES), &tmap_b, kb * kBk<kFp8>,
                           wrow, full_leader);
          ++issued;
          if (++prod_stage == STAGES2) {
            prod_stage = 0;
            prod_phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // -------------------------------------------------- MMA issuer (leader)
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int u = pair; u < total && ok && !*abort_flag; u += num_pairs) {
      const int c = u / m_pairs;
      const int tiles = chunk_first_tile(c + 1, T, num_chunks) - chunk_first_tile(c, T, num_chunks);
      for (int t = 0; t < tiles && ok; ++t) {
        if (!mbar_wait(smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1, abort_flag)) {
          raise_abort2(sh, err);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(smem_u32(&sh->full[stage]), phase, abort_flag)) {
            raise_abort2(sh, err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = smem_desc_sw128(smem_u32(a_tiles + stage * A2_BYTES));
          const uint64_t b_desc = smem_desc_sw128(smem_u32(b_tiles + stage * B2_BYTES));
#pragma unroll
          for (int kk = 0; kk < ROW_BYTES / 32; ++kk)
            mma_pair<kFp8>(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, (kb | kk) != 0);
          mma_commit_pair(smem_u32(&sh->empty[stage]));
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair(smem_u32(&sh->tmem_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else if (warp >= 2) {
    // -------------------------------------------------- epilogue (both CTAs)
    const int quarter = warp & 3;
    const int row_in_tile = static_cast<int>(rank) * 128 + quarter * 32 + lane;
    const uint32_t empty_leader[2] = {map_to_rank(smem_u32(&sh->tmem_empty[0]), 0),
                                      map_to_rank(smem_u32(&sh->tmem_empty[1]), 0)};
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int u = pair; u < total && ok; u += num_pairs) {
      const int c = u / m_pairs, mp = u % m_pairs;
      const int row = mp * 256 + row_in_tile;
      const int t0 = chunk_first_tile(c, T, num_chunks);
      const int t1 = chunk_first_tile(c + 1, T, num_chunks);
      int s = 0;
      while (t0 >= tab.tile0[s + 1]) ++s;
      float best = __int_as_float(0xff800000);
      int32_t best_id = kNoId;
      for (int t = t0; t < t1; ++t) {
        if (t >= tab.tile0[s + 1]) {
          // shard edge inside the unit: flush the finished shard's partial
          if (row < M) ws[(static_cast<size_t>(s) * M + row) * num_chunks + c] = {best, best_id};
          best = __int_as_float(0xff800000);
          best_id = kNoId;
          while (t >= tab.tile0[s + 1]) ++s;
        }
        ok = mbar_wait(smem_u32(&sh->tmem_full[acc]), acc_phase, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) raise_abort2(sh, err);
          break;
        }
        tc_fence_after();
        const int col0 = (t - tab.tile0[s]) * BN;
        const int valid = tab.valid[s];
        const int32_t id_base = tab.start[s];
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
#pragma unroll 1
        for (int q = 0; q < BN / 32; ++q) {
          uint32_t r[32];
          tmem_ld32(taddr + q * 32, r);
          tmem_ld_wait();
          const int cbase = col0 + q * 32;
          if (cbase + 32 <= valid) {
            scan32(r, id_base + cbase, best, best_id);
          } else if (cbase < valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float x = __uint_as_float(r[i]);
              if (cbase + i < valid && scan_better(x, best)) {
                best = x;
                best_id = id_base + cbase + i;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(smem_u32(&sh->tmem_empty[acc]));
          else
            mbar_arrive_remote(empty_leader[acc]);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (ok && row < M)
        ws[(static_cast<size_t>(s) * M + row) * num_chunks + c] = {best, best_id};
    }
  }

  pdl_launch_dependents();
  __syncthreads();
  if (*abort_flag) {
    const int zero = 0;
    if (warp == 0 && lane == 0) {
      if (leader) {
        // the leader's full barriers count the copies of both CTAs
        const long long outstanding = issued < STAGES2 ? issued : STAGES2;
        for (long long i = 1; i <= outstanding; ++i) {
          int s = prod_stage - static_cast<int>(i);
          uint32_t ph = prod_phase;
          if (s < 0) {
            s += STAGES2;
            ph ^= 1;
          }
          mbar_wait(smem_u32(&sh->full[s]), ph, &zero);
        }
      } else if (issued > 0) {
        // the follower's copies complete on the leader's barriers, which it
        // cannot wait on: give them a bounded 1 ms to land
        const unsigned long long t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
    if (warp == 1 && lane == 0 && leader) {
      mma_commit_pair(smem_u32(&sh->drain));
      mbar_wait(smem_u32(&sh->drain), 0, &zero);
    }
  }
  // the peer may still read this CTA's shared memory or write its TMEM
  tc_fence_before();
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// One warp per row: lanes stride over the row's partials (contiguous,
// row-major workspace) and merge them with the (value, id) order.
// Values of the fp8 variant are raw accumulators of the E4M3 codes until
// here; the positive row and weight scales (which cannot change the argmax of
// a row) are applied to the winning value only.
// The shards whose partials one finalize launch merges: row r of the output
// (shard s = r / M, hidden row r % M) merges the cnt[s] partials at
// ws[r * stride + lo[s] ...], and reports shard start[s]'s first id when no
// partial has a valid id (or when cnt[s] is 0: a shard without valid ids).
struct FinalizeShards {
  int n;
  int32_t start[kMaxLmShards];
  int32_t lo[kMaxLmShards];
  int32_t cnt[kMaxLmShards];
};

__global__ void lmhead_finalize_kernel(const sga_stat *__restrict__ ws, int M, int stride,
                                       const __grid_constant__ FinalizeShards shards,
                                       sga_stat *__restrict__ out,
                                       const float *__restrict__ row_scale, float w_scale,
                                       int scaled) {
  pdl_wait();  // the partials of the GEMM kernel are complete and visible
  pdl_launch_dependents();  // the next kernel may start its prologue
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= shards.n * M) return;
  const int s_idx = r / M;
  const int shard_start = shards.start[s_idx];
  const int count = shards.cnt[s_idx];
  float bv = __int_as_float(0xff800000);
  int32_t bi = kNoId;
  const sga_stat *row = ws + static_cast<size_t>(r) * stride + shards.lo[s_idx];
  constexpr int kInFlight = 4;  // loads issued before the first compare
  for (int n0 = lane; n0 < count; n0 += 32 * kInFlight) {
    sga_stat c[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int n = n0 + 32 * u;
      if (n < count) {
        c[u] = row[n];
      } else {
        c[u].v = __int_as_float(0xff800000);
        c[u].id = kNoId;
      }
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u)
      if (pair_beats(c[u].v, c[u].id, bv, bi)) {
        bv = c[u].v;
        bi = c[u].id;
      }
  }
  warp_argmax(bv, bi);
  if (lane == 0) {
    sga_stat s;
    s.v = scaled ? bv * ((row_scale ? row_scale[r % M] : 1.0f) * w_scale) : bv;
    s.id = bi == kNoId ? shard_start : bi;
    out[r] = s;
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// ever arrives at; the wait gives up after limit_ns, the kernel records
// SGA_DEVERR_TIMEOUT and returns, and the context stays usable.
__global__ void selftest_timeout_kernel(unsigned long long limit_ns, uint32_t *err,
                                        unsigned long long *waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int no_abort;
  if (threadIdx.x != 0) return;
  no_abort = 0;
  mbar_init(smem_u32(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const unsigned long long t0 = global_timer_ns();
  if (!mbar_wait(smem_u32(&bar), 0, &no_abort, limit_ns)) atomicOr(err, SGA_DEVERR_TIMEOUT);
  if (waited_ns) *waited_ns = global_timer_ns() - t0;
}

// Number of 2-CTA clusters of the 2-SM kernel that fit on the current device
// at once (queried once per device and operand type).
template <bool kFp8>
int resident_pairs(int num_sms) {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM2_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, lmhead_argmax_2sm_kernel<kFp8>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[dev] = n > num_sms / 2 ? num_sms / 2 : n;
  }
  return cache[dev];
}

// 2-SM kernel (M > SGA_LMHEAD_DECODE_MAX_M) over every shard of the table in one launch; the
// weight map spans map_rows rows.  Sets *chunks to the partial slots per
// (shard, row) (0 when there is no tile: nothing is launched).
template <bool kFp8>
cudaError_t launch_gemm_2sm(const void *hidden, int64_t M, int64_t H, const void *weight,
                            int64_t map_rows, const GemmShardTable &tab, sga_stat *ws,
                            int num_sms, uint32_t *err, cudaStream_t stream, int *chunks) {
  *chunks = 0;
  const int T = tab.tile0[tab.n];
  if (T == 0) return cudaSuccess;
  if (num_sms < 2) return cudaErrorNotSupported;
  const int num_kb = static_cast<int>(H / kBk<kFp8>);
  CUtensorMap map_a, map_b;
  if (!make_map(&map_a, hidden, M, H, 128, kFp8) || !make_map(&map_b, weight, map_rows, H, 128, kFp8))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(lmhead_argmax_2sm_kernel<kFp8>),
                                SMEM2_BYTES, kFp8 ? 2 : 0);
  if (e != cudaSuccess) return e;
  // A persistent grid must be fully resident: a cluster needs both CTAs in
  // one GPC, so fewer than num_sms / 2 pairs may fit at once.
  const int resident = resident_pairs<kFp8>(num_sms);
  if (resident <= 0) return cudaErrorLaunchOutOfResources;
  const int m_pairs = static_cast<int>((M + 255) / 256);
  int C = resident / m_pairs;
  if (C < 1) C = 1;
  if (C > T) C = T;
  if (C > kMaxChunks) C = kMaxChunks;
  const int units = m_pairs * C;
  const int pairs = units < resident ? units : resident;
  *chunks = C;
  return launch_pdl(lmhead_argmax_2sm_kernel<kFp8>, 2 * pairs, SMEM2_BYTES, stream, map_a, map_b,
                    static_cast<int>(M), num_kb, m_pairs, C, tab, ws, err);
}

}  // namespace

cudaError_t launch_selftest_timeout(unsigned long long limit_ns, uint32_t *err,
                                    unsigned long long *waited_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, err, waited_ns);
  return cudaGetLastError();
}

// Workspace (partial statistics) of one call:
//   M <= 128 (decode kernels): not used (the CTAs merge in library-owned
//     memory); the size keeps the earlier per-CTA partials' count, one
//     partial per (shard, row, CTA), the CTAs of a launch at most
//     kDecMaxParts, for one shard at least one per 256-id tile, so that
//     callers' buffers stay valid;
//   M >= 129 (2-SM kernel, one launch for every shard): one partial per
//     (shard, row, chunk), at most min(kMaxChunks, tiles of all shards)
//     chunks.
size_t lmhead_workspace_bytes(int64_t M, int64_t width) {
  return lmhead_shards_workspace_bytes(M, 1, &width);
}

size_t lmhead_shards_workspace_bytes(int64_t M, int num_shards, const int64_t *widths) {
  int64_t all_tiles = 0, most_tiles = 0;
  for (int s = 0; s < num_shards; ++s) {
    const int64_t t = (widths[s] + BN - 1) / BN;
    all_tiles += t;
    if (t > most_tiles) most_tiles = t;
  }
  if (M <= SGA_LMHEAD_DECODE_MAX_M) {
    if (num_shards == 1) {
      int64_t parts = (widths[0] + 127) / 128;
      if (parts > kDecMaxParts) parts = kDecMaxParts;
      if (parts < most_tiles) parts = most_tiles;
      return static_cast<size_t>(parts * M) * sizeof(sga_stat);
    }
    return static_cast<size_t>(num_shards) * static_cast<size_t>(M) * kDecMaxParts *
           sizeof(sga_stat);
  }
  const int64_t chunks = all_tiles < kMaxChunks ? all_tiles : kMaxChunks;
  return static_cast<size_t>(num_shards) * static_cast<size_t>(M) *
         static_cast<size_t>(chunks) * sizeof(sga_stat);
}

namespace {

// The finalize launch over every (shard, row) of a step: 8 rows per block;
// programmatic dependent launch lets the blocks become resident while the
// GEMM kernel drains (they wait in pdl_wait()).
cudaError_t launch_finalize(const sga_stat *ws, int64_t M, int ws_stride,
                            const FinalizeShards &shards, sga_stat *out,
                            const float *row_scale, float w_scale, bool fp8,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((shards.n * M + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lmhead_finalize_kernel, ws, static_cast<int>(M), ws_stride,
                            shards, out, row_scale, w_scale, fp8 ? 1 : 0);
}

}  // namespace

cudaError_t launch_lmhead_argmax(const void *hidden, int64_t M, int64_t H, const void *weight,
                                 int64_t shard_start, int64_t width, int64_t valid,
                                 sga_stat *out, void *workspace, int num_sms, uint32_t *err,
                                 cudaStream_t stream, bool fp8, const float *row_scale,
                                 float w_scale) {
  return launch_lmhead_argmax_shards(hidden, M, H, weight, 1, &shard_start, &width, &valid, out,
                                     workspace, num_sms, err, stream, fp8, row_scale, w_scale);
}

cudaError_t launch_lmhead_argmax_shards(const void *hidden, int64_t M, int64_t H,
                                        const void *weight, int num_shards,
                                        const int64_t *starts, const int64_t *widths,
                                        const int64_t *valids, sga_stat *out, void *workspace,
                                        int num_sms, uint32_t *err, cudaStream_t stream,
                                        bool fp8, const float *row_scale, float w_scale) {
  (void)widths;
  sga_stat *ws = static_cast<sga_stat *>(workspace);
  FinalizeShards fs = {};
  fs.n = num_shards;
  for (int s = 0; s < num_shards; ++s) fs.start[s] = static_cast<int32_t>(starts[s]);

  if (M <= SGA_LMHEAD_DECODE_MAX_M) {
    // decode sizes: every shard in one launch, which also merges its CTAs'
    // winners (no finalize launch, no workspace)
    int64_t row0s[kMaxLmShards];
    for (int s = 0; s < num_shards; ++s) row0s[s] = starts[s] - starts[0];
    bool launched = false;
    const cudaError_t e = launch_lmhead_decode(fp8, hidden, M, H, weight, num_shards, starts,
                                               row0s, valids, out, row_scale, w_scale, num_sms,
                                               err, stream, &launched);
    if (e != cudaSuccess || launched) return e;
    // every shard is padding: the finalize with no partials reports them
    return launch_finalize(ws, M, 0, fs, out, row_scale, w_scale, fp8, stream);
  }

  // 2-SM kernel: every shard in one launch, one finalize for all of them
  GemmShardTable tab = {};
  tab.n = num_shards;
  int64_t map_rows = 0;
  int tiles = 0;
  for (int s = 0; s < num_shards; ++s) {
    tab.start[s] = static_cast<int32_t>(starts[s]);
    tab.row0[s] = static_cast<int32_t>(starts[s] - starts[0]);
    tab.valid[s] = static_cast<int32_t>(valids[s]);
    tab.tile0[s] = tiles;
    tiles += static_cast<int>((valids[s] + BN - 1) / BN);
    if (valids[s] > 0 && tab.row0[s] + valids[s] > map_rows) map_rows = tab.row0[s] + valids[s];
  }
  tab.tile0[num_shards] = tiles;
  int chunks = 0;
  const cudaError_t e =
      fp8 ? launch_gemm_2sm<true>(hidden, M, H, weight, map_rows, tab, ws, num_sms, err, stream,
                                  &chunks)
          : launch_gemm_2sm<false>(hidden, M, H, weight, map_rows, tab, ws, num_sms, err, stream,
                                   &chunks);
  if (e != cudaSuccess) return e;
  for (int s = 0; s < num_shards; ++s) {
    if (tab.tile0[s + 1] > tab.tile0[s]) {
      fs.lo[s] = chunk_of_tile(tab.tile0[s], tiles, chunks);
      fs.cnt[s] = chunk_of_tile(tab.tile0[s + 1] - 1, tiles, chunks) - fs.lo[s] + 1;
    }
  }
  return launch_finalize(ws, M, chunks, fs, out, row_scale, w_scale, fp8, stream);
}

}  // namespace sga

// ---------------------------------------------------------------------------
// Scratch for sga_lmhead_argmax_noalloc: the per-tile partial statistics live
// in this fixed array instead of a caller-provided workspace.  Host code must
// not use the array's name as a device pointer (on the host it only stands in
// for the symbol); lmhead_noalloc_scratch() looks up its device address once
// per device, with that device current, and again if the device's context
// has changed since (a device reset reloads the module, and the array may
// move).
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoallocScratchBytes = SGA_LMHEAD_NOALLOC_SCRATCH_BYTES;
constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
sga_stat *g_noalloc_ptr[kNoallocMaxDevices];
uintptr_t g_noalloc_ctx[kNoallocMaxDevices];
}  // namespace

static __device__ __align__(256) sga_stat g_lmhead_noalloc_scratch[kNoallocScratchBytes / sizeof(sga_stat)];

namespace sga {

size_t lmhead_noalloc_scratch_bytes() { return kNoallocScratchBytes; }

cudaError_t lmhead_noalloc_scratch(sga_stat **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  const uintptr_t ctx = current_context_key();
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lmhead_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<sga_stat *>(p);
    g_noalloc_ctx[dev] = current_context_key();
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace sga
