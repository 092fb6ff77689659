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
// Kernel structure (one CTA per SM, persistent, warp-specialised):
//   warp 0      TMA producer: A (hidden, 128 x 64) and B (weight, 256 x 64)
//               bf16 tiles, 128-byte swizzle, into a 4-stage shared ring.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//               and issues tcgen05.mma (M=128, N=256, K=16) from one lane.
//   warps 2..5  epilogue: tcgen05.ld of each accumulator row (one TMEM lane
//               per thread), argmax over the tile's valid columns, partial
//               stat to the workspace, then release the accumulator so the
//               MMA of the next tile overlaps this epilogue.
// Work items are (vocab tile, row tile) with the row tile fastest, so the CTAs
// running at the same time share weight tiles through L2 and the weight is
// streamed from HBM about once.  A small second kernel reduces each row's
// per-tile partials (one warp per row, row-major workspace).
//
// The decode-size kernel (M <= 64, weight as the MMA's 128-row operand) is in
// lmhead_decode.cu; the PTX and host helpers both use are in tcgen05.cuh.
//
// Every mbarrier wait is bounded in time; on expiry the CTA records
// SGA_DEVERR_TIMEOUT, stops issuing work, waits (bounded) for its own copies
// and MMAs in flight, frees its TMEM and exits.
#include "tcgen05.cuh"

namespace sga {
namespace {

constexpr int BM = 128;          // rows of hidden per tile (TMEM lanes)
#ifndef SGA_LMHEAD_STAGES
#define SGA_LMHEAD_STAGES 4
#endif
#ifndef SGA_LMHEAD_2SM
#define SGA_LMHEAD_2SM 1  // 2-SM tiles when M >= SGA_LMHEAD_2SM_MIN_M
#endif
#ifndef SGA_LMHEAD_2SM_MIN_M
#define SGA_LMHEAD_2SM_MIN_M 129
#endif
constexpr int STAGES = SGA_LMHEAD_STAGES;
constexpr int A_BYTES = BM * ROW_BYTES;   // 16 KB
constexpr int B_BYTES = BN * ROW_BYTES;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;      // double-buffered accumulator
// At least 120 KB so that one CTA (holding all 512 TMEM columns) runs per SM.
constexpr int SMEM_NEEDED = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/;
constexpr int SMEM_BYTES = SMEM_NEEDED > 120 * 1024 ? SMEM_NEEDED : 120 * 1024;

// One MMA of a K step (16 bf16 or 32 fp8 = 32 bytes of each row), M = BM,
// N = BN, issued by one thread of this CTA.
template <bool kFp8>
__device__ __forceinline__ void mma_1sm(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t accumulate) {
  constexpr uint32_t idesc = instr_desc<kFp8>(BM, BN);
  if constexpr (kFp8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

struct Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(Shared *sh, uint32_t *err) {
  *reinterpret_cast<volatile int *>(&sh->abort) = 1;
  atomicOr(err, SGA_DEVERR_TIMEOUT);
}

template <bool kFp8>
__global__ void __launch_bounds__(THREADS, 1)
    lmhead_argmax_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b, int M, int num_kb,
                         int m_tiles, int n_tiles, int valid, int shard_start,
                         sga_stat *__restrict__ ws, uint32_t *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *a_tiles = base;
  uint8_t *b_tiles = base + STAGES * A_BYTES;
  Shared *sh = reinterpret_cast<Shared *>(base + STAGES * STAGE_BYTES);
  const volatile int *abort_flag = &sh->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh->tmem_full[b]), 1);
      mbar_init(smem_u32(&sh->tmem_empty[b]), 4 * 32);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  // launched with programmatic stream serialisation: everything above (barrier
  // set-up, TMEM allocation) overlaps the previous kernel's tail; inputs and
  // the workspace are touched only after that kernel has completed
  pdl_wait();
  const int total = m_tiles * n_tiles;

  int prod_stage = 0;
  uint32_t prod_phase = 0;
  long long issued = 0;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      for (int item = blockIdx.x; item < total && !*abort_flag; item += gridDim.x) {
        const int n = item / m_tiles, m = item % m_tiles;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(smem_u32(&sh->empty[prod_stage]), prod_phase ^ 1, abort_flag)) {
            raise_abort(sh, err);
            break;
          }
          const uint32_t full = smem_u32(&sh->full[prod_stage]);
          mbar_expect_tx(full, STAGE_BYTES);
          tma_load_2d(smem_u32(a_tiles + prod_stage * A_BYTES), &tmap_a, kb * kBk<kFp8>, m * BM,
                      full);
          tma_load_2d(smem_u32(b_tiles + prod_stage * B_BYTES), &tmap_b, kb * kBk<kFp8>, n * BN,
                      full);
          ++issued;
          if (++prod_stage == STAGES) {
            prod_stage = 0;
            prod_phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int item = blockIdx.x; item < total && !*abort_flag; item += gridDim.x) {
        if (!mbar_wait(smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1, abort_flag)) {
          raise_abort(sh, err);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(smem_u32(&sh->full[stage]), phase, abort_flag)) {
            raise_abort(sh, err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = smem_desc_sw128(smem_u32(a_tiles + stage * A_BYTES));
          const uint64_t b_desc = smem_desc_sw128(smem_u32(b_tiles + stage * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < ROW_BYTES / 32; ++kk)  // 32 bytes = 2 descriptor units
            mma_1sm<kFp8>(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, (kb | kk) != 0);
          mma_commit(smem_u32(&sh->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&sh->tmem_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
    const int row_in_tile = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const int n = item / m_tiles, m = item % m_tiles;
      bool ok = mbar_wait(smem_u32(&sh->tmem_full[acc]), acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort(sh, err);
        break;
      }
      tc_fence_after();
      float best = __int_as_float(0xff800000);
      int32_t best_id = kNoId;
      const int col0 = n * BN;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_ld_wait();
        const int cbase = col0 + c * 32;
        if (cbase < valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = __uint_as_float(r[i]);
            if (cbase + i < valid && scan_better(x, best)) {
              best = x;
              best_id = shard_start + cbase + i;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sh->tmem_empty[acc]));
      const int row = m * BM + row_in_tile;
      if (row < M) {
        sga_stat st;
        st.v = best;
        st.id = best_id;
        ws[static_cast<size_t>(row) * n_tiles + n] = st;
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  pdl_launch_dependents();
  __syncthreads();
  if (*abort_flag) {
    // Let this CTA's own copies and MMAs land before its shared memory and
    // tensor memory are released (bounded as well).
    const int zero = 0;
    if (warp == 0 && lane == 0) {
      const long long outstanding = issued < STAGES ? issued : STAGES;
      for (long long i = 1; i <= outstanding; ++i) {
        int s = prod_stage - static_cast<int>(i);
        uint32_t ph = prod_phase;
        if (s < 0) {
          s += STAGES;
          ph ^= 1;
        }
        mbar_wait(smem_u32(&sh->full[s]), ph, &zero);
      }
    }
    if (warp == 1 && lane == 0) {
      mma_commit(smem_u32(&sh->drain));
      mbar_wait(smem_u32(&sh->drain), 0, &zero);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// 2-SM variant (tcgen05 cta_group::2): a cluster of two CTAs computes a
// 256-row x 256-id tile.  Each CTA stages its own 128 rows of hidden and its
// own 128 weight rows (half of the tile's ids), so per SM the shared-memory
// stage is 32 KB instead of 48 KB and the L2 traffic per MMA is 2/3 of the
// 1-SM kernel's; six stages fit.  The even CTA (leader) issues every MMA; the
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

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA tile copy into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

template <bool kFp8>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t accumulate) {
  constexpr uint32_t idesc = instr_desc<kFp8>(256, 256);  // M = 256 across the pair
  if constexpr (kFp8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrive once on `bar` in both CTAs of the pair when the MMAs issued so far
// have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void raise_abort2(Shared2 *sh, uint32_t *err) {
  *reinterpret_cast<volatile int *>(&sh->abort) = 1;
  atomicOr(err, SGA_DEVERR_TIMEOUT);
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    lmhead_argmax_2sm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                             const __grid_constant__ CUtensorMap tmap_b, int M, int num_kb,
                             int m_pairs, int n_tiles, int valid, int shard_start,
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
  const int total = m_pairs * n_tiles;

  int prod_stage = 0;
  uint32_t prod_phase = 0;
  long long issued = 0;

  if (warp == 0 && lane == 0) {
    // -------------------------------------------------------------- producer
    for (int item = pair; item < total && !*abort_flag; item += num_pairs) {
      const int n = item / m_pairs, mp = item % m_pairs;
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
                         n * 256 + static_cast<int>(rank) * 128, full_leader);
        ++issued;
        if (++prod_stage == STAGES2) {
          prod_stage = 0;
          prod_phase ^= 1;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // -------------------------------------------------- MMA issuer (leader)
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int item = pair; item < total && !*abort_flag; item += num_pairs) {
      if (!mbar_wait(smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1, abort_flag)) {
        raise_abort2(sh, err);
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      bool ok = true;
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
  } else if (warp >= 2) {
    // -------------------------------------------------- epilogue (both CTAs)
    const int quarter = warp & 3;
    const int row_in_tile = static_cast<int>(rank) * 128 + quarter * 32 + lane;
    const uint32_t empty_leader[2] = {map_to_rank(smem_u32(&sh->tmem_empty[0]), 0),
                                      map_to_rank(smem_u32(&sh->tmem_empty[1]), 0)};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = pair; item < total; item += num_pairs) {
      const int n = item / m_pairs, mp = item % m_pairs;
      bool ok = mbar_wait(smem_u32(&sh->tmem_full[acc]), acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort2(sh, err);
        break;
      }
      tc_fence_after();
      float best = __int_as_float(0xff800000);
      int32_t best_id = kNoId;
      const int col0 = n * BN;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_ld_wait();
        const int cbase = col0 + c * 32;
        if (cbase < valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = __uint_as_float(r[i]);
            if (cbase + i < valid && scan_better(x, best)) {
              best = x;
              best_id = shard_start + cbase + i;
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
      const int row = mp * 256 + row_in_tile;
      if (row < M) {
        sga_stat st;
        st.v = best;
        st.id = best_id;
        ws[static_cast<size_t>(row) * n_tiles + n] = st;
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
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

// One warp per row: lanes stride over the row's per-tile partials (contiguous,
// row-major workspace) and merge them with the (value, id) order.
// Values of the fp8 variant are raw accumulators of the E4M3 codes until
// here; the positive row and weight scales (which cannot change the argmax of
// a row) are applied to the winning value only.
// The shards whose partials one finalize launch merges: row r of the output
// (shard r / M, hidden row r % M) reports shard start[r / M]'s first id when
// no partial has a valid id.
struct FinalizeShards {
  int n;
  int32_t start[kMaxLmShards];
};

__global__ void lmhead_finalize_kernel(const sga_stat *__restrict__ ws, int M, int n_tiles,
                                       const __grid_constant__ FinalizeShards shards,
                                       sga_stat *__restrict__ out,
                                       const float *__restrict__ row_scale, float w_scale,
                                       int scaled) {
  pdl_wait();  // the partials of the GEMM kernel are complete and visible
  pdl_launch_dependents();  // the next kernel may start its prologue
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= shards.n * M) return;
  const int shard_start = shards.start[r / M];
  float bv = __int_as_float(0xff800000);
  int32_t bi = kNoId;
  const sga_stat *row = ws + static_cast<size_t>(r) * n_tiles;
  constexpr int kInFlight = 4;  // loads issued before the first compare
  for (int n0 = lane; n0 < n_tiles; n0 += 32 * kInFlight) {
    sga_stat c[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int n = n0 + 32 * u;
      if (n < n_tiles) {
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

// Partial statistics go to ws[row * (*ws_stride) + part]; *ws_stride <=
// n_tiles, so a workspace of M x n_tiles stats always suffices.
template <bool kFp8>
cudaError_t launch_gemm(const void *hidden, int64_t M, int64_t H, const void *weight,
                        int64_t shard_start, int64_t valid, sga_stat *ws, int n_tiles, int num_sms,
                        uint32_t *err, cudaStream_t stream, int *ws_stride) {
  const int num_kb = static_cast<int>(H / kBk<kFp8>);
  *ws_stride = n_tiles;
  if (M <= SGA_LMHEAD_DECODE_MAX_M) {
    const int64_t row0 = 0;
    return launch_lmhead_decode(kFp8, hidden, M, H, weight, 1, &shard_start, &row0, &valid, ws,
                                num_sms, err, stream, ws_stride);
  }
  if (SGA_LMHEAD_2SM && M >= SGA_LMHEAD_2SM_MIN_M && num_sms >= 2) {
    // 2-SM tiles (256 rows per CTA pair)
    CUtensorMap map_a, map_b;
    if (!make_map(&map_a, hidden, M, H, 128, kFp8) || !make_map(&map_b, weight, valid, H, 128, kFp8))
      return cudaErrorInvalidValue;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(lmhead_argmax_2sm_kernel<kFp8>),
                                  SMEM2_BYTES, kFp8 ? 2 : 0);
    if (e != cudaSuccess) return e;
    const int m_pairs = static_cast<int>((M + 255) / 256);
    const int total = m_pairs * n_tiles;
    // A persistent grid must be fully resident: a cluster needs both CTAs in
    // one GPC, so fewer than num_sms / 2 pairs may fit at once.
    const int resident = resident_pairs<kFp8>(num_sms);
    if (resident <= 0) return cudaErrorLaunchOutOfResources;
    const int pairs = total < resident ? total : resident;
    return launch_pdl(lmhead_argmax_2sm_kernel<kFp8>, 2 * pairs, SMEM2_BYTES, stream, map_a,
                      map_b, static_cast<int>(M), num_kb, m_pairs, n_tiles,
                      static_cast<int>(valid), static_cast<int>(shard_start), ws, err);
  }
  CUtensorMap map_a, map_b;
  if (!make_map(&map_a, hidden, M, H, BM, kFp8) || !make_map(&map_b, weight, valid, H, BN, kFp8))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(lmhead_argmax_kernel<kFp8>),
                                SMEM_BYTES, kFp8 ? 3 : 1);
  if (e != cudaSuccess) return e;
  const int m_tiles = static_cast<int>((M + BM - 1) / BM);
  const int total = m_tiles * n_tiles;
  const int grid = total < num_sms ? total : num_sms;
  return launch_pdl(lmhead_argmax_kernel<kFp8>, grid, SMEM_BYTES, stream, map_a, map_b,
                    static_cast<int>(M), num_kb, m_tiles, n_tiles, static_cast<int>(valid),
                    static_cast<int>(shard_start), ws, err);
}

}  // namespace

cudaError_t launch_selftest_timeout(unsigned long long limit_ns, uint32_t *err,
                                    unsigned long long *waited_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, err, waited_ns);
  return cudaGetLastError();
}

// Partials per row: one per 256-id tile, and for decode sizes at least one per
// CTA of the decode kernel (up to kDecMaxParts), so that narrow shards still
// spread over every SM.  For M <= 64 the extra is at most 128 KB.
// Workspace of launch_lmhead_argmax_shards: decode sizes keep num_shards x M
// x (CTAs of the launch, at most kDecMaxParts) partials; larger M reuses one
// shard's workspace per shard.
size_t lmhead_shards_workspace_bytes(int64_t M, int num_shards, const int64_t *widths) {
  if (M <= SGA_LMHEAD_DECODE_MAX_M)
    return static_cast<size_t>(num_shards) * static_cast<size_t>(M) * kDecMaxParts *
           sizeof(sga_stat);
  size_t most = 0;
  for (int s = 0; s < num_shards; ++s) {
    const size_t b = lmhead_workspace_bytes(M, widths[s]);
    if (b > most) most = b;
  }
  return most;
}

size_t lmhead_workspace_bytes(int64_t M, int64_t width) {
  int64_t parts = (width + BN - 1) / BN;
  if (M <= SGA_LMHEAD_DECODE_MAX_M) {
    int64_t dec = (width + 127) / 128;
    if (dec > kDecMaxParts) dec = kDecMaxParts;
    if (dec > parts) parts = dec;
  }
  return static_cast<size_t>(parts * M) * sizeof(sga_stat);
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
  (void)width;
  sga_stat *ws = static_cast<sga_stat *>(workspace);
  const int n_tiles = static_cast<int>((valid + BN - 1) / BN);
  int ws_stride = n_tiles;  // partials per row in the workspace
  if (n_tiles > 0) {
    const cudaError_t e =
        fp8 ? launch_gemm<true>(hidden, M, H, weight, shard_start, valid, ws, n_tiles, num_sms,
                                err, stream, &ws_stride)
            : launch_gemm<false>(hidden, M, H, weight, shard_start, valid, ws, n_tiles, num_sms,
                                 err, stream, &ws_stride);
    if (e != cudaSuccess) return e;
  }
  FinalizeShards fs = {};
  fs.n = 1;
  fs.start[0] = static_cast<int32_t>(shard_start);
  return launch_finalize(ws, M, ws_stride, fs, out, row_scale, w_scale, fp8, stream);
}

cudaError_t launch_lmhead_argmax_shards(const void *hidden, int64_t M, int64_t H,
                                        const void *weight, int num_shards,
                                        const int64_t *starts, const int64_t *widths,
                                        const int64_t *valids, sga_stat *out, void *workspace,
                                        int num_sms, uint32_t *err, cudaStream_t stream,
                                        bool fp8, const float *row_scale, float w_scale) {
  sga_stat *ws = static_cast<sga_stat *>(workspace);
  if (M > SGA_LMHEAD_DECODE_MAX_M) {
    // tensor-bound sizes: one GEMM + finalize per shard, the workspace reused
    // (each launch waits for the previous one before touching it)
    const size_t row_bytes = static_cast<size_t>(H) * (fp8 ? 1 : 2);
    for (int s = 0; s < num_shards; ++s) {
      const void *w = static_cast<const char *>(weight) +
                      static_cast<size_t>(starts[s] - starts[0]) * row_bytes;
      const cudaError_t e =
          launch_lmhead_argmax(hidden, M, H, w, starts[s], widths[s], valids[s], out + s * M,
                               workspace, num_sms, err, stream, fp8, row_scale, w_scale);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  // decode sizes: every shard in one launch, one finalize for all of them
  int64_t row0s[kMaxLmShards];
  FinalizeShards fs = {};
  fs.n = num_shards;
  for (int s = 0; s < num_shards; ++s) {
    row0s[s] = starts[s] - starts[0];
    fs.start[s] = static_cast<int32_t>(starts[s]);
  }
  int ws_stride = 0;
  const cudaError_t e = launch_lmhead_decode(fp8, hidden, M, H, weight, num_shards, starts, row0s,
                                             valids, ws, num_sms, err, stream, &ws_stride);
  if (e != cudaSuccess) return e;
  return launch_finalize(ws, M, ws_stride, fs, out, row_scale, w_scale, fp8, stream);
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
