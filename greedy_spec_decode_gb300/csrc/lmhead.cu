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
// Every mbarrier wait is bounded in time; on expiry the CTA records
// SGA_DEVERR_TIMEOUT, stops issuing work, waits (bounded) for its own copies
// and MMAs in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace sga {
namespace {

constexpr int BM = 128;          // rows of hidden per tile (TMEM lanes)
constexpr int BN = 256;          // vocab ids per tile (TMEM columns)
constexpr int ROW_BYTES = 128;   // one 128-byte swizzled K-block row of a tile
// K-block in elements: 64 bf16 or 128 fp8 (E4M3) per 128-byte row
template <bool kFp8>
constexpr int kBk = kFp8 ? 128 : 64;
#ifndef SGA_LMHEAD_STAGES
#define SGA_LMHEAD_STAGES 4
#endif
#ifndef SGA_LMHEAD_2SM
#define SGA_LMHEAD_2SM 1  // 2-SM tiles when M >= SGA_LMHEAD_2SM_MIN_M
#endif
#ifndef SGA_LMHEAD_2SM_MIN_M
#define SGA_LMHEAD_2SM_MIN_M 129
#endif
#ifndef SGA_LMHEAD_DECODE_MAX_M
// Swapped-operand decode kernel for M <= this (0: off; at most 64).  Measured:
// an N = 128 variant for M = 65..128 was slower than the 1-SM kernel (graph
// replay, 2 shards: M = 128 bf16 210 vs 201 us, fp8 122 vs 114 us).
#define SGA_LMHEAD_DECODE_MAX_M 64
#endif
static_assert(SGA_LMHEAD_DECODE_MAX_M <= 64, "the decode kernel holds at most 64 hidden rows");
constexpr int STAGES = SGA_LMHEAD_STAGES;
constexpr int A_BYTES = BM * ROW_BYTES;   // 16 KB
constexpr int B_BYTES = BN * ROW_BYTES;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;           // 6 warps
constexpr int TMEM_COLS = 2 * BN;      // double-buffered accumulator
// At least 120 KB so that one CTA (holding all 512 TMEM columns) runs per SM.
constexpr int SMEM_NEEDED = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/;
constexpr int SMEM_BYTES = SMEM_NEEDED > 120 * 1024 ? SMEM_NEEDED : 120 * 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Wait for the phase of `parity` to complete, at most limit_ns.  Returns
// false on expiry (and on an abort raised by another role of this CTA).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int *abort_flag,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Bring one box of a tensor into L2 (no shared-memory destination, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored as 128-byte rows
// with the 128-byte swizzle (what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B):
// start address >> 4, leading offset unused (1), stride between 8-row groups
// 1024 B, descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma: fp32 accumulator (bits 4-5 = 1),
// A/B formats (bits 7-9, 10-12: bf16 = 1 for kind::f16, E4M3 = 0 for
// kind::f8f6f4), both operands K-major, N >> 3 at bit 17, M >> 4 at bit 24.
template <bool kFp8>
__host__ __device__ constexpr uint32_t instr_desc(uint32_t m, uint32_t n) {
  return (1u << 4) | (kFp8 ? 0u : ((1u << 7) | (1u << 10))) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

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

// Arrive once on `bar` when every tcgen05.mma issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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
// Decode-size variant (M <= 64 hidden rows): the operands swap roles.  The
// weight tile is the MMA's A operand (M = 128 vocab ids per MMA, two MMAs per
// 256-id tile) and the hidden rows are its B operand (N = kN = 16, 32 or 64
// columns).  A stage then holds 32-64 KB of weight and only kN x 128 B of
// hidden per K chunk (instead of 128 hidden rows, mostly zero fill), and each
// weight row is read 256-512 contiguous bytes at a time: at these sizes the
// kernel is a weight stream, paced by the length of its DRAM runs and the
// bytes in flight.
// TMEM lane = vocab id, TMEM column = hidden row.  The epilogue reduces each
// group of 32 (or 16) rows across the 32 lanes of a warp with a butterfly
// transpose-reduce in the (value, id) order, after which each lane holds one
// row's winner and keeps that row's running best; the four epilogue warps
// merge through shared memory at the end and each CTA writes one partial per
// row to the workspace (row stride = number of CTAs); the finalize kernel
// merges the CTAs' partials.
// ---------------------------------------------------------------------------
// K chunks (128-byte columns of the weight) per stage: 1 -> a stage holds 256
// weight rows x 128 B (a 256-id tile in two 128-row halves); 2 -> 128 rows x
// 256 B (a 128-id tile: twice the contiguous bytes per row); 4 -> 128 rows x
// 512 B.  Measured on GB300 (2 shards of 75968 x 4096, per step, bf16 / fp8):
//   N = 16 (M <= 16): 1 chunk 199 / 113 us, 2 chunks 201 / 113, 4 chunks
//                     193 / 108 (3 stages of 72 KB)
//   N = 32, 64:       1 chunk 203-208 / 117-122 us, 2 chunks 196-200 /
//                     110-115, 4 chunks 201-206 / 115-119 (only 2 stages)
// Longer contiguous runs per weight row pay more than extra bytes in flight.
#ifndef SGA_LMHEAD_DEC_PREFETCH
// L2 prefetch of the first stages before the PDL wait.  Measured (graph
// replay, 8 shards of 18992 ids): bf16 M = 1 223.7 -> 219.7 us per step, fp8
// 137.6 -> 133.2 us; 2 shards of 75968 ids unchanged.
#define SGA_LMHEAD_DEC_PREFETCH 1
#endif
#ifndef SGA_LMHEAD_DEC_CHUNKS_N16
#define SGA_LMHEAD_DEC_CHUNKS_N16 4
#endif
#ifndef SGA_LMHEAD_DEC_CHUNKS
#define SGA_LMHEAD_DEC_CHUNKS 2
#endif
template <int kN>
constexpr int dec_chunks = kN <= 16 ? SGA_LMHEAD_DEC_CHUNKS_N16 : SGA_LMHEAD_DEC_CHUNKS;
template <int kN>
constexpr int dec_halves = dec_chunks<kN> >= 2 ? 1 : 2;  // 128-id halves per tile
constexpr int DEC_SUB_BYTES = 128 * ROW_BYTES;            // one 128-row x 128-byte box
constexpr int kDecMaxParts = 256;  // CTAs (partials per row) of one decode launch, at most
template <int kN>
constexpr int dec_a_bytes = dec_chunks<kN> * dec_halves<kN> * DEC_SUB_BYTES;
template <int kN>
constexpr int dec_stage_bytes = dec_a_bytes<kN> + dec_chunks<kN> * kN * ROW_BYTES;
template <int kN>
constexpr int dec_stages = (227 * 1024 - 4096) / dec_stage_bytes<kN>;  // 3, 5, 4

template <int kN>
struct SharedDec {
  uint64_t full[dec_stages<kN>];
  uint64_t empty[dec_stages<kN>];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float part_v[4][kN];
  int32_t part_i[4][kN];
};

template <int kN>
constexpr int dec_smem_bytes =
    1024 + dec_stages<kN> * dec_stage_bytes<kN> + static_cast<int>(sizeof(SharedDec<kN>));
static_assert(dec_smem_bytes<16> <= 227 * 1024 && dec_smem_bytes<32> <= 227 * 1024 &&
                  dec_smem_bytes<64> <= 227 * 1024,
              "decode-size LM-head ring exceeds shared memory");

template <int kN>
__device__ __forceinline__ void raise_abort_dec(SharedDec<kN> *sh, uint32_t *err) {
  *reinterpret_cast<volatile int *>(&sh->abort) = 1;
  atomicOr(err, SGA_DEVERR_TIMEOUT);
}

// One MMA of a K step with M = 128 (weight rows) and N = kN (hidden rows).
template <bool kFp8, int kN>
__device__ __forceinline__ void mma_dec(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t accumulate) {
  constexpr uint32_t idesc = instr_desc<kFp8>(128, kN);
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Load kN accumulator columns of this warp's 32 TMEM lanes (x16 loads).
template <int kN>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[kN]) {
#pragma unroll
  for (int c = 0; c < kN / 16; ++c) tmem_ld16(taddr + 16 * c, r + 16 * c);
}

__device__ __forceinline__ void keep_better(float &v, int32_t &i, float ov, int32_t oi) {
  if (pair_beats(ov, oi, v, i)) {
    v = ov;
    i = oi;
  }
}

// Transpose-reduce of G rows (G = 16 or 32) across the 32 lanes of a warp:
// lane l holds x[k] = the logit of row k at its own vocab id `id`.  Each
// butterfly step pairs lane l with l ^ s; the lane with bit s set keeps the
// upper half of its current rows and receives the partner's values of them,
// the other lane keeps the lower half, and both merge with the (value, id)
// order.  After 31 merges (instead of 5 shuffle rounds per row), lane l holds
// the argmax over the warp's 32 ids of row l (G = 32) or row l / 2 (G = 16).
template <int kCnt, int kS>
__device__ __forceinline__ void butterfly_step(float *x, int32_t *xi, int lane) {
  if constexpr (kS >= 1) {
    if constexpr (kCnt > 1) {
      constexpr int kHalf = kCnt / 2;
      const bool upper = (lane & kS) != 0;
#pragma unroll
      for (int k = 0; k < kHalf; ++k) {
        const float sv = upper ? x[k] : x[kHalf + k];
        const int32_t si = upper ? xi[k] : xi[kHalf + k];
        float kv = upper ? x[kHalf + k] : x[k];
        int32_t ki = upper ? xi[kHalf + k] : xi[k];
        keep_better(kv, ki, __shfl_xor_sync(0xffffffffu, sv, kS),
                    __shfl_xor_sync(0xffffffffu, si, kS));
        x[k] = kv;
        xi[k] = ki;
      }
      butterfly_step<kHalf, kS / 2>(x, xi, lane);
    } else {
      keep_better(x[0], xi[0], __shfl_xor_sync(0xffffffffu, x[0], kS),
                  __shfl_xor_sync(0xffffffffu, xi[0], kS));
      butterfly_step<1, kS / 2>(x, xi, lane);
    }
  }
}

template <int G>
__device__ __forceinline__ void rows_argmax(float (&x)[G], int32_t id, int lane, float &out_v,
                                            int32_t &out_i) {
  int32_t xi[G];
#pragma unroll
  for (int k = 0; k < G; ++k) xi[k] = id;
  butterfly_step<G, 16>(x, xi, lane);
  out_v = x[0];
  out_i = xi[0];
}

template <bool kFp8, int kN>
__global__ void __launch_bounds__(THREADS, 1)
    lmhead_argmax_decode_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                const __grid_constant__ CUtensorMap tmap_h, int M, int num_kb,
                                int n_tiles, int valid, int shard_start,
                                sga_stat *__restrict__ ws, uint32_t *err) {
  constexpr int kStages = dec_stages<kN>;
  constexpr int kStageBytes = dec_stage_bytes<kN>;
  constexpr int kChunks = dec_chunks<kN>;
  constexpr int kHalves = dec_halves<kN>;
  constexpr int kTileIds = 128 * kHalves;
  constexpr int kCols = 2 * kHalves * kN;  // halves x two accumulator buffers
  constexpr int kG = kN < 32 ? kN : 32;  // rows per butterfly group
  constexpr int kSlots = kN / kG;         // groups (rows held per lane)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  SharedDec<kN> *sh = reinterpret_cast<SharedDec<kN> *>(base + kStages * kStageBytes);
  const volatile int *abort_flag = &sh->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (SGA_LMHEAD_DEC_PREFETCH && threadIdx.x == 64 && blockIdx.x < n_tiles) {
    // Warm L2 with what the ring loads first (this CTA's first tile, one
    // ring's worth of K blocks) while the previous kernel drains.  A prefetch
    // only moves lines into L2, which stays coherent with any later write, so
    // it may precede griddepcontrol.wait.
    const int n = blockIdx.x;
    for (int kb = 0; kb < num_kb && kb < kStages * kChunks; ++kb)
      for (int h = 0; h < kHalves; ++h)
        tma_prefetch_2d(&tmap_w, kb * kBk<kFp8>, n * kTileIds + h * 128);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
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
                 "r"(kCols)
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

  int prod_stage = 0;
  uint32_t prod_phase = 0;
  long long issued = 0;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      for (int n = blockIdx.x; n < n_tiles && !*abort_flag; n += gridDim.x) {
        for (int kb = 0; kb < num_kb; kb += kChunks) {
          if (!mbar_wait(smem_u32(&sh->empty[prod_stage]), prod_phase ^ 1, abort_flag)) {
            raise_abort_dec(sh, err);
            break;
          }
          const int chunks = num_kb - kb < kChunks ? num_kb - kb : kChunks;
          const uint32_t full = smem_u32(&sh->full[prod_stage]);
          const uint32_t stage_addr = smem_u32(base + prod_stage * kStageBytes);
          mbar_expect_tx(full, chunks * (kHalves * DEC_SUB_BYTES + kN * ROW_BYTES));
          for (int c = 0; c < chunks; ++c) {
            for (int h = 0; h < kHalves; ++h)
              tma_load_2d(stage_addr + (c * kHalves + h) * DEC_SUB_BYTES, &tmap_w,
                          (kb + c) * kBk<kFp8>, n * kTileIds + h * 128, full);
            tma_load_2d(stage_addr + dec_a_bytes<kN> + c * kN * ROW_BYTES, &tmap_h,
                        (kb + c) * kBk<kFp8>, 0, full);
          }
          ++issued;
          if (++prod_stage == kStages) {
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
      for (int n = blockIdx.x; n < n_tiles && !*abort_flag; n += gridDim.x) {
        if (!mbar_wait(smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1, abort_flag)) {
          raise_abort_dec(sh, err);
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < num_kb; kb += kChunks) {
          if (!mbar_wait(smem_u32(&sh->full[stage]), phase, abort_flag)) {
            raise_abort_dec(sh, err);
            ok = false;
            break;
          }
          tc_fence_after();
          const int chunks = num_kb - kb < kChunks ? num_kb - kb : kChunks;
          const uint32_t stage_addr = smem_u32(base + stage * kStageBytes);
          for (int c = 0; c < chunks; ++c) {
            const uint64_t b_desc = smem_desc_sw128(stage_addr + dec_a_bytes<kN> + c * kN * ROW_BYTES);
#pragma unroll
            for (int h = 0; h < kHalves; ++h) {
              const uint64_t a_desc =
                  smem_desc_sw128(stage_addr + (c * kHalves + h) * DEC_SUB_BYTES);
              const uint32_t d_tmem = tmem_base + (acc * kHalves + h) * kN;
#pragma unroll
              for (int kk = 0; kk < ROW_BYTES / 32; ++kk)  // 32 bytes = 2 descriptor units
                mma_dec<kFp8, kN>(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk,
                                  (kb | c | kk) != 0);
            }
          }
          mma_commit(smem_u32(&sh->empty[stage]));
          if (++stage == kStages) {
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
    float rv[kSlots];
    int32_t ri[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
      rv[s] = __int_as_float(0xff800000);
      ri[s] = kNoId;
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int n = blockIdx.x; n < n_tiles; n += gridDim.x) {
      bool ok = mbar_wait(smem_u32(&sh->tmem_full[acc]), acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort_dec(sh, err);
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < kHalves; ++h) {
        const int local = n * kTileIds + h * 128 + quarter * 32 + lane;  // shard-local id
        const bool live = local < valid;
        const int32_t id = live ? shard_start + local : kNoId;
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + (acc * kHalves + h) * kN;
#pragma unroll
        for (int g = 0; g < kSlots; ++g) {
          uint32_t r[kG];  // one group of columns at a time
          tmem_ld_cols<kG>(taddr + g * kG, r);
          tmem_ld_wait();
          float x[kG];
#pragma unroll
          for (int k = 0; k < kG; ++k)
            x[k] = live ? __uint_as_float(r[k]) : __int_as_float(0xff800000);
          float v;
          int32_t i;
          rows_argmax<kG>(x, id, lane, v, i);
          keep_better(rv[g], ri[g], v, i);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sh->tmem_empty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
#pragma unroll
    for (int g = 0; g < kSlots; ++g) {
      // lane l holds row l of the group (kG = 32) or row l / 2 (kG = 16; both
      // lanes of a pair hold it)
      if (kG == 32 || (lane & 1) == 0) {
        const int j = g * kG + (kG == 32 ? lane : lane >> 1);
        sh->part_v[quarter][j] = rv[g];
        sh->part_i[quarter][j] = ri[g];
      }
    }
  }

  pdl_launch_dependents();
  __syncthreads();
  if (*abort_flag) {
    // Let this CTA's own copies and MMAs land before its shared memory and
    // tensor memory are released (bounded as well).
    const int zero = 0;
    if (warp == 0 && lane == 0) {
      const long long outstanding = issued < kStages ? issued : kStages;
      for (long long i = 1; i <= outstanding; ++i) {
        int s = prod_stage - static_cast<int>(i);
        uint32_t ph = prod_phase;
        if (s < 0) {
          s += kStages;
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
  if (threadIdx.x < M) {
    // merge the four epilogue warps' bests of row threadIdx.x (any order: the
    // (value, id) order is total)
    float v = sh->part_v[0][threadIdx.x];
    int32_t id = sh->part_i[0][threadIdx.x];
#pragma unroll
    for (int q = 1; q < 4; ++q) {
      const float cv = sh->part_v[q][threadIdx.x];
      const int32_t ci = sh->part_i[q][threadIdx.x];
      if (pair_beats(cv, ci, v, id)) {
        v = cv;
        id = ci;
      }
    }
    sga_stat st;
    st.v = v;
    st.id = id;
    ws[static_cast<size_t>(threadIdx.x) * gridDim.x + blockIdx.x] = st;
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kCols)
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
__global__ void lmhead_finalize_kernel(const sga_stat *__restrict__ ws, int M, int n_tiles,
                                       int shard_start, sga_stat *__restrict__ out,
                                       const float *__restrict__ row_scale, float w_scale,
                                       int scaled) {
  pdl_wait();  // the partials of the GEMM kernel are complete and visible
  pdl_launch_dependents();  // the next kernel may start its prologue
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= M) return;
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
    s.v = scaled ? bv * ((row_scale ? row_scale[r] : 1.0f) * w_scale) : bv;
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

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor map over a row-major [rows, cols] matrix of bf16 or fp8 (E4M3,
// stored as bytes); box = box_rows x one 128-byte row (64 bf16 or 128 fp8
// columns), 128-byte swizzle, zero fill outside.
bool make_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, int box_rows,
              bool fp8) {
  auto encode = get_encode_fn();
  if (encode == nullptr) return false;
  const int elt = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * elt)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(ROW_BYTES / elt), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared-memory limit once per device (slot picks the
// kernel), so that later calls, including calls inside a stream capture, make
// no function-attribute call.
cudaError_t set_smem_once(const void *kernel, int bytes, int slot) {
  static std::mutex mu;
  static bool done[12][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[slot][dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[slot][dev] = true;
  }
  return cudaSuccess;
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

// Launch a GEMM kernel (THREADS threads per CTA) with programmatic stream
// serialisation; the kernel calls griddepcontrol.wait after its prologue.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <bool kFp8, int kN>
cudaError_t launch_decode(const void *hidden, int64_t M, int64_t H, const void *weight,
                          int64_t shard_start, int64_t valid, sga_stat *ws, int n_tiles,
                          int num_sms, uint32_t *err, cudaStream_t stream, int *ws_stride) {
  CUtensorMap map_w, map_h;
  if (!make_map(&map_w, weight, valid, H, 128, kFp8) || !make_map(&map_h, hidden, M, H, kN, kFp8))
    return cudaErrorInvalidValue;
  auto kern = lmhead_argmax_decode_kernel<kFp8, kN>;
  const int slot = 4 + (kFp8 ? 4 : 0) + (kN == 16 ? 0 : kN == 32 ? 1 : kN == 64 ? 2 : 3);
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), dec_smem_bytes<kN>, slot);
  if (e != cudaSuccess) return e;
  // one CTA per SM, at most one per tile; the workspace holds
  // min(ceil(width / 128), kDecMaxParts) partials per row for M <= 64
  (void)n_tiles;
  const int tile_ids = 128 * dec_halves<kN>;
  const int dec_tiles = static_cast<int>((valid + tile_ids - 1) / tile_ids);
  int grid = dec_tiles < num_sms ? dec_tiles : num_sms;
  if (grid > kDecMaxParts) grid = kDecMaxParts;
  *ws_stride = grid;
  return launch_pdl(kern, grid, dec_smem_bytes<kN>, stream, map_w, map_h, static_cast<int>(M),
                    static_cast<int>(H / kBk<kFp8>), dec_tiles, static_cast<int>(valid),
                    static_cast<int>(shard_start), ws, err);
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
    if (M <= 16)
      return launch_decode<kFp8, 16>(hidden, M, H, weight, shard_start, valid, ws, n_tiles,
                                     num_sms, err, stream, ws_stride);
    if (M <= 32)
      return launch_decode<kFp8, 32>(hidden, M, H, weight, shard_start, valid, ws, n_tiles,
                                     num_sms, err, stream, ws_stride);
    return launch_decode<kFp8, 64>(hidden, M, H, weight, shard_start, valid, ws, n_tiles,
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
size_t lmhead_workspace_bytes(int64_t M, int64_t width) {
  int64_t parts = (width + BN - 1) / BN;
  if (M <= SGA_LMHEAD_DECODE_MAX_M) {
    int64_t dec = (width + 127) / 128;
    if (dec > kDecMaxParts) dec = kDecMaxParts;
    if (dec > parts) parts = dec;
  }
  return static_cast<size_t>(parts * M) * sizeof(sga_stat);
}

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
  // 8 rows per block; programmatic dependent launch lets the blocks become
  // resident while the GEMM kernel drains (they wait in pdl_wait()).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((M + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lmhead_finalize_kernel, static_cast<const sga_stat *>(ws),
                            static_cast<int>(M), ws_stride, static_cast<int>(shard_start), out,
                            row_scale, w_scale, fp8 ? 1 : 0);
}

}  // namespace sga

// ---------------------------------------------------------------------------
// Scratch for sga_lmhead_argmax_noalloc: the per-tile partial statistics live
// in this fixed array instead of a caller-provided workspace.  Host code must
// not use the array's name as a device pointer (on the host it only stands in
// for the symbol); lmhead_noalloc_scratch() looks up its device address once
// per device, with that device current.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoallocScratchBytes = SGA_LMHEAD_NOALLOC_SCRATCH_BYTES;
constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
sga_stat *g_noalloc_ptr[kNoallocMaxDevices];
}  // namespace

static __device__ __align__(256) sga_stat g_lmhead_noalloc_scratch[kNoallocScratchBytes / sizeof(sga_stat)];

namespace sga {

size_t lmhead_noalloc_scratch_bytes() { return kNoallocScratchBytes; }

cudaError_t lmhead_noalloc_scratch(sga_stat **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lmhead_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<sga_stat *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace sga
