// lmhead_decode.cu -- fused LM head + per-shard argmax at decode sizes
// (M <= 128 hidden rows: one CTA per SM up to M = 64, CTA pairs above) on the
// tcgen05 tensor cores, with the weight as the MMA's 128-row operand.
//
// vLLM PR #62604, Purpose (vocab-parallel LM head) and item 2 (fused
// get_top_tokens); vLLM PR #39419, Changes (lm_head on the hidden states,
// then the local argmax).  At decode sizes the step is a weight stream, so
// these kernels are shaped for HBM, not for the tensor pipe.
#include <atomic>

#include "tcgen05.cuh"

namespace sga {
namespace {

// ---------------------------------------------------------------------------
// One-CTA decode kernel (M <= 64 hidden rows): the operands swap roles.  The
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
// row's winner and keeps that row's running best; at each shard edge the
// four epilogue warps merge through shared memory and the CTA merges its
// winners into library-owned keys (atomicMax); the last CTA writes the stats.
// CTAs take tiles one at a time from a counter of the launch, so an SM that
// the memory system serves faster streams more of the weight.
// ---------------------------------------------------------------------------
// K chunks (128-byte columns of the weight) per stage: 1 -> a stage holds 256
// weight rows x 128 B (a 256-id tile in two 128-row halves); 2 -> 128 rows x
// 256 B (a 128-id tile: twice the contiguous bytes per row); 4 -> 128 rows x
// 512 B.  Measured on GB300 (2 shards of 75968 x 4096, per step, bf16 / fp8):
//   N = 16 (M <= 16): 1 chunk 199 / 113 us, 2 chunks 201 / 113, 4 chunks
//                     193 / 108 (3 stages of 72 KB)
//   N = 32, 64:       1 chunk 203-208 / 117-122 us, 2 chunks 196-200 /
//                     110-115, 4 chunks 201-206 / 115-119 (only 2 stages);
//                     later, alternating on one box (M = 24 / 32 / 48 / 64):
//                     2 chunks (4-5 stages) 181.5 / 181.4 / 184.0 / 183.9
//                     and 97.0 / 96.7 / 99.0 / 98.5 us, 3 chunks (3 stages)
//                     180.8 / 180.6 / 183.4 / 183.3 and 96.5 / 96.3 / 98.7 /
//                     98.4, 4 chunks 185.0-188.0 and 99.0-102.0
// Longer contiguous runs per weight row pay more than extra bytes in flight,
// up to the point where the ring has only 2 stages.
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
#define SGA_LMHEAD_DEC_CHUNKS 3
#endif
template <int kN>
constexpr int dec_chunks = kN <= 16 ? SGA_LMHEAD_DEC_CHUNKS_N16 : SGA_LMHEAD_DEC_CHUNKS;
template <int kN>
constexpr int dec_halves = dec_chunks<kN> >= 2 ? 1 : 2;  // 128-id halves per tile
constexpr int DEC_SUB_BYTES = 128 * ROW_BYTES;            // one 128-row x 128-byte box
template <int kN>
constexpr int dec_a_bytes = dec_chunks<kN> * dec_halves<kN> * DEC_SUB_BYTES;
template <int kN>
constexpr int dec_stage_bytes = dec_a_bytes<kN> + dec_chunks<kN> * kN * ROW_BYTES;
template <int kN>
constexpr int dec_stages = (227 * 1024 - 4096) / dec_stage_bytes<kN>;  // 3, 3, 3

constexpr int kTileQ = 8;  // entries of the tile queue

template <int kN>
struct SharedDec {
  uint64_t full[dec_stages<kN>];
  uint64_t empty[dec_stages<kN>];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int is_last;
  float part_v[4][kN];
  int32_t part_i[4][kN];
  // the CTA's tiles, in the order the producer took them: entry k % kTileQ
  // holds the k-th (-1 after the last); ready: 1 arrival (the producer),
  // free: 5 (the MMA lane and the four epilogue warps, once read)
  uint64_t tile_ready[kTileQ];
  uint64_t tile_free[kTileQ];
  int32_t tile_q[kTileQ];
};

// Cross-CTA merge of a decode launch, in library-owned device memory: each
// CTA folds its (shard, row) winners into 64-bit keys with atomicMax; the
// last CTA to finish (a ticket) turns the keys into the statistics, scales
// fp8 values, and resets keys and ticket to zero for the next launch that
// uses the slot.  A launch takes slot (call number mod kMergeSlots); launches
// that share a slot must not overlap on the GPU.
constexpr int kMergeSlots = 32;
constexpr int kMergeKeys = kMaxLmShards * SGA_LMHEAD_DECODE_MAX_M;  // shards x rows
__device__ unsigned long long g_dec_keys[kMergeSlots][kMergeKeys];
__device__ unsigned int g_dec_ticket[kMergeSlots];
// the next tile of a launch: CTAs take tiles one at a time, so SMs that the
// memory system serves faster take more (cleared with the slot)
__device__ unsigned int g_dec_next[kMergeSlots];

// The merge slot of a call: one counter for every decode launch of the
// process (all kernels and types), so that at most 32 calls in flight never
// share a slot.
int take_merge_slot() {
  static std::atomic<unsigned> next_slot{0};
  return static_cast<int>(next_slot.fetch_add(1) % kMergeSlots);
}

// Key of a (value, id) pair whose unsigned order is the argmax order: the
// high word orders values (NaN above +inf, +0 and -0 equal), the low word
// (0xffffffff - id) puts the lower id above on equal values.  Key 0 is below
// every pair (an empty slot).
__device__ __forceinline__ unsigned long long merge_key(float v, int32_t id) {
  const uint32_t b = __float_as_uint(v);
  uint32_t o;
  if (is_nan(v))
    o = 0xffffffffu;
  else if ((b & 0x7fffffffu) == 0)
    o = 0x80000000u;
  else
    o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | (0xffffffffu - static_cast<uint32_t>(id));
}

// The pair of a nonzero key (a NaN comes back as the canonical quiet NaN,
// -0 as +0).
__device__ __forceinline__ void merge_unkey(unsigned long long key, float &v, int32_t &id) {
  const uint32_t o = static_cast<uint32_t>(key >> 32);
  id = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(key));
  if (o == 0xffffffffu)
    v = __uint_as_float(0x7fc00000u);
  else
    v = __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// The shards of one launch (one, or all the shards a GPU holds): shard s
// covers global ids [start, start + valid) (its non-padding ids) at weight
// rows row0 .. row0 + valid - 1 of the launch's weight map, and its tiles are
// numbers tile0[s] .. tile0[s + 1] - 1 of the launch.
struct DecShardTable {
  int n;
  int32_t start[kMaxLmShards];
  int32_t row0[kMaxLmShards];
  int32_t valid[kMaxLmShards];
  int32_t tile0[kMaxLmShards + 1];
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

// The end of every decode launch, after the CTA's merges and its barrier:
// each CTA takes one ticket (also after an abort, so the count always returns
// to zero) and the last one turns the keys into statistics and clears the
// slot (keys, tile counter, ticket) for a later launch.  The keys, the tile
// counter and the ticket are touched by atomics alone, which are performed in
// L2: every merge of a CTA was performed before its epilogue threads passed
// their fence, so before the CTA's barrier and its ticket, and the last CTA's
// exchanges are issued after it has seen every ticket (no further fence
// needed; each measured at about 0.3 us on the launch's critical path).
__device__ __forceinline__ void finish_launch(int *is_last, const DecShardTable &tab, int M,
                                              int slot, sga_stat *__restrict__ out,
                                              const float *__restrict__ row_scale,
                                              float w_scale, int scaled) {
  if (threadIdx.x == 0) *is_last = atomicAdd(&g_dec_ticket[slot], 1u) == gridDim.x - 1;
  __syncthreads();
  if (*is_last) {
    for (int r = threadIdx.x; r < tab.n * M; r += blockDim.x) {
      const unsigned long long key = atomicExch(&g_dec_keys[slot][r], 0ull);
      sga_stat st;
      if (key == 0) {
        st.v = __int_as_float(0xff800000);  // no element of the shard: its first id, -inf
        st.id = tab.start[r / M];
      } else {
        merge_unkey(key, st.v, st.id);
        if (scaled) st.v *= (row_scale ? row_scale[r % M] : 1.0f) * w_scale;
      }
      out[r] = st;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      atomicExch(&g_dec_next[slot], 0u);
      atomicExch(&g_dec_ticket[slot], 0u);
    }
  }
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
                                const __grid_constant__ DecShardTable tab, int slot,
                                sga_stat *__restrict__ out, const float *__restrict__ row_scale,
                                float w_scale, int scaled, uint32_t *err) {
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
  const int n_tiles = tab.tile0[tab.n];

  if (SGA_LMHEAD_DEC_PREFETCH && threadIdx.x == 64 && blockIdx.x < n_tiles) {
    // Warm L2 with what the ring loads first (the CTA's first tile,
    // blockIdx.x; one ring's worth of K blocks) while the previous kernel
    // drains.  A prefetch
    // only moves lines into L2, which stays coherent with any later write, so
    // it may precede griddepcontrol.wait.
    const int n = blockIdx.x;
    int s = 0;
    while (n >= tab.tile0[s + 1]) ++s;
    const int row = tab.row0[s] + (n - tab.tile0[s]) * kTileIds;
    for (int kb = 0; kb < num_kb && kb < kStages * kChunks; ++kb)
      for (int h = 0; h < kHalves; ++h)
        tma_prefetch_2d(&tmap_w, kb * kBk<kFp8>, row + h * 128);
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
    for (int q = 0; q < kTileQ; ++q) {
      mbar_init(smem_u32(&sh->tile_ready[q]), 1);
      mbar_init(smem_u32(&sh->tile_free[q]), 1 + 4);
    }
    sh->abort = 0;
    sh->is_last = 0;
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
      // The CTA's first tile is its own (blockIdx.x: no round trip before the
      // first copy, and the tile the L2 prefetch warmed); the others come
      // from the launch's counter, offset by the grid, one at a time (the
      // next one is taken while the current one streams).  They go to the
      // MMA lane and the epilogue through the tile queue and only increase.
      int s = 0;  // the shard of tile n
      int n = blockIdx.x;
      for (int k = 0; !*abort_flag; ++k) {
        const int q = k % kTileQ;
        if (k >= kTileQ &&
            !mbar_wait(smem_u32(&sh->tile_free[q]), ((k / kTileQ) - 1) & 1, abort_flag)) {
          raise_abort_dec(sh, err);
          break;
        }
        sh->tile_q[q] = n < n_tiles ? n : -1;
        mbar_arrive(smem_u32(&sh->tile_ready[q]));
        if (n >= n_tiles) break;
        const int n_next =
            static_cast<int>(gridDim.x) + static_cast<int>(atomicAdd(&g_dec_next[slot], 1u));
        while (n >= tab.tile0[s + 1]) ++s;
        const int row = tab.row0[s] + (n - tab.tile0[s]) * kTileIds;
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
                          (kb + c) * kBk<kFp8>, row + h * 128, full);
            tma_load_2d(stage_addr + dec_a_bytes<kN> + c * kN * ROW_BYTES, &tmap_h,
                        (kb + c) * kBk<kFp8>, 0, full);
          }
          ++issued;
          if (++prod_stage == kStages) {
            prod_stage = 0;
            prod_phase ^= 1;
          }
        }
        n = n_next;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int k = 0; !*abort_flag; ++k) {
        const int q = k % kTileQ;
        if (!mbar_wait(smem_u32(&sh->tile_ready[q]), (k / kTileQ) & 1, abort_flag)) {
          raise_abort_dec(sh, err);
          break;
        }
        const int n = sh->tile_q[q];
        mbar_arrive(smem_u32(&sh->tile_free[q]));
        if (n < 0) break;
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
    // The CTA's tiles cross each shard edge at most once, in shard order.  At
    // every edge (and for every shard without a tile of this CTA) the four
    // epilogue warps flush the shard's per-row bests: each writes its rows'
    // bests to shared memory, then epilogue thread e < M merges row e's four
    // and stores the CTA's partial of (shard, row e).  Every warp flushes
    // every shard exactly once, in order, also after an abort, so the
    // 128-thread barriers of the flushes always match.
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
    const int e = static_cast<int>(threadIdx.x) - 64;  // epilogue thread 0 .. 127
    float rv[kSlots];
    int32_t ri[kSlots];
#pragma unroll
    for (int g = 0; g < kSlots; ++g) {
      rv[g] = __int_as_float(0xff800000);
      ri[g] = kNoId;
    }
    auto flush = [&](int s) {
#pragma unroll
      for (int g = 0; g < kSlots; ++g) {
        // lane l holds row l of the group (kG = 32) or row l / 2 (kG = 16;
        // both lanes of a pair hold it)
        if (kG == 32 || (lane & 1) == 0) {
          const int j = g * kG + (kG == 32 ? lane : lane >> 1);
          sh->part_v[quarter][j] = rv[g];
          sh->part_i[quarter][j] = ri[g];
        }
        rv[g] = __int_as_float(0xff800000);
        ri[g] = kNoId;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (e < M) {
        // (any order: the (value, id) order is total)
        float v = sh->part_v[0][e];
        int32_t id = sh->part_i[0][e];
#pragma unroll
        for (int q = 1; q < 4; ++q) keep_better(v, id, sh->part_v[q][e], sh->part_i[q][e]);
        if (id != kNoId) atomicMax(&g_dec_keys[slot][s * M + e], merge_key(v, id));
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // before the next flush's writes
    };
    int cur = 0;  // the shard whose bests rv / ri hold
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = 0;; ++t) {
      const int q = t % kTileQ;
      bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sh->tile_ready[q]),
                                                  (t / kTileQ) & 1, abort_flag));
      if (!ok) {
        if (lane == 0) raise_abort_dec(sh, err);
        break;
      }
      const int n = sh->tile_q[q];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->tile_free[q]));
      if (n < 0) break;
      while (n >= tab.tile0[cur + 1]) flush(cur++);
      ok = mbar_wait(smem_u32(&sh->tmem_full[acc]), acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort_dec(sh, err);
        break;
      }
      tc_fence_after();
      const int tile_local = (n - tab.tile0[cur]) * kTileIds;
#pragma unroll 1
      for (int h = 0; h < kHalves; ++h) {
        const int local = tile_local + h * 128 + quarter * 32 + lane;  // shard-local id
        const bool live = local < tab.valid[cur];
        const int32_t id = live ? tab.start[cur] + local : kNoId;
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
    while (cur < tab.n) flush(cur++);
    __threadfence();  // this CTA's merges before its ticket
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
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kCols)
                 : "memory");
  }
  finish_launch(&sh->is_last, tab, M, slot, out, row_scale, w_scale, scaled);
}

// ---------------------------------------------------------------------------
// Pair variant for 65 <= M <= 128 hidden rows (kN = 128): a cluster of two
// CTAs issues tcgen05.mma.cta_group::2 with M = 256 weight rows (each CTA
// holds 128 of them, a 256-id tile per pair) and N = kN hidden rows, each CTA
// holding kN / 2 of those.  A one-CTA kernel at N = 128 must stage as many
// hidden bytes as weight bytes per stage; split across the pair, a stage is
// 2 K blocks x (128 weight rows + 64 hidden rows) per CTA, 4 stages.  Each
// CTA's tensor memory receives its 128 ids x kN hidden rows, so the epilogue
// is the one-CTA kernel's.  Pair p takes tiles p, p + pairs, ...
// ---------------------------------------------------------------------------
#ifndef SGA_LMHEAD_PAIR_CHUNKS
// K blocks per stage: 2 (4 stages of 256 bytes per weight row); measured
// against 3 (3 stages, 384 bytes) and 1 (9 stages, 128 bytes), alternating on
// one box, M = 96 / 128, graph replay: bf16 191.0 / 192.0 us against 191.7 /
// 192.8 and 190.4 / 191.3; fp8 106.2 / 107.7 against 106.9 / 109.0 and 108.1 /
// 109.8.  A tile queue fed by the leader (tiles from the launch's counter, as
// in the one-CTA kernel) was slower: 197.8 - 199.6 us against 195.5 - 197.3
// (bf16) and 109.5 - 111.0 against 107.5 - 110.0 (fp8), on boxes where the
// one-SM GEMM kernel it replaces took 205.7 - 206.8 and 116.5 - 117.4 us.
#define SGA_LMHEAD_PAIR_CHUNKS 2
#endif
constexpr int kPairChunks = SGA_LMHEAD_PAIR_CHUNKS;           // K blocks per stage
constexpr int kPairABytes = kPairChunks * DEC_SUB_BYTES;      // 128 weight rows
template <int kN>
constexpr int pair_b_bytes = kPairChunks * (kN / 2) * ROW_BYTES;  // this CTA's hidden rows
template <int kN>
constexpr int pair_stage_bytes = kPairABytes + pair_b_bytes<kN>;
template <int kN>
constexpr int pair_stages = (227 * 1024 - 4096) / pair_stage_bytes<kN>;

template <int kN>
struct SharedPair {
  uint64_t full[pair_stages<kN>];   // leader: both CTAs' copies of a stage landed
  uint64_t empty[pair_stages<kN>];  // both: the stage's MMAs are done
  uint64_t tmem_full[2];            // both: an accumulator is complete
  uint64_t tmem_empty[2];           // leader: the pair's 8 epilogue warps read it
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int is_last;
  float part_v[4][kN];
  int32_t part_i[4][kN];
};

template <int kN>
constexpr int pair_smem_bytes =
    1024 + pair_stages<kN> * pair_stage_bytes<kN> + static_cast<int>(sizeof(SharedPair<kN>));
static_assert(pair_stages<128> >= 3 && pair_smem_bytes<128> <= 227 * 1024,
              "pair decode ring exceeds shared memory");

template <int kN>
__device__ __forceinline__ void raise_abort_pair(SharedPair<kN> *sh, uint32_t *err) {
  *reinterpret_cast<volatile int *>(&sh->abort) = 1;
  atomicOr(err, SGA_DEVERR_TIMEOUT);
}

template <bool kFp8, int kN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    lmhead_argmax_decode_pair_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                     const __grid_constant__ CUtensorMap tmap_h, int M,
                                     int num_kb, const __grid_constant__ DecShardTable tab,
                                     int slot, sga_stat *__restrict__ out,
                                     const float *__restrict__ row_scale, float w_scale,
                                     int scaled, uint32_t *err) {
  constexpr int kStages = pair_stages<kN>;
  constexpr int kStageBytes = pair_stage_bytes<kN>;
  constexpr int kChunks = kPairChunks;
  constexpr int kHalfN = kN / 2;           // hidden rows in each CTA's B half
  constexpr int kTileIds = 256;            // 128 weight rows per CTA
  constexpr int kCols = 2 * kN;            // two accumulator buffers
  constexpr int kG = 32;                   // rows per butterfly group
  constexpr int kSlots = kN / kG;          // groups (rows held per lane)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  SharedPair<kN> *sh = reinterpret_cast<SharedPair<kN> *>(base + kStages * kStageBytes);
  const volatile int *abort_flag = &sh->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);
  const int n_tiles = tab.tile0[tab.n];

  if (SGA_LMHEAD_DEC_PREFETCH && threadIdx.x == 64 && pair < n_tiles) {
    // warm L2 with this CTA's rows of its first tile (one ring of K blocks)
    int s = 0;
    while (pair >= tab.tile0[s + 1]) ++s;
    const int row = tab.row0[s] + (pair - tab.tile0[s]) * kTileIds + static_cast<int>(rank) * 128;
    for (int kb = 0; kb < num_kb && kb < kStages * kChunks; ++kb)
      tma_prefetch_2d(&tmap_w, kb * kBk<kFp8>, row);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh->tmem_full[b]), 1);
      mbar_init(smem_u32(&sh->tmem_empty[b]), 8);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort = 0;
    sh->is_last = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  pdl_wait();

  int prod_stage = 0;
  uint32_t prod_phase = 0;
  long long issued = 0;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------- producer (both CTAs)
    int s = 0;
    for (int n = pair; n < n_tiles && !*abort_flag; n += num_pairs) {
      while (n >= tab.tile0[s + 1]) ++s;
      const int row =
          tab.row0[s] + (n - tab.tile0[s]) * kTileIds + static_cast<int>(rank) * 128;
      for (int kb = 0; kb < num_kb; kb += kChunks) {
        if (!mbar_wait(smem_u32(&sh->empty[prod_stage]), prod_phase ^ 1, abort_flag)) {
          raise_abort_pair(sh, err);
          break;
        }
        const int chunks = num_kb - kb < kChunks ? num_kb - kb : kChunks;
        const uint32_t full_leader = map_to_rank(smem_u32(&sh->full[prod_stage]), 0);
        const uint32_t stage_addr = smem_u32(base + prod_stage * kStageBytes);
        // the leader's barrier counts the bytes of both CTAs
        if (leader)
          mbar_expect_tx(smem_u32(&sh->full[prod_stage]),
                         2 * chunks * (DEC_SUB_BYTES + kHalfN * ROW_BYTES));
        for (int c = 0; c < chunks; ++c) {
          tma_load_2d_pair(stage_addr + c * DEC_SUB_BYTES, &tmap_w, (kb + c) * kBk<kFp8>, row,
                           full_leader);
          tma_load_2d_pair(stage_addr + kPairABytes + c * kHalfN * ROW_BYTES, &tmap_h,
                           (kb + c) * kBk<kFp8>, static_cast<int>(rank) * kHalfN, full_leader);
        }
        ++issued;
        if (++prod_stage == kStages) {
          prod_stage = 0;
          prod_phase ^= 1;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // -------------------------------------------------- MMA issuer (leader)
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int n = pair; n < n_tiles && !*abort_flag; n += num_pairs) {
      if (!mbar_wait(smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1, abort_flag)) {
        raise_abort_pair(sh, err);
        break;
      }
      tc_fence_after();
      bool ok = true;
      for (int kb = 0; kb < num_kb; kb += kChunks) {
        if (!mbar_wait(smem_u32(&sh->full[stage]), phase, abort_flag)) {
          raise_abort_pair(sh, err);
          ok = false;
          break;
        }
        tc_fence_after();
        const int chunks = num_kb - kb < kChunks ? num_kb - kb : kChunks;
        const uint32_t stage_addr = smem_u32(base + stage * kStageBytes);
        for (int c = 0; c < chunks; ++c) {
          const uint64_t a_desc = smem_desc_sw128(stage_addr + c * DEC_SUB_BYTES);
          const uint64_t b_desc = smem_desc_sw128(stage_addr + kPairABytes + c * kHalfN * ROW_BYTES);
#pragma unroll
          for (int kk = 0; kk < ROW_BYTES / 32; ++kk)  // 32 bytes = 2 descriptor units
            mma_pair<kFp8, kN>(tmem_base + acc * kN, a_desc + 2 * kk, b_desc + 2 * kk,
                               (kb | c | kk) != 0);
        }
        mma_commit_pair(smem_u32(&sh->empty[stage]));
        if (++stage == kStages) {
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
    // ------------------------------------------------- epilogue (both CTAs)
    // As in the one-CTA kernel: TMEM lane = this CTA's weight row (vocab id),
    // column = hidden row; every warp flushes every shard exactly once, in
    // order, also after an abort, so the 128-thread barriers always match.
    const int quarter = warp & 3;
    const int e = static_cast<int>(threadIdx.x) - 64;  // epilogue thread 0 .. 127
    const uint32_t empty_leader[2] = {map_to_rank(smem_u32(&sh->tmem_empty[0]), 0),
                                      map_to_rank(smem_u32(&sh->tmem_empty[1]), 0)};
    float rv[kSlots];
    int32_t ri[kSlots];
#pragma unroll
    for (int g = 0; g < kSlots; ++g) {
      rv[g] = __int_as_float(0xff800000);
      ri[g] = kNoId;
    }
    auto flush = [&](int s) {
#pragma unroll
      for (int g = 0; g < kSlots; ++g) {
        const int j = g * kG + lane;  // lane l holds row l of group g
        sh->part_v[quarter][j] = rv[g];
        sh->part_i[quarter][j] = ri[g];
        rv[g] = __int_as_float(0xff800000);
        ri[g] = kNoId;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (e < M) {
        float v = sh->part_v[0][e];
        int32_t id = sh->part_i[0][e];
#pragma unroll
        for (int q = 1; q < 4; ++q) keep_better(v, id, sh->part_v[q][e], sh->part_i[q][e]);
        if (id != kNoId) atomicMax(&g_dec_keys[slot][s * M + e], merge_key(v, id));
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // before the next flush's writes
    };
    int cur = 0;  // the shard whose bests rv / ri hold
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int n = pair; n < n_tiles; n += num_pairs) {
      while (n >= tab.tile0[cur + 1]) flush(cur++);
      bool ok = mbar_wait(smem_u32(&sh->tmem_full[acc]), acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_abort_pair(sh, err);
        break;
      }
      tc_fence_after();
      const int local = (n - tab.tile0[cur]) * kTileIds + static_cast<int>(rank) * 128 +
                        quarter * 32 + lane;  // shard-local id of this lane
      const bool live = local < tab.valid[cur];
      const int32_t id = live ? tab.start[cur] + local : kNoId;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kN;
#pragma unroll
      for (int g = 0; g < kSlots; ++g) {
        uint32_t r[kG];
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
    while (cur < tab.n) flush(cur++);
    __threadfence();  // this CTA's merges before its ticket
  }

  pdl_launch_dependents();
  __syncthreads();
  if (*abort_flag) {
    const int zero = 0;
    if (warp == 0 && lane == 0) {
      if (leader) {
        // the leader's full barriers count the copies of both CTAs
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
                 "r"(kCols)
                 : "memory");
  }
  finish_launch(&sh->is_last, tab, M, slot, out, row_scale, w_scale, scaled);
}

template <bool kFp8, int kN>
cudaError_t launch_decode(const void *hidden, int64_t M, int64_t H, const void *weight,
                          int num_shards, const int64_t *starts, const int64_t *row0s,
                          const int64_t *valids, sga_stat *out, const float *row_scale,
                          float w_scale, int num_sms, uint32_t *err, cudaStream_t stream,
                          bool *launched) {
  const int tile_ids = 128 * dec_halves<kN>;
  DecShardTable tab = {};
  tab.n = num_shards;
  int64_t map_rows = 0;  // weight rows the launch reads: up to the last shard's last valid row
  for (int s = 0; s < num_shards; ++s) {
    tab.start[s] = static_cast<int32_t>(starts[s]);
    tab.row0[s] = static_cast<int32_t>(row0s[s]);
    tab.valid[s] = static_cast<int32_t>(valids[s]);
    tab.tile0[s + 1] = tab.tile0[s] + static_cast<int32_t>((valids[s] + tile_ids - 1) / tile_ids);
    if (valids[s] > 0 && row0s[s] + valids[s] > map_rows) map_rows = row0s[s] + valids[s];
  }
  const int n_tiles = tab.tile0[num_shards];
  // one CTA per SM, at most one per tile and kDecMaxParts
  int grid = n_tiles < num_sms ? n_tiles : num_sms;
  if (grid > kDecMaxParts) grid = kDecMaxParts;
  *launched = grid > 0;
  if (grid == 0) return cudaSuccess;  // every shard is padding: the caller reports it
  CUtensorMap map_w, map_h;
  if (!make_map(&map_w, weight, map_rows, H, 128, kFp8) || !make_map(&map_h, hidden, M, H, kN, kFp8))
    return cudaErrorInvalidValue;
  auto kern = lmhead_argmax_decode_kernel<kFp8, kN>;
  const int slot = 4 + (kFp8 ? 4 : 0) + (kN == 16 ? 0 : kN == 32 ? 1 : kN == 64 ? 2 : 3);
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), dec_smem_bytes<kN>, slot);
  if (e != cudaSuccess) return e;
  const int merge_slot = take_merge_slot();
  return launch_pdl(kern, grid, dec_smem_bytes<kN>, stream, map_w, map_h, static_cast<int>(M),
                    static_cast<int>(H / kBk<kFp8>), tab, merge_slot, out, row_scale, w_scale,
                    kFp8 ? 1 : 0, err);
}

template <bool kFp8, int kN>
cudaError_t launch_decode_pair(const void *hidden, int64_t M, int64_t H, const void *weight,
                               int num_shards, const int64_t *starts, const int64_t *row0s,
                               const int64_t *valids, sga_stat *out, const float *row_scale,
                               float w_scale, int num_sms, uint32_t *err, cudaStream_t stream,
                               bool *launched) {
  constexpr int kTileIds = 256;  // per CTA pair
  DecShardTable tab = {};
  tab.n = num_shards;
  int64_t map_rows = 0;
  for (int s = 0; s < num_shards; ++s) {
    tab.start[s] = static_cast<int32_t>(starts[s]);
    tab.row0[s] = static_cast<int32_t>(row0s[s]);
    tab.valid[s] = static_cast<int32_t>(valids[s]);
    tab.tile0[s + 1] = tab.tile0[s] + static_cast<int32_t>((valids[s] + kTileIds - 1) / kTileIds);
    if (valids[s] > 0 && row0s[s] + valids[s] > map_rows) map_rows = row0s[s] + valids[s];
  }
  const int n_tiles = tab.tile0[num_shards];
  // one pair per two SMs, at most one per tile
  int pairs = num_sms / 2;
  if (pairs > n_tiles) pairs = n_tiles;
  if (pairs > kDecMaxParts / 2) pairs = kDecMaxParts / 2;
  *launched = pairs > 0;
  if (pairs == 0) return cudaSuccess;  // every shard is padding: the caller reports it
  CUtensorMap map_w, map_h;
  if (!make_map(&map_w, weight, map_rows, H, 128, kFp8) ||
      !make_map(&map_h, hidden, M, H, kN / 2, kFp8))
    return cudaErrorInvalidValue;
  auto kern = lmhead_argmax_decode_pair_kernel<kFp8, kN>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), pair_smem_bytes<kN>,
                                12 + (kFp8 ? 1 : 0));
  if (e != cudaSuccess) return e;
  const int merge_slot = take_merge_slot();
  return launch_pdl(kern, 2 * pairs, pair_smem_bytes<kN>, stream, map_w, map_h,
                    static_cast<int>(M), static_cast<int>(H / kBk<kFp8>), tab, merge_slot, out,
                    row_scale, w_scale, kFp8 ? 1 : 0, err);
}

}  // namespace

cudaError_t launch_lmhead_decode(bool fp8, const void *hidden, int64_t M, int64_t H,
                                 const void *weight, int num_shards, const int64_t *starts,
                                 const int64_t *row0s, const int64_t *valids, sga_stat *out,
                                 const float *row_scale, float w_scale, int num_sms,
                                 uint32_t *err, cudaStream_t stream, bool *launched) {
#define SGA_DEC_LAUNCH(F, N)                                                                 \
  launch_decode<F, N>(hidden, M, H, weight, num_shards, starts, row0s, valids, out, row_scale, \
                      w_scale, num_sms, err, stream, launched)
  if (M <= 16) return fp8 ? SGA_DEC_LAUNCH(true, 16) : SGA_DEC_LAUNCH(false, 16);
  if (M <= 32) return fp8 ? SGA_DEC_LAUNCH(true, 32) : SGA_DEC_LAUNCH(false, 32);
  if (M <= kDecSingleMaxM) return fp8 ? SGA_DEC_LAUNCH(true, 64) : SGA_DEC_LAUNCH(false, 64);
#undef SGA_DEC_LAUNCH
  // 65 <= M <= 128: CTA pairs
  return fp8 ? launch_decode_pair<true, 128>(hidden, M, H, weight, num_shards, starts, row0s,
                                             valids, out, row_scale, w_scale, num_sms, err,
                                             stream, launched)
             : launch_decode_pair<false, 128>(hidden, M, H, weight, num_shards, starts, row0s,
                                              valids, out, row_scale, w_scale, num_sms, err,
                                              stream, launched);
}

}  // namespace sga
