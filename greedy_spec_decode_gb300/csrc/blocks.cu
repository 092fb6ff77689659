// blocks.cu -- block-granular statistics of vocab shards: per row, the
// (max, id) of every fixed global block of ids that meets a shard; one launch
// covers one shard or all the shards a GPU holds.
//
// vLLM PR #62604, Purpose item 1: each rank reduces its shard to per-block
// (max, token id) statistics, only those are all-gathered, and one kernel
// finishes the global argmax from them; the blocks keep the global boundaries
// of the unsharded kernels (8192 ids for draft positions, 1024 for the bonus
// position), also where a block straddles a shard edge.  The gathered block
// statistics feed the same reduce / verify kernels as per-shard statistics,
// with num_shards = the total number of block slots per row.
//
// Row r uses block size B = draft_block unless it is the bonus row of a
// request (row cu[i+1] + i), which uses bonus_block.  With b0 = shard_start / B,
// piece p covers global ids [max(start, (b0+p)B), min(end, (b0+p+1)B)).  Every
// row gets n_slots stats (the larger of the two block counts); slots past a
// row's own count hold (-inf, end - 1), which never wins because a real piece
// precedes it.  Output layout: out[(slot0_s + p) * rows + r] (piece-major,
// shards in order, like the shard-major gathered buffer).
//
// Design: the grid is (row group, part): a row group is one request (its K_i
// draft rows and its bonus row, read from two entries of cu_num_draft, so no
// warp ever searches for the kind of its row) or, without cu_num_draft, 16
// draft rows.  The group's real pieces (per shard, K_i x draft count + bonus
// count) are dealt round-robin to the parts x 4 warps of the group; a warp
// streams its
// piece with 16-byte loads, kUnroll in flight per lane, keeps the best
// vector in registers (the steps of the per-shard kernel), merges across
// the warp and stores one stat.  The empty slots (all but a few of a draft
// row's slots when the bonus block is the smaller one) are plain stores,
// spread over every thread of the group.  Parts are chosen so that the grid
// is one wave of resident CTAs.  A piece is at most one block (8192 ids
// = 16 KB of bf16): too short for the per-shard kernel's bulk-copy ring.
#include "common.cuh"
#include "scan.cuh"

namespace sga {
namespace {

// Tuning knobs (compile-time): warps per CTA, 16-byte loads in flight per
// lane, and the resident CTAs per SM the grid is sized for (0: the
// occupancy calculator's number).  Measured on GB300, large-verify shape
// (4096 x 202048 bf16, 3 shards, blocks 8192 / 1024, one launch per shard):
// 4 warps x 16 loads 254.5 us for the three launches (6.50 TB/s); 2 x 16 and
// 4 x 32 within 1 us of it; 8 x 8 302 us; 16 x 16 283 us; sizing the grid for
// 2 CTAs per SM instead of the occupancy limit 486 us.  Before the grid was
// sized to one wave (a partial second wave of a third of the CTAs) 8 x 8
// took 383 us.
#ifndef SGA_BLOCKS_WARPS
#define SGA_BLOCKS_WARPS 4
#endif
#ifndef SGA_BLOCKS_UNROLL
#define SGA_BLOCKS_UNROLL 16
#endif
#ifndef SGA_BLOCKS_CTAS_PER_SM
#define SGA_BLOCKS_CTAS_PER_SM 0
#endif
constexpr int kWarpsPerCta = SGA_BLOCKS_WARPS;
constexpr int kUnroll = SGA_BLOCKS_UNROLL;
constexpr int kGroupRows = 16;   // rows per group without a request layout

// The shards of one launch: shard s covers global ids [start, start + width),
// held at column col of `logits`, and owns the slots slot0 .. slot0 + slots - 1
// of every row in the gathered statistics.
struct BlockShardTable {
  int n;
  int32_t start[kMaxBlockShards];
  int32_t col[kMaxBlockShards];
  int32_t width[kMaxBlockShards];
  int32_t slot0[kMaxBlockShards];
  int32_t slots[kMaxBlockShards];
};

// Argmax (value, global id) of the non-padding ids [lo, hi) of row r, the
// shard's column 0 being global id shard_start; computed by the whole warp,
// every lane returns the result.  hi <= lo: no element, (-inf, lo).
template <bool kBf16>
__device__ __forceinline__ sga_stat piece_argmax(const char *__restrict__ row, int32_t shard_start,
                                                 int32_t lo, int32_t hi, int lane) {
  constexpr int kElt = kBf16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;
  const int n = hi > lo ? hi - lo : 0;
  const char *q = row + static_cast<int64_t>(lo - shard_start) * kElt;
  int head = static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(q) & 15u)) & 15u) / kElt);
  if (head > n) head = n;
  const int nvec = (n - head) / kVec;
  const int tail = n - head - nvec * kVec;

  float best = __int_as_float(0xff800000);  // -inf
  int32_t best_id = kNoId;
  if (lane < head) {
    const float x = load_elem<kBf16>(q, lane);
    if (scan_better(x, best)) {
      best = x;
      best_id = lo + lane;
    }
  }
  const uint4 *vp = reinterpret_cast<const uint4 *>(q + head * kElt);
  float vbest = __int_as_float(0xff800000);
  int vbest_idx = -1;
  uint4 vraw = make_uint4(0u, 0u, 0u, 0u);
  int v = lane;
  for (; v + (kUnroll - 1) * 32 < nvec; v += kUnroll * 32) {
    uint4 a[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) a[u] = ld_stream_v4(vp + v + u * 32);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float m = vec_max<kBf16>(a[u]);
      if (scan_better(m, vbest)) {
        vbest = m;
        vbest_idx = v + u * 32;
        vraw = a[u];
      }
    }
  }
#pragma unroll 4
  for (; v < nvec; v += 32) {
    const uint4 a = ld_stream_v4(vp + v);
    const float m = vec_max<kBf16>(a);
    if (scan_better(m, vbest)) {
      vbest = m;
      vbest_idx = v;
      vraw = a;
    }
  }
  if (vbest_idx >= 0) scan_vec<kBf16>(vraw, lo + head + vbest_idx * kVec, best, best_id);
  if (lane < tail) {
    const int j = head + nvec * kVec + lane;
    const float x = load_elem<kBf16>(q, j);
    if (scan_better(x, best)) {
      best = x;
      best_id = lo + j;
    }
  }
  warp_argmax(best, best_id);
  sga_stat st;
  st.v = best;  // -inf when nothing beat -inf
  st.id = best_id == kNoId ? lo : best_id;
  return st;
}

// grid.x = groups x parts; CTA b: group b / parts, part b % parts.  The
// shards of the table are processed in one launch: a group's real pieces are
// numbered shard by shard (then row, then piece), so consecutive items still
// stream consecutive memory.  Ids and block sizes are below 2^24 + 1 and a
// group's pieces below 2^31, so the per-piece arithmetic is 32-bit.
template <bool kBf16>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    block_argmax_kernel(const char *__restrict__ logits, int64_t ld_bytes, int64_t rows,
                        const __grid_constant__ BlockShardTable tab, int32_t org_vocab,
                        int32_t draft_block, int32_t bonus_block, int parts,
                        const int32_t *__restrict__ cu, sga_stat *__restrict__ out,
                        uint32_t *err) {
  constexpr int kElt = kBf16 ? 2 : 4;
  __shared__ int32_t cnt_d[kMaxBlockShards], cnt_b[kMaxBlockShards];
  __shared__ int32_t item0[kMaxBlockShards + 1], empty0[kMaxBlockShards + 1];
  pdl_wait();
  const int g = static_cast<int>(blockIdx.x / parts);
  const int part = static_cast<int>(blockIdx.x % parts);
  const int lane = threadIdx.x & 31;
  int64_t first;  // first row of the group
  int n_draft;    // draft rows first .. first + n_draft - 1
  int n_bonus;    // 1: row first + n_draft is the group's bonus row
  if (cu != nullptr) {
    const int32_t c0 = cu[g], c1 = cu[g + 1];
    first = static_cast<int64_t>(c0) + g;
    n_draft = c1 - c0;
    n_bonus = 1;
    if (c1 < c0 || c0 < 0 || first + n_draft >= rows) {
      if (part == 0 && threadIdx.x == 0) atomicOr(err, SGA_DEVERR_LAYOUT);
      return;  // CTA-uniform: before any barrier
    }
  } else {
    first = static_cast<int64_t>(g) * kGroupRows;
    n_draft = static_cast<int>(min(static_cast<int64_t>(kGroupRows), rows - first));
    n_bonus = 0;
  }
  // per shard: block counts, and where its pieces and empty slots start in
  // the group's numbering
  if (threadIdx.x == 0) {
    int32_t items = 0, empties = 0;
    for (int s = 0; s < tab.n; ++s) {
      const int32_t st = tab.start[s], en = st + tab.width[s];
      const int32_t cd = (en - 1) / draft_block - st / draft_block + 1;
      const int32_t cb = (en - 1) / bonus_block - st / bonus_block + 1;
      cnt_d[s] = cd;
      cnt_b[s] = cb;
      item0[s] = items;
      empty0[s] = empties;
      items += n_draft * cd + n_bonus * cb;
      empties += n_draft * (tab.slots[s] - cd) + n_bonus * (tab.slots[s] - cb);
    }
    item0[tab.n] = items;
    empty0[tab.n] = empties;
  }
  __syncthreads();

  // real pieces, dealt round-robin to the group's warps
  const int n_items = item0[tab.n];
  const int workers = parts * kWarpsPerCta;
  int s = 0;  // each warp's items increase, so its shard index only advances
  for (int32_t t = part * kWarpsPerCta + (threadIdx.x >> 5); t < n_items; t += workers) {
    while (t >= item0[s + 1]) ++s;
    const int32_t u = t - item0[s];
    const int32_t sd = n_draft * cnt_d[s];
    int32_t rr, p, B;
    if (u < sd) {
      rr = u / cnt_d[s];
      p = u - rr * cnt_d[s];
      B = draft_block;
    } else {
      rr = n_draft;
      p = u - sd;
      B = bonus_block;
    }
    const int32_t st = tab.start[s], en = st + tab.width[s];
    const int32_t b = st / B + p;
    const int32_t lo = max(st, b * B);
    const int32_t hi = min(min(en, b * B + B), org_vocab);
    const int64_t r = first + rr;
    const sga_stat stat = piece_argmax<kBf16>(
        logits + r * ld_bytes + static_cast<int64_t>(tab.col[s]) * kElt, st, lo, hi, lane);
    if (lane == 0) out[static_cast<int64_t>(tab.slot0[s] + p) * rows + r] = stat;
  }
  pdl_launch_dependents();

  // empty slots: (-inf, the shard's last id), consecutive threads on
  // consecutive rows
  const int n_empty = empty0[tab.n];
  s = 0;
  for (int32_t t = part * static_cast<int32_t>(blockDim.x) + threadIdx.x; t < n_empty;
       t += parts * static_cast<int32_t>(blockDim.x)) {
    while (t >= empty0[s + 1]) ++s;
    const int32_t u = t - empty0[s];
    const int32_t ed = n_draft * (tab.slots[s] - cnt_d[s]);
    sga_stat empty;
    empty.v = __int_as_float(0xff800000);
    empty.id = tab.start[s] + tab.width[s] - 1;
    int64_t slot, r;
    if (u < ed) {
      slot = cnt_d[s] + u / n_draft;
      r = first + u % n_draft;
    } else {
      slot = cnt_b[s] + (u - ed);
      r = first + n_draft;
    }
    out[(tab.slot0[s] + slot) * rows + r] = empty;
  }
}

// Resident CTAs per SM of one instantiation, looked up once per device.
template <bool kBf16>
int resident_per_sm() {
  if (SGA_BLOCKS_CTAS_PER_SM > 0) return SGA_BLOCKS_CTAS_PER_SM;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, block_argmax_kernel<kBf16>,
                                                      kWarpsPerCta * 32, 0) != cudaSuccess ||
        n < 1)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace

int64_t block_count(int64_t shard_start, int64_t shard_width, int64_t block) {
  return (shard_start + shard_width - 1) / block - shard_start / block + 1;
}

int64_t block_slots(int64_t shard_start, int64_t shard_width, int64_t draft_block,
                    int64_t bonus_block) {
  const int64_t a = block_count(shard_start, shard_width, draft_block);
  const int64_t b = block_count(shard_start, shard_width, bonus_block);
  return a > b ? a : b;
}

cudaError_t launch_block_argmax_table(const void *logits, int dtype, int64_t rows, int64_t ld,
                                      int num_shards, const int64_t *starts, const int64_t *cols,
                                      const int64_t *widths, int64_t org_vocab,
                                      int64_t draft_block, int64_t bonus_block, int num_reqs,
                                      const int32_t *cu_num_draft, sga_stat *out, int num_sms,
                                      uint32_t *err, cudaStream_t stream) {
  const bool bf16 = dtype == SGA_BF16;
  BlockShardTable tab = {};
  tab.n = num_shards;
  int32_t slot = 0;
  for (int s = 0; s < num_shards; ++s) {
    tab.start[s] = static_cast<int32_t>(starts[s]);
    tab.col[s] = static_cast<int32_t>(cols[s]);
    tab.width[s] = static_cast<int32_t>(widths[s]);
    tab.slot0[s] = slot;
    tab.slots[s] = static_cast<int32_t>(block_slots(starts[s], widths[s], draft_block, bonus_block));
    slot += tab.slots[s];
  }
  const int64_t groups = cu_num_draft != nullptr ? num_reqs : (rows + kGroupRows - 1) / kGroupRows;
  // one wave: as many parts per group as the resident CTAs allow (the work of
  // a group splits evenly over its parts, so a partial second wave would
  // only add a tail), at least 1, at most 64
  const int64_t resident =
      static_cast<int64_t>(num_sms) * (bf16 ? resident_per_sm<true>() : resident_per_sm<false>());
  int64_t parts = resident / groups;
  if (parts < 1) parts = 1;
  if (parts > 64) parts = 64;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(groups * parts));
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int elt = bf16 ? 2 : 4;
  const char *base = static_cast<const char *>(logits);
  auto kern = bf16 ? block_argmax_kernel<true> : block_argmax_kernel<false>;
  return cudaLaunchKernelEx(
      &cfg, kern, base, ld * elt, rows, tab,
      static_cast<int32_t>(org_vocab < SGA_MAX_VOCAB ? org_vocab : SGA_MAX_VOCAB),
      static_cast<int32_t>(draft_block), static_cast<int32_t>(bonus_block),
      static_cast<int>(parts), cu_num_draft, out, err);
}

cudaError_t launch_block_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                                int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                                int64_t draft_block, int64_t bonus_block, int num_reqs,
                                const int32_t *cu_num_draft, sga_stat *out, int num_sms,
                                uint32_t *err, cudaStream_t stream) {
  const int64_t col = 0;
  return launch_block_argmax_table(logits, dtype, rows, ld, 1, &shard_start, &col, &shard_width,
                                   org_vocab, draft_block, bonus_block, num_reqs, cu_num_draft,
                                   out, num_sms, err, stream);
}

}  // namespace sga
