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
// Design.  The work items of a launch are numbered flat: request by request
// (its K_i draft rows and its bonus row), inside a request shard by shard,
// then row, then item, so consecutive numbers are consecutive memory.  An
// item is one piece, or up to four consecutive short pieces of one row and
// shard (up to four of at most 2 KB each, such as the 1024-id bonus blocks of
// bf16 logits, or two of at most 4 KB), which a warp scans at once with a
// group of 8 or 16 lanes per piece, so that every lane keeps as many loads in
// flight as on a long piece.  With
// D = the draft-row items and Bn = the bonus-row items of all the shards of
// the launch, request i's items start at number cu[i] * D + i * Bn, a closed
// form: a warp finds the request of its first item with one binary search
// over cu_num_draft and then walks forward.  Every CTA of the grid (one wave
// of resident CTAs) takes an equal contiguous range of numbers, so the load is
// balanced whatever the number of requests and their K_i; inside that range
// its warps take the items one at a time from a counter in shared memory (a
// CTA's warps read neighbouring items), so that warps the memory system
// serves faster take more.  A
// warp (or lane group) scans a piece as the per-shard kernel scans a row:
// 16-byte vectors with kUnroll streaming loads in flight per lane, the best
// vector kept in registers and searched once; the element head (to the
// first 16-byte boundary) and tail are loaded before the vectors so that
// their latency overlaps; then a merge across the lanes and one stat.  The
// empty slots (all but a few of a draft row's slots when the bonus block is
// the smaller one) are plain stores, one thread per row.  Without
// cu_num_draft every row is a request of one draft row and no bonus row.
#include "common.cuh"
#include "scan.cuh"

namespace sga {
namespace {

// Tuning knobs (compile-time): warps per CTA, 16-byte loads in flight per
// lane, the CTAs per SM the registers are budgeted for (the second launch
// bound: without it the compiler keeps the kernel near 48 registers, too few
// for the loads in flight), the resident CTAs per SM the grid is sized for
// (0: the occupancy calculator's number), and how a CTA's range is split
// (1: round-robin over its warps, 0: a contiguous sub-range per warp).
// Measured on GB300 with CUDA events around each launch (launches kept
// apart, one process), large-verify logits (202048 bf16 ids, 3 shards in one
// launch, blocks 8192 / 1024), 256 requests, for K_i = 15 (4096 rows) /
// K_i uniform in 0..15 (2271 rows) / 64 requests of K_i = 15 and 192 of
// K_i = 0 (1216 rows):
//   4 warps x 16 loads, 5 CTAs per SM, round-robin, short pieces four at a
//     time: 239.7 / 147.5 / 84.0 us;
//   the same with one piece per warp: 244.7 / 170.0 / 119.8 us;
//   8 loads, 8 CTAs per SM: 241.6 / 141.3 / 84.0 us;
//   on a slower box, registers budgeted for 5 / 6 / 7 / 8 CTAs per SM (96 /
//     80 / 72 / 64 registers): 243.7 / 247.8 / 249.9 / 243.7 us at
//     K_i = 15, 147.5 / 147.5 / 147.5 / 143.5 us for the mixed K_i, 85.9 /
//     86.0 / 88.1 / 86.0 us skewed; 8 warps at 3 per SM 243.7 / 145.4 /
//     86.1 us.  8 CTAs per SM with 16 loads is chosen;
//   one piece per warp, K_i = 15 only: a contiguous sub-range per warp
//     268.3 us; 8 CTAs per SM with 8 loads 258-271 us; 10 per SM 268-278 us;
//     12 per SM with 4 loads 284.7 us; two, four or eight waves of smaller
//     CTAs 274.4, 262.1, 256.0 us; no programmatic dependent launch: no
//     change.
// The earlier kernel (whole CTAs per request, as many for a request of 0
// drafts as for one of 15, one piece per warp) took 250.2 / 189.2 / 162.4
// us.  Tried and dropped since (same process, median of 30 launches; K_i =
// 15 / K_i uniform in 1..15): an L2 prefetch of each warp's next item
// (255.0 -> 276.5 / 149.5 -> 171.6 us); the per-shard kernel's bulk-copy
// ring with a CTA per (row, shard) walking the pieces in order (whole
// vectors from the ring, a 128-thread reduction and barrier per piece):
// 483-500 / 331-339 us against 254-258 / 150-152 us -- issue-bound (ncu: 97 M
// warp instructions for 414 MB), because a 2 KB bonus piece gives each of
// the 128 threads one vector and still costs a full CTA reduction; CTA
// ranges balanced by bytes (rows cut into equal parts, found by a 32-ary
// search over cu_num_draft) instead of by items: 274 / 166 us against 258 /
// 152 us; the empty slots written by the warp of each row's first item,
// during the stream, instead of after it: 266 / 154 us.
// Per-warp timestamps of the round-robin kernel showed warps with equal work
// finishing up to 30 us apart inside one SM (mixed K_i: first warp 104 us,
// median 130 us, last 146 us): the memory system serves warps unevenly.
// Items taken one at a time from a shared counter per CTA (the current
// kernel): 8 warps x 4 CTAs per SM 248.1 / 143.4 us (0.988 / 0.960 of copy);
// 4 x 8 per SM 252.2 / 147.5; 16 x 2 per SM 251.5 / 152.6; one CTA of 32
// warps per SM 270 / 174; 8 x 4 with 8 loads in flight 250.1 / 145.4 us.
#ifndef SGA_BLOCKS_DYNAMIC
// 1: the warps of a CTA take its items one at a time from a shared-memory
// counter (8-warp CTAs, 4 per SM).  0: 4-warp CTAs, items dealt round-robin.
#define SGA_BLOCKS_DYNAMIC 1
#endif
#ifndef SGA_BLOCKS_WARPS
#define SGA_BLOCKS_WARPS (SGA_BLOCKS_DYNAMIC ? 8 : 4)
#endif
#ifndef SGA_BLOCKS_UNROLL
#define SGA_BLOCKS_UNROLL 16
#endif
#ifndef SGA_BLOCKS_MIN_CTAS
#define SGA_BLOCKS_MIN_CTAS (SGA_BLOCKS_DYNAMIC ? 4 : 8)
#endif
#ifndef SGA_BLOCKS_CTAS_PER_SM
#define SGA_BLOCKS_CTAS_PER_SM 0
#endif
#ifndef SGA_BLOCKS_INTERLEAVE
#define SGA_BLOCKS_INTERLEAVE 1
#endif
constexpr int kWarpsPerCta = SGA_BLOCKS_WARPS;
constexpr int kUnroll = SGA_BLOCKS_UNROLL;
// Short pieces are taken several at a time, one per group of lanes, so that
// a lane still has up to kUnroll loads in flight: pieces of at most
// kShortPieceBytes four at a time (groups of 8 lanes), of at most twice that
// two at a time (groups of 16 lanes).  A 1024-id bonus block is 2 KB of bf16
// (4 vectors per lane of a whole warp, 16 per lane of a group of 8) or 4 KB
// of fp32.
#ifndef SGA_BLOCKS_SHORT_PIECE_BYTES
#define SGA_BLOCKS_SHORT_PIECE_BYTES 2048
#endif
constexpr int64_t kShortPieceBytes = SGA_BLOCKS_SHORT_PIECE_BYTES;

// Pieces per work item for a block size (host side).
inline int32_t group_for(int64_t block_ids, int elt) {
  const int64_t bytes = block_ids * elt;
  return bytes <= kShortPieceBytes ? 4 : (bytes <= 2 * kShortPieceBytes ? 2 : 1);
}

// The shards of one launch: shard s covers global ids [start, start + width),
// held at column col of `logits`, owns the slots slot0 .. slot0 + slots - 1 of
// every row in the gathered statistics, and meets cnt_d draft blocks and
// cnt_b bonus blocks.  A work item is up to group_d consecutive pieces of one
// draft row (group_b of one bonus row) in one shard: items_d = ceil(cnt_d /
// group_d) and items_b = ceil(cnt_b / group_b) items per row, and pre_d /
// pre_b are their prefix sums over the shards (pre_d[n] = D, pre_b[n] = Bn).
struct BlockShardTable {
  int n;
  int32_t start[kMaxBlockShards];
  int32_t col[kMaxBlockShards];
  int32_t width[kMaxBlockShards];
  int32_t slot0[kMaxBlockShards];
  int32_t slots[kMaxBlockShards];
  int32_t cnt_d[kMaxBlockShards];
  int32_t cnt_b[kMaxBlockShards];
  int32_t items_d[kMaxBlockShards];
  int32_t items_b[kMaxBlockShards];
  int32_t pre_d[kMaxBlockShards + 1];
  int32_t pre_b[kMaxBlockShards + 1];
};

// One piece: the non-padding ids [lo, lo + n) of one row inside one block
// and one shard, at address q in the logits, and where its stat goes.
struct Piece {
  const char *q;
  int32_t lo;
  int32_t n;
  int64_t out_idx;
};

// How a piece splits into an element head up to the first 16-byte boundary,
// whole 16-byte vectors and an element tail.
template <bool kBf16>
struct Split {
  int head, nvec, tail;
  __device__ __forceinline__ explicit Split(const Piece &pc) {
    constexpr int kElt = kBf16 ? 2 : 4;
    constexpr int kVec = 16 / kElt;
    head = static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(pc.q) & 15u)) & 15u) / kElt);
    if (head > pc.n) head = pc.n;
    nvec = (pc.n - head) / kVec;
    tail = pc.n - head - nvec * kVec;
  }
};

// One request of the launch: its first row, its k draft rows, whether row
// first + k is its bonus row, the number of its first piece and its piece
// count, and whether its rows lie inside [0, rows).  Without cu_num_draft,
// request g is row g alone, a draft row.
struct Request {
  int64_t first;
  int64_t item0;
  int32_t k;
  int32_t bonus;
  int32_t n_items;
  bool valid;
};

__device__ __forceinline__ int64_t clamp_rows(int32_t c, int64_t rows) {
  return c < 0 ? 0 : (c > rows ? rows : static_cast<int64_t>(c));
}

// Number of the first piece of request g (cu_num_draft entries clamped to
// [0, rows], so that a broken layout still gives numbers in range).
__device__ __forceinline__ int64_t item0_of(int64_t g, const int32_t *__restrict__ cu,
                                            int64_t rows, int32_t d, int32_t bn) {
  if (cu == nullptr) return g * d;
  return clamp_rows(__ldg(cu + g), rows) * d + g * bn;
}

__device__ __forceinline__ Request request_of(int64_t g, const int32_t *__restrict__ cu,
                                              int64_t rows, int32_t d, int32_t bn) {
  Request q;
  if (cu == nullptr) {
    q.first = g;
    q.k = 1;
    q.bonus = 0;
    q.item0 = g * d;
    q.n_items = d;
    q.valid = true;
    return q;
  }
  const int32_t c0 = __ldg(cu + g), c1 = __ldg(cu + g + 1);
  q.first = static_cast<int64_t>(c0) + g;
  q.k = c1 - c0;
  q.bonus = 1;
  q.valid = c0 >= 0 && c1 >= c0 && static_cast<int64_t>(c1) + g < rows;
  q.item0 = clamp_rows(c0, rows) * d + g * bn;
  q.n_items = q.valid ? q.k * d + bn : 0;
  return q;
}

// The request holding piece number t: the largest g in [0, n) whose first
// piece is at or before t.
__device__ __forceinline__ int64_t request_at(int64_t t, int64_t n, const int32_t *__restrict__ cu,
                                              int64_t rows, int32_t d, int32_t bn) {
  if (cu == nullptr) return t / d;
  int64_t lo = 0, hi = n - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (item0_of(mid, cu, rows, d, bn) <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Work item u (0 <= u < q.n_items) of request q: row r, shard s, block size
// B and pieces p0 .. p0 + np - 1.  `s` is the caller's shard cursor inside
// the request: its items only increase, so it only advances.
struct Item {
  int64_t r;
  int s;
  int32_t B;
  int32_t p0;
  int32_t np;
  int32_t g;  // pieces per item of the item's row kind (1, 2 or 4)
};

__device__ __forceinline__ Item item_of(int32_t u, int &s, const Request &q,
                                        const BlockShardTable &tab, int32_t draft_block,
                                        int32_t bonus_block, int32_t group_d, int32_t group_b) {
  while (u >= q.k * tab.pre_d[s + 1] + q.bonus * tab.pre_b[s + 1]) ++s;
  const int32_t v = u - (q.k * tab.pre_d[s] + q.bonus * tab.pre_b[s]);
  const int32_t sd = q.k * tab.items_d[s];
  int32_t rr, gi, g, cnt;
  Item it;
  if (v < sd) {
    rr = v / tab.items_d[s];
    gi = v - rr * tab.items_d[s];
    it.B = draft_block;
    g = group_d;
    cnt = tab.cnt_d[s];
  } else {
    rr = q.k;
    gi = v - sd;
    it.B = bonus_block;
    g = group_b;
    cnt = tab.cnt_b[s];
  }
  it.r = q.first + rr;
  it.s = s;
  it.p0 = gi * g;
  it.np = min(g, cnt - it.p0);
  it.g = g;
  return it;
}

// Piece p of an item's row and shard: ids [max(start, b B), min(end, (b+1) B,
// org_vocab)) with b = start / B + p.  active = false gives an empty piece.
template <bool kBf16>
__device__ __forceinline__ Piece piece_at(const Item &it, int32_t p, bool active,
                                          const BlockShardTable &tab, int32_t org_vocab,
                                          const char *logits, int64_t ld_bytes, int64_t rows) {
  constexpr int kElt = kBf16 ? 2 : 4;
  const int32_t st = tab.start[it.s], en = st + tab.width[it.s];
  const int32_t b = st / it.B + p;
  const int32_t lo = max(st, b * it.B);
  const int32_t hi = min(min(en, b * it.B + it.B), org_vocab);
  Piece pc;
  pc.lo = lo;
  pc.n = active && hi > lo ? hi - lo : 0;
  pc.q = logits + it.r * ld_bytes + static_cast<int64_t>(tab.col[it.s] + (lo - st)) * kElt;
  pc.out_idx = static_cast<int64_t>(tab.slot0[it.s] + p) * rows + it.r;
  return pc;
}

// (value, id) argmax over groups of kW lanes (kW a power of two <= 32):
// every lane ends with its group's result.
template <int kW>
__device__ __forceinline__ void group_argmax(float &v, int32_t &id) {
#pragma unroll
  for (int off = kW / 2; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int32_t oi = __shfl_xor_sync(0xffffffffu, id, off);
    if (pair_beats(ov, oi, v, id)) {
      v = ov;
      id = oi;
    }
  }
}

// Argmax (value, global id) of one piece, computed by a group of kW lanes of
// the warp (sl = the lane's index in its group, kW >= 8 so that a group
// covers the element head and tail); every lane of the group returns the
// result.  No element: (-inf, lo).  Per lane the scan order is ascending ids
// (head element, vectors, tail element), then the merge across the group
// takes the full (value, id) order.  All 32 lanes of the warp call it.
template <bool kBf16, int kW>
__device__ __forceinline__ sga_stat piece_argmax(const Piece &pc, int sl) {
  constexpr int kElt = kBf16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;
  static_assert(kW >= 8 && kW <= 32 && (kW & (kW - 1)) == 0, "group of 8, 16 or 32 lanes");
  const Split<kBf16> sp(pc);
  // the lane's head and tail elements, loaded first so that their latency
  // overlaps the vector loads
  float head_x = __int_as_float(0xff800000), tail_x = __int_as_float(0xff800000);
  if (sl < sp.head) head_x = load_elem<kBf16>(pc.q, sl);
  if (sl < sp.tail) tail_x = load_elem<kBf16>(pc.q, sp.head + sp.nvec * kVec + sl);

  const uint4 *vp = reinterpret_cast<const uint4 *>(pc.q + sp.head * kElt);
  float vbest = __int_as_float(0xff800000);
  int vbest_idx = -1;
  uint4 vraw = make_uint4(0u, 0u, 0u, 0u);
  int v = sl;
  for (; v + (kUnroll - 1) * kW < sp.nvec; v += kUnroll * kW) {
    uint4 a[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) a[u] = ld_stream_v4(vp + v + u * kW);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float m = vec_max<kBf16>(a[u]);
      if (scan_better(m, vbest)) {
        vbest = m;
        vbest_idx = v + u * kW;
        vraw = a[u];
      }
    }
  }
#pragma unroll 4
  for (; v < sp.nvec; v += kW) {
    const uint4 a = ld_stream_v4(vp + v);
    const float m = vec_max<kBf16>(a);
    if (scan_better(m, vbest)) {
      vbest = m;
      vbest_idx = v;
      vraw = a;
    }
  }

  float best = __int_as_float(0xff800000);
  int32_t best_id = kNoId;
  if (sl < sp.head && scan_better(head_x, best)) {
    best = head_x;
    best_id = pc.lo + sl;
  }
  if (vbest_idx >= 0) scan_vec<kBf16>(vraw, pc.lo + sp.head + vbest_idx * kVec, best, best_id);
  if (sl < sp.tail && scan_better(tail_x, best)) {
    best = tail_x;
    best_id = pc.lo + sp.head + sp.nvec * kVec + sl;
  }
  group_argmax<kW>(best, best_id);
  sga_stat st;
  st.v = best;  // -inf when nothing beat -inf
  st.id = best_id == kNoId ? pc.lo : best_id;
  return st;
}

// Up to 32 / kW short pieces of one item, one per group of kW lanes; every
// lane of the warp takes part (the groups past the item's pieces scan an
// empty piece and store nothing).
template <bool kBf16, int kW>
__device__ __forceinline__ void scan_group(const Item &it, int lane, const BlockShardTable &tab,
                                           int32_t org_vocab, const char *logits,
                                           int64_t ld_bytes, int64_t rows,
                                           sga_stat *__restrict__ out) {
  const int sub = lane / kW, sl = lane % kW;
  const bool act = sub < it.np;
  const Piece pc =
      piece_at<kBf16>(it, it.p0 + (act ? sub : 0), act, tab, org_vocab, logits, ld_bytes, rows);
  const sga_stat stat = piece_argmax<kBf16, kW>(pc, sl);
  if (act && sl == 0) out[pc.out_idx] = stat;
}

// grid.x = C = resident CTAs (at most); of the T work items, CTA c takes
// those numbered [T c / C, T (c + 1) / C), its warp j every kWarpsPerCta-th
// of them from the j-th on (or, without interleaving, warp w of W takes
// [T w / W, T (w + 1) / W)).  num_groups = num_reqs with cu_num_draft, else
// rows.  Ids and block sizes are below 2^24 + 1 and rows x slots below 2^28,
// so the arithmetic inside a request is 32-bit.
template <bool kBf16>
__global__ void __launch_bounds__(kWarpsPerCta * 32, SGA_BLOCKS_MIN_CTAS)
    block_argmax_kernel(const char *__restrict__ logits, int64_t ld_bytes, int64_t rows,
                        const __grid_constant__ BlockShardTable tab, int32_t org_vocab,
                        int32_t draft_block, int32_t bonus_block, int32_t group_d,
                        int32_t group_b, int64_t num_groups,
                        const int32_t *__restrict__ cu, sga_stat *__restrict__ out,
                        uint32_t *err) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int32_t d = tab.pre_d[tab.n], bn = cu != nullptr ? tab.pre_b[tab.n] : 0;
  const int64_t n_items =
      cu != nullptr ? clamp_rows(__ldg(cu + num_groups), rows) * d + num_groups * bn
                    : rows * d;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
  const int warp = static_cast<int>(threadIdx.x >> 5);
  // this warp's numbers: t0, t0 + step, ... below t1
  int64_t t0, t1, step;
  if (SGA_BLOCKS_INTERLEAVE) {
    // the CTA's contiguous range, dealt round-robin to its warps
    t0 = n_items * blockIdx.x / gridDim.x + warp;
    t1 = n_items * (blockIdx.x + 1) / gridDim.x;
    step = kWarpsPerCta;
  } else {
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp;
    t0 = n_items * w / n_warps;
    t1 = n_items * (w + 1) / n_warps;
    step = 1;
  }

#if SGA_BLOCKS_DYNAMIC
  // the CTA's contiguous range [t0 - warp, t1); each warp takes the next
  // number from a shared counter, so the warps of an SM that the memory
  // system serves faster take more items and all of them finish together
  __shared__ unsigned long long next_item;
  if (threadIdx.x == 0) next_item = static_cast<unsigned long long>(t0 - warp);
  __syncthreads();
  unsigned long long grabbed = 0;
  if (lane == 0) grabbed = atomicAdd(&next_item, 1ull);
  int64_t t = static_cast<int64_t>(__shfl_sync(0xffffffffu, grabbed, 0));
  if (t < t1) {
    int64_t g = request_at(t, num_groups, cu, rows, d, bn);
    Request q = request_of(g, cu, rows, d, bn);
    int64_t next0 = g + 1 < num_groups ? item0_of(g + 1, cu, rows, d, bn) : INT64_MAX;
    int s = 0;
    while (t < t1) {
      // the next number, taken now so that the atomic's latency overlaps
      // this item (the numbers a warp takes only increase)
      if (lane == 0) grabbed = atomicAdd(&next_item, 1ull);
      while (t >= next0) {
        ++g;
        q = request_of(g, cu, rows, d, bn);
        next0 = g + 1 < num_groups ? item0_of(g + 1, cu, rows, d, bn) : INT64_MAX;
        s = 0;
      }
      const int64_t u = t - q.item0;
      if (u >= 0 && u < q.n_items) {  // else a request outside the rows or a hole
        const Item it = item_of(static_cast<int32_t>(u), s, q, tab, draft_block, bonus_block,
                                group_d, group_b);
        if (it.g == 1) {
          const Piece pc =
              piece_at<kBf16>(it, it.p0, true, tab, org_vocab, logits, ld_bytes, rows);
          const sga_stat stat = piece_argmax<kBf16, 32>(pc, lane);
          if (lane == 0) out[pc.out_idx] = stat;
        } else if (it.g == 2) {
          scan_group<kBf16, 16>(it, lane, tab, org_vocab, logits, ld_bytes, rows, out);
        } else {
          scan_group<kBf16, 8>(it, lane, tab, org_vocab, logits, ld_bytes, rows, out);
        }
      }
      t = static_cast<int64_t>(__shfl_sync(0xffffffffu, grabbed, 0));
    }
  }
  (void)step;
#else
  if (t0 < t1) {
    int64_t g = request_at(t0, num_groups, cu, rows, d, bn);
    Request q = request_of(g, cu, rows, d, bn);
    int64_t next0 = g + 1 < num_groups ? item0_of(g + 1, cu, rows, d, bn) : INT64_MAX;
    int s = 0;
    for (int64_t t = t0; t < t1;) {
      while (t >= next0) {
        ++g;
        q = request_of(g, cu, rows, d, bn);
        next0 = g + 1 < num_groups ? item0_of(g + 1, cu, rows, d, bn) : INT64_MAX;
        s = 0;
      }
      const int64_t u = t - q.item0;
      if (u < 0 || u >= q.n_items) {
        // a request outside the rows (flagged below) or a hole in a broken
        // layout: nothing to scan up to the next request (this warp's first
        // number at or after it)
        if (next0 >= t1) break;
        t += (next0 - t + step - 1) / step * step;
        continue;
      }
      const Item it = item_of(static_cast<int32_t>(u), s, q, tab, draft_block, bonus_block,
                              group_d, group_b);
      if (it.g == 1) {
        // one piece, the whole warp
        const Piece pc = piece_at<kBf16>(it, it.p0, true, tab, org_vocab, logits, ld_bytes, rows);
        const sga_stat stat = piece_argmax<kBf16, 32>(pc, lane);
        if (lane == 0) out[pc.out_idx] = stat;
      } else if (it.g == 2) {
        scan_group<kBf16, 16>(it, lane, tab, org_vocab, logits, ld_bytes, rows, out);
      } else {
        scan_group<kBf16, 8>(it, lane, tab, org_vocab, logits, ld_bytes, rows, out);
      }
      t += step;
    }
  }
#endif
  pdl_launch_dependents();

  const int64_t n_threads = n_warps * 32;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (cu != nullptr) {
    // every request whose rows leave [0, rows) is flagged, however the walk
    // above went
    for (int64_t g = tid; g < num_groups; g += n_threads)
      if (!request_of(g, cu, rows, d, bn).valid) atomicOr(err, SGA_DEVERR_LAYOUT);
  }
  // empty slots: (-inf, the shard's last id), one thread per row,
  // consecutive threads on consecutive rows
  for (int64_t r = tid; r < rows; r += n_threads) {
    bool bonus_row = false;
    if (cu != nullptr) {
      int64_t lo = 0, hi = num_groups - 1;  // the request whose rows start at or before r
      while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (clamp_rows(__ldg(cu + mid), rows) + mid <= r) lo = mid;
        else hi = mid - 1;
      }
      const Request q = request_of(lo, cu, rows, d, bn);
      if (!q.valid || r < q.first || r > q.first + q.k) continue;  // no request holds row r
      bonus_row = r == q.first + q.k;
    }
    for (int sh = 0; sh < tab.n; ++sh) {
      sga_stat empty;
      empty.v = __int_as_float(0xff800000);
      empty.id = tab.start[sh] + tab.width[sh] - 1;
      for (int p = bonus_row ? tab.cnt_b[sh] : tab.cnt_d[sh]; p < tab.slots[sh]; ++p)
        out[static_cast<int64_t>(tab.slot0[sh] + p) * rows + r] = empty;
    }
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
  const int elt = bf16 ? 2 : 4;
  // short pieces (the bonus rows' 1024-id blocks) go several at a time
  const int32_t group_d = group_for(draft_block, elt);
  const int32_t group_b = group_for(bonus_block, elt);
  BlockShardTable tab = {};
  tab.n = num_shards;
  int32_t slot = 0;
  for (int s = 0; s < num_shards; ++s) {
    tab.start[s] = static_cast<int32_t>(starts[s]);
    tab.col[s] = static_cast<int32_t>(cols[s]);
    tab.width[s] = static_cast<int32_t>(widths[s]);
    tab.slot0[s] = slot;
    tab.slots[s] = static_cast<int32_t>(block_slots(starts[s], widths[s], draft_block, bonus_block));
    tab.cnt_d[s] = static_cast<int32_t>(block_count(starts[s], widths[s], draft_block));
    tab.cnt_b[s] = static_cast<int32_t>(block_count(starts[s], widths[s], bonus_block));
    tab.items_d[s] = (tab.cnt_d[s] + group_d - 1) / group_d;
    tab.items_b[s] = (tab.cnt_b[s] + group_b - 1) / group_b;
    tab.pre_d[s + 1] = tab.pre_d[s] + tab.items_d[s];
    tab.pre_b[s + 1] = tab.pre_b[s] + tab.items_b[s];
    slot += tab.slots[s];
  }
  const bool by_request = cu_num_draft != nullptr;
  const int64_t groups = by_request ? num_reqs : rows;
  // work items of a well-formed layout (rows = cu[num_reqs] + num_reqs); the
  // kernel takes the count from cu_num_draft itself, this only sizes the grid
  const int64_t pieces = by_request ? (rows - num_reqs) * tab.pre_d[num_shards] +
                                          static_cast<int64_t>(num_reqs) * tab.pre_b[num_shards]
                                    : rows * tab.pre_d[num_shards];
  // one wave of resident CTAs, fewer when there are fewer pieces than warps
  const int per_sm = bf16 ? resident_per_sm<true>() : resident_per_sm<false>();
  int64_t ctas = static_cast<int64_t>(num_sms) * per_sm;
  const int64_t need = (pieces + kWarpsPerCta - 1) / kWarpsPerCta;
  if (need < ctas) ctas = need;
  if (ctas < 1) ctas = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const char *base = static_cast<const char *>(logits);
  auto kern = bf16 ? block_argmax_kernel<true> : block_argmax_kernel<false>;
  return cudaLaunchKernelEx(
      &cfg, kern, base, ld * elt, rows, tab,
      static_cast<int32_t>(org_vocab < SGA_MAX_VOCAB ? org_vocab : SGA_MAX_VOCAB),
      static_cast<int32_t>(draft_block), static_cast<int32_t>(bonus_block), group_d, group_b,
      groups,
      cu_num_draft, out, err);
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
