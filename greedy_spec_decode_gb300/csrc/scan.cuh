// scan.cuh -- element and 16-byte-vector steps of the argmax scan over a
// contiguous run of logits (fp32 or bf16), shared by the per-shard kernel
// (argmax.cu) and the block-granular kernel (blocks.cu).
#pragma once

#include "common.cuh"

namespace sga {
namespace {

template <bool kBf16>
__device__ __forceinline__ float load_elem(const char *p, int j) {
  if (kBf16) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p) + j);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  } else {
    return __ldg(reinterpret_cast<const float *>(p) + j);
  }
}

// NaN-propagating maximum of the elements of one 16-byte vector.
template <bool kBf16>
__device__ __forceinline__ float vec_max(const uint4 a) {
  if (kBf16) {
    const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(a.x, a.y), max_nan_bf16x2(a.z, a.w));
    return max_nan(bf16_lo(m), bf16_hi(m));
  } else {
    return max_nan(max_nan(__uint_as_float(a.x), __uint_as_float(a.y)),
                   max_nan(__uint_as_float(a.z), __uint_as_float(a.w)));
  }
}

// First element of a vector (ids id, id+1, ...) that the scan rule would
// take over `best`; updates (best, best_id).
template <bool kBf16>
__device__ __forceinline__ void scan_vec(const uint4 a, int32_t id, float &best, int32_t &best_id) {
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (kBf16) {
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
    } else {
      const float x = __uint_as_float(w[k]);
      if (scan_better(x, best)) {
        best = x;
        best_id = id + k;
      }
    }
  }
}

// The scan rule over gathered statistics: entries (s, row) for s = 0..n-1
// (n >= 1) at stats[s * stride + row], visited in ascending s (ascending
// ids), the first NaN sticking and ties keeping the lower s.  The loads go
// in batches of eight, each batch issued (bounds-predicated, so a short list
// of two to seven shards is one batch) before its comparisons, so that one
// memory latency covers eight entries; the comparison order is the plain
// sequential one.
__device__ __forceinline__ sga_stat reduce_stats(const sga_stat *__restrict__ stats, int n,
                                                 int64_t stride, int64_t row) {
  sga_stat b;
  b.v = 0.0f;
  b.id = 0;
  for (int s = 0; s < n; s += 8) {
    sga_stat c[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s + u < n) c[u] = stats[static_cast<int64_t>(s + u) * stride + row];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s + u < n && (s + u == 0 || scan_better(c[u].v, b.v))) b = c[u];
  }
  return b;
}

}  // namespace
}  // namespace sga
