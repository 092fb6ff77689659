// common.cuh -- device helpers shared by the sga kernels (argmax order,
// widening, loads, warp merge, programmatic dependent launch) and, through
// launchers.h, the internal launcher declarations used by sga_abi.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sga.h"

namespace sga {

// Sentinel id of "no element seen yet": larger than every real id, so any
// recorded element beats it under the argmax order below.
constexpr int32_t kNoId = 0x7fffffff;

__device__ __forceinline__ bool is_nan(float x) { return x != x; }

// Scan rule (vLLM PR #62604, Purpose item 2: "lowest id on ties, NaN wins, as
// torch.argmax"): while ids are visited in ascending order, a candidate
// replaces the running best when the best is not NaN and the candidate is NaN
// or strictly greater.  This keeps the first NaN and the lowest tied id.
__device__ __forceinline__ bool scan_better(float cand, float best) {
  return !is_nan(best) && (is_nan(cand) || cand > best);
}

// The same order as a comparison of two (value, id) pairs visited in any
// order: NaN beats numbers, larger beats smaller (+0 == -0), then lower id.
// Ids are unique within a row, so this is a strict total order and any
// reduction tree gives the same winner.
__device__ __forceinline__ bool pair_beats(float av, int32_t ai, float bv, int32_t bi) {
  const bool an = is_nan(av), bn = is_nan(bv);
  if (an || bn) return an && (!bn || ai < bi);
  return av > bv || (av == bv && ai < bi);
}

// Exact widening of bf16 bits to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xffff0000u); }

// 16-byte streaming load that bypasses L1 (each logit is read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// max with NaN propagation (NaN if either input is NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Packed bf16x2 max with NaN propagation.
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel of the stream drains;
// pdl_wait() blocks until that kernel has completed and its writes are
// visible, pdl_launch_dependents() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void warp_argmax(float &v, int32_t &id) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int32_t oi = __shfl_xor_sync(0xffffffffu, id, off);
    if (pair_beats(ov, oi, v, id)) {
      v = ov;
      id = oi;
    }
  }
}

}  // namespace sga

#include "launchers.h"
