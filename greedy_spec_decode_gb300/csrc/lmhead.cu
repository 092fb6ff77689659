// lmhead.cu -- fused LM-head GEMM + per-shard argmax (tcgen05 / TMEM / TMA).
#include "common.cuh"

namespace sga {

size_t lmhead_workspace_bytes(int64_t M, int64_t width) {
  const int64_t n_tiles = (width + 255) / 256;
  return static_cast<size_t>(n_tiles * M) * sizeof(sga_stat);
}

cudaError_t launch_lmhead_argmax(const void *, int64_t, int64_t, const void *, int64_t, int64_t,
                                 int64_t, sga_stat *, void *, int, uint32_t *, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace sga
