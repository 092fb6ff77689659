/* A C99 client of libsga.so: include/sga.h must compile as plain C and the
 * library must be usable with nothing but the CUDA runtime.
 *
 *   abi_client host   -- argument validation only (no GPU needed)
 *   abi_client gpu    -- argmax of 2 shards + reduce on cudaMalloc'd buffers,
 *                        checked against a brute-force scan written here
 * Exit status 0 on success. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "sga.h"

static int host_checks(void) {
  int bad = 0;
  if (sga_version() != SGA_VERSION) bad |= 1;
  /* unknown dtype, empty batch and a NULL pointer are rejected or accepted
   * before any CUDA call */
  if (sga_local_argmax((const void *)0x10000, 9, 4, 10, 0, 10, 10, (sga_stat *)0x10000, 0) !=
      SGA_ERR_DTYPE)
    bad |= 2;
  if (sga_local_argmax(0, SGA_BF16, 0, 10, 0, 10, 10, 0, 0) != SGA_OK) bad |= 4;
  if (sga_greedy_verify((const sga_stat *)0x10000, 1, 3, 0, 0, 3, 0, 0, 0, 0, 0, 0) != SGA_ERR_NULL)
    bad |= 8;
  if (sga_status_string(SGA_ERR_SHARD) == 0 || strlen(sga_status_string(SGA_ERR_SHARD)) == 0)
    bad |= 16;
  if (sizeof(sga_stat) != 8) bad |= 32;
  /* block-granular statistics: slot count is host arithmetic; a zero block
   * size is rejected before any CUDA call */
  if (sga_block_slots(67350, 67349, 8192, 1024) != 67) bad |= 64;
  if (sga_local_argmax_blocks((const void *)0x10000, SGA_BF16, 4, 100, 0, 100, 100, 0, 16, 0, 0,
                              (sga_stat *)0x10000, 0) != SGA_ERR_SIZE)
    bad |= 64;
  /* the LM head over several shards in one call: the workspace size is host
   * arithmetic, and overlapping shards are rejected before any CUDA call */
  {
    const int64_t starts[2] = {0, 40}, widths[2] = {64, 64};
    const size_t ws = sga_lmhead_argmax_shards_workspace(16, 2, widths);
    if (ws != 2u * 16u * 256u * 8u) bad |= 128;
    if (sga_lmhead_argmax_shards((const void *)0x10000, 16, 64, (const void *)0x10000, 2, starts,
                                 widths, 128, (sga_stat *)0x10000, (void *)0x10000, ws,
                                 0) != SGA_ERR_SHARD)
      bad |= 128;
  }
  return bad;
}

/* Declarations of the few CUDA runtime calls used, so the client needs no CUDA
 * header (the library links the runtime statically; this client links
 * libcudart dynamically). */
typedef int cudaError_t;
extern cudaError_t cudaMalloc(void **ptr, size_t size);
extern cudaError_t cudaFree(void *ptr);
extern cudaError_t cudaMemcpy(void *dst, const void *src, size_t count, int kind);
extern cudaError_t cudaDeviceSynchronize(void);

static int gpu_checks(void) {
  enum { R = 5, V = 1000 };
  float *x = (float *)malloc(sizeof(float) * R * V);
  for (int i = 0; i < R * V; ++i) x[i] = (float)((i * 7919) % 1009) - 500.0f;
  x[2 * V + 640] = 1e6f; /* a clear winner in shard 1 of row 2 */
  void *dx = 0, *dstats = 0, *dids = 0;
  int bad = 0;
  if (cudaMalloc(&dx, sizeof(float) * R * V) || cudaMalloc(&dstats, 16 * R) ||
      cudaMalloc(&dids, 4 * R))
    return 64;
  cudaMemcpy(dx, x, sizeof(float) * R * V, 1 /* host to device */);
  if (sga_local_argmax(dx, SGA_F32, R, V, 0, 600, V, (sga_stat *)dstats, 0) != SGA_OK) bad |= 128;
  if (sga_local_argmax((const float *)dx + 600, SGA_F32, R, V, 600, 400, V,
                       (sga_stat *)dstats + R, 0) != SGA_OK)
    bad |= 256;
  if (sga_shard_reduce((const sga_stat *)dstats, 2, R, 0, (int32_t *)dids, 0, 0, 0) != SGA_OK)
    bad |= 512;
  cudaDeviceSynchronize();
  int32_t ids[R];
  cudaMemcpy(ids, dids, sizeof(ids), 2 /* device to host */);
  for (int r = 0; r < R; ++r) {
    int best = 0;
    for (int j = 1; j < V; ++j)
      if (x[r * V + j] > x[r * V + best]) best = j;
    if (ids[r] != best) bad |= 1024;
  }
  if (ids[2] != 640) bad |= 2048;
  uint32_t word = 1;
  if (sga_device_error(&word) != SGA_OK || word != 0) bad |= 4096;
  cudaFree(dx);
  cudaFree(dstats);
  cudaFree(dids);
  free(x);
  return bad;
}

int main(int argc, char **argv) {
  int bad = host_checks();
  if (argc > 1 && strcmp(argv[1], "gpu") == 0) bad |= gpu_checks();
  printf("abi_client: %s (flags %d)\n", bad ? "FAIL" : "ok", bad);
  return bad ? 1 : 0;
}
