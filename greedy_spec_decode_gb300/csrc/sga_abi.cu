// sga_abi.cu -- the extern "C" entry points of libsga.so: host-side argument
// validation (before any CUDA call, so a bad call enqueues nothing), the
// per-device cache (SM count, compute capability, address of the device error
// word) and dispatch to the kernel launchers.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

// OR-ed by kernels instead of trapping; read by sga_device_error().
__device__ uint32_t g_sga_error_word;

namespace {

struct DeviceInfo {
  bool ready;
  uintptr_t ctx;  // context the entry was looked up in
  int status;     // SGA_OK or the error the set-up hit
  int num_sms;
  uint32_t *err;
};

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

// Per-device facts for the current device, looked up once per context.
int current_device(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SGA_ERR_DEVICE;
  const uintptr_t ctx = sga::current_context_key();
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo &d = g_devices[dev];
  if (!d.ready || ctx == 0 || ctx != d.ctx) {
    int major = 0, minor = 0, sms = 0;
    d.status = SGA_OK;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      d.status = SGA_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      d.status = SGA_ERR_DEVICE;  // the library carries sm_103a code only
    } else {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_sga_error_word) != cudaSuccess) d.status = SGA_ERR_CUDA;
      d.err = static_cast<uint32_t *>(p);
      d.num_sms = sms;
    }
    d.ctx = sga::current_context_key();  // the look-up above made a context current
    d.ready = true;
  }
  *out = d;
  return d.status;
}

}  // namespace

namespace sga {

uintptr_t current_context_key() {
  using GetCurrent = CUresult (*)(CUcontext *);
  static GetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCurrent>(p);
  });
  if (fn == nullptr) return 1;  // no driver entry point: one context per device assumed
  CUcontext c = nullptr;
  if (fn(&c) != CUDA_SUCCESS) return 0;
  return reinterpret_cast<uintptr_t>(c);
}

}  // namespace sga

namespace {

bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

int check_shard(int64_t shard_start, int64_t shard_width, int64_t org_vocab) {
  if (shard_start < 0 || shard_width <= 0) return SGA_ERR_SHARD;
  if (shard_start + shard_width > SGA_MAX_VOCAB) return SGA_ERR_VOCAB;
  if (org_vocab <= 0 || org_vocab > SGA_MAX_VOCAB) return SGA_ERR_VOCAB;
  return SGA_OK;
}

// Number of ids of [shard_start, shard_start + width) below org_vocab.
int64_t valid_ids(int64_t shard_start, int64_t width, int64_t org_vocab) {
  int64_t v = org_vocab - shard_start;
  if (v < 0) v = 0;
  return v < width ? v : width;
}

int launch_status(cudaError_t e) {
  if (e != cudaSuccess) return SGA_ERR_CUDA;
  return SGA_OK;
}

}  // namespace

extern "C" {

int sga_version(void) { return SGA_VERSION; }

const char *sga_status_string(int status) {
  switch (status) {
    case SGA_OK: return "ok";
    case SGA_ERR_NULL: return "a required pointer is NULL";
    case SGA_ERR_SIZE: return "a size or count is negative or out of range";
    case SGA_ERR_SHARD: return "shard outside the vocabulary or wider than the row stride";
    case SGA_ERR_VOCAB: return "org_vocab <= 0 or an id would reach 2^24";
    case SGA_ERR_DTYPE: return "unknown dtype";
    case SGA_ERR_ALIGN: return "pointer not aligned as required";
    case SGA_ERR_WORKSPACE: return "workspace too small";
    case SGA_ERR_MAXK: return "max_k outside [1, SGA_MAX_K]";
    case SGA_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case SGA_ERR_DEVICE: return "current device is not compute capability 10.3 (GB300)";
    case SGA_ERR_UNSUPPORTED: return "shape not supported by this kernel";
    default: return "unknown status";
  }
}

int sga_local_argmax(const void *logits, int dtype, int64_t rows, int64_t ld,
                     int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                     sga_stat *out_stats, sga_stream stream) {
  if (dtype != SGA_F32 && dtype != SGA_BF16) return SGA_ERR_DTYPE;
  if (rows < 0 || rows > (int64_t(1) << 28)) return SGA_ERR_SIZE;
  int st = check_shard(shard_start, shard_width, org_vocab);
  if (st != SGA_OK) return st;
  if (ld < shard_width) return SGA_ERR_SHARD;
  if (rows == 0) return SGA_OK;
  if (logits == nullptr || out_stats == nullptr) return SGA_ERR_NULL;
  if (misaligned(logits, dtype == SGA_BF16 ? 2 : 4) || misaligned(out_stats, 8))
    return SGA_ERR_ALIGN;
  DeviceInfo d;
  if ((st = current_device(&d)) != SGA_OK) return st;
  return launch_status(sga::launch_local_argmax(
      logits, dtype, rows, ld, shard_start, shard_width,
      valid_ids(shard_start, shard_width, org_vocab), out_stats, d.num_sms, d.err,
      static_cast<cudaStream_t>(stream)));
}

int sga_local_argmax_shards(const void *logits, int dtype, int64_t rows, int64_t ld,
                            int num_shards, const int64_t *shard_starts,
                            const int64_t *shard_widths, int64_t org_vocab,
                            sga_stat *out_stats, sga_stream stream) {
  if (dtype != SGA_F32 && dtype != SGA_BF16) return SGA_ERR_DTYPE;
  if (num_shards < 1 || num_shards > sga::kMaxShardsPerLaunch) return SGA_ERR_SIZE;
  if (rows < 0 || rows * num_shards > (int64_t(1) << 28)) return SGA_ERR_SIZE;
  if (shard_starts == nullptr || shard_widths == nullptr) return SGA_ERR_NULL;
  int64_t cols[sga::kMaxShardsPerLaunch], valids[sga::kMaxShardsPerLaunch];
  for (int s = 0; s < num_shards; ++s) {
    const int st = check_shard(shard_starts[s], shard_widths[s], org_vocab);
    if (st != SGA_OK) return st;
    if (s > 0 && shard_starts[s] < shard_starts[s - 1] + shard_widths[s - 1]) return SGA_ERR_SHARD;
    cols[s] = shard_starts[s] - shard_starts[0];
    valids[s] = valid_ids(shard_starts[s], shard_widths[s], org_vocab);
  }
  if (cols[num_shards - 1] + shard_widths[num_shards - 1] > ld) return SGA_ERR_SHARD;
  if (rows == 0) return SGA_OK;
  if (logits == nullptr || out_stats == nullptr) return SGA_ERR_NULL;
  if (misaligned(logits, dtype == SGA_BF16 ? 2 : 4) || misaligned(out_stats, 8))
    return SGA_ERR_ALIGN;
  DeviceInfo d;
  const int st = current_device(&d);
  if (st != SGA_OK) return st;
  return launch_status(sga::launch_local_argmax_table(logits, dtype, rows, ld, num_shards,
                                                      shard_starts, cols, valids, out_stats,
                                                      d.num_sms, d.err,
                                                      static_cast<cudaStream_t>(stream)));
}

int64_t sga_block_slots(int64_t shard_start, int64_t shard_width, int64_t draft_block,
                        int64_t bonus_block) {
  const int st = check_shard(shard_start, shard_width, 1);
  if (st != SGA_OK) return st;
  if (draft_block < 1 || draft_block > SGA_MAX_VOCAB || bonus_block < 1 ||
      bonus_block > SGA_MAX_VOCAB)
    return SGA_ERR_SIZE;
  return sga::block_slots(shard_start, shard_width, draft_block, bonus_block);
}

int sga_local_argmax_blocks(const void *logits, int dtype, int64_t rows, int64_t ld,
                            int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                            int64_t draft_block, int64_t bonus_block, int num_reqs,
                            const int32_t *cu_num_draft, sga_stat *out_stats,
                            sga_stream stream) {
  if (dtype != SGA_F32 && dtype != SGA_BF16) return SGA_ERR_DTYPE;
  int st = check_shard(shard_start, shard_width, org_vocab);
  if (st != SGA_OK) return st;
  const int64_t slots = sga_block_slots(shard_start, shard_width, draft_block, bonus_block);
  if (slots < 0) return static_cast<int>(slots);
  if (rows < 0 || rows * slots > (int64_t(1) << 28)) return SGA_ERR_SIZE;
  if (ld < shard_width) return SGA_ERR_SHARD;
  if (cu_num_draft != nullptr && num_reqs < 1) return SGA_ERR_SIZE;
  if (rows == 0) return SGA_OK;
  if (logits == nullptr || out_stats == nullptr) return SGA_ERR_NULL;
  if (misaligned(logits, dtype == SGA_BF16 ? 2 : 4) || misaligned(out_stats, 8) ||
      misaligned(cu_num_draft, 4))
    return SGA_ERR_ALIGN;
  DeviceInfo d;
  if ((st = current_device(&d)) != SGA_OK) return st;
  return launch_status(sga::launch_block_argmax(logits, dtype, rows, ld, shard_start, shard_width,
                                                org_vocab, draft_block, bonus_block, num_reqs,
                                                cu_num_draft, out_stats, d.num_sms, d.err,
                                                static_cast<cudaStream_t>(stream)));
}

int sga_local_argmax_blocks_shards(const void *logits, int dtype, int64_t rows, int64_t ld,
                                   int num_shards, const int64_t *shard_starts,
                                   const int64_t *shard_widths, int64_t org_vocab,
                                   int64_t draft_block, int64_t bonus_block, int num_reqs,
                                   const int32_t *cu_num_draft, sga_stat *out_stats,
                                   sga_stream stream) {
  if (dtype != SGA_F32 && dtype != SGA_BF16) return SGA_ERR_DTYPE;
  if (num_shards < 1 || num_shards > sga::kMaxBlockShards) return SGA_ERR_SIZE;
  if (shard_starts == nullptr || shard_widths == nullptr) return SGA_ERR_NULL;
  int64_t cols[sga::kMaxBlockShards];
  int64_t slots = 0;
  for (int s = 0; s < num_shards; ++s) {
    int st = check_shard(shard_starts[s], shard_widths[s], org_vocab);
    if (st != SGA_OK) return st;
    if (s > 0 && shard_starts[s] < shard_starts[s - 1] + shard_widths[s - 1]) return SGA_ERR_SHARD;
    const int64_t n = sga_block_slots(shard_starts[s], shard_widths[s], draft_block, bonus_block);
    if (n < 0) return static_cast<int>(n);
    slots += n;
    cols[s] = shard_starts[s] - shard_starts[0];
  }
  if (cols[num_shards - 1] + shard_widths[num_shards - 1] > ld) return SGA_ERR_SHARD;
  if (rows < 0 || rows * slots > (int64_t(1) << 28)) return SGA_ERR_SIZE;
  if (cu_num_draft != nullptr && num_reqs < 1) return SGA_ERR_SIZE;
  if (rows == 0) return SGA_OK;
  if (logits == nullptr || out_stats == nullptr) return SGA_ERR_NULL;
  if (misaligned(logits, dtype == SGA_BF16 ? 2 : 4) || misaligned(out_stats, 8) ||
      misaligned(cu_num_draft, 4))
    return SGA_ERR_ALIGN;
  DeviceInfo d;
  const int st = current_device(&d);
  if (st != SGA_OK) return st;
  return launch_status(sga::launch_block_argmax_table(
      logits, dtype, rows, ld, num_shards, shard_starts, cols, shard_widths, org_vocab,
      draft_block, bonus_block, num_reqs, cu_num_draft, out_stats, d.num_sms, d.err,
      static_cast<cudaStream_t>(stream)));
}

int sga_shard_reduce(const sga_stat *stats, int num_shards, int64_t rows, float *out_vals,
                     int32_t *out_ids, const int64_t *d2t, int64_t d2t_len,
                     sga_stream stream) {
  if (num_shards < 1 || num_shards > 4096) return SGA_ERR_SIZE;
  if (rows < 0 || rows > (int64_t(1) << 40)) return SGA_ERR_SIZE;
  if (d2t != nullptr && d2t_len < 0) return SGA_ERR_SIZE;
  if (rows == 0) return SGA_OK;
  if (stats == nullptr || out_ids == nullptr) return SGA_ERR_NULL;
  if (misaligned(stats, 8) || misaligned(out_ids, 4) || misaligned(out_vals, 4) ||
      misaligned(d2t, 8))
    return SGA_ERR_ALIGN;
  DeviceInfo d;
  int st = current_device(&d);
  if (st != SGA_OK) return st;
  return launch_status(sga::launch_shard_reduce(stats, num_shards, rows, out_vals, out_ids, d2t,
                                                d2t_len, d.err,
                                                static_cast<cudaStream_t>(stream)));
}

int sga_greedy_verify(const sga_stat *stats, int num_shards, int num_reqs,
                      const int32_t *cu_num_draft, const int32_t *draft_tokens, int max_k,
                      int32_t *out_sampled, int32_t *out_num_sampled,
                      int32_t *out_num_rejected, int32_t *out_bonus,
                      int32_t *out_target_ids, sga_stream stream) {
  return sga_greedy_verify_prefill(stats, num_shards, num_reqs, cu_num_draft, draft_tokens,
                                   nullptr, max_k, out_sampled, out_num_sampled,
                                   out_num_rejected, out_bonus, out_target_ids, stream);
}

int sga_greedy_verify_prefill(const sga_stat *stats, int num_shards, int num_reqs,
                              const int32_t *cu_num_draft, const int32_t *draft_tokens,
                              const uint8_t *in_prefill, int max_k, int32_t *out_sampled,
                              int32_t *out_num_sampled, int32_t *out_num_rejected,
                              int32_t *out_bonus, int32_t *out_target_ids, sga_stream stream) {
  if (num_shards < 1 || num_shards > 4096) return SGA_ERR_SIZE;
  if (num_reqs < 0 || num_reqs > (1 << 26)) return SGA_ERR_SIZE;
  if (max_k < 1 || max_k > SGA_MAX_K) return SGA_ERR_MAXK;
  if (num_reqs == 0) return SGA_OK;
  if (stats == nullptr || cu_num_draft == nullptr || out_sampled == nullptr ||
      out_num_sampled == nullptr || out_num_rejected == nullptr || out_bonus == nullptr)
    return SGA_ERR_NULL;
  if (misaligned(stats, 8) || misaligned(cu_num_draft, 4) || misaligned(draft_tokens, 4) ||
      misaligned(out_sampled, 4) || misaligned(out_num_sampled, 4) ||
      misaligned(out_num_rejected, 4) || misaligned(out_bonus, 4) ||
      misaligned(out_target_ids, 4))
    return SGA_ERR_ALIGN;
  DeviceInfo d;
  int st = current_device(&d);
  if (st != SGA_OK) return st;
  return launch_status(sga::launch_greedy_verify(
      stats, num_shards, num_reqs, cu_num_draft, draft_tokens, max_k, out_sampled,
      out_num_sampled, out_num_rejected, out_bonus, out_target_ids, d.err,
      static_cast<cudaStream_t>(stream), in_prefill));
}

size_t sga_lmhead_argmax_workspace(int64_t M, int64_t shard_width) {
  if (M <= 0 || shard_width <= 0) return 0;
  return sga::lmhead_workspace_bytes(M, shard_width);
}

int sga_lmhead_argmax(const void *hidden, int64_t M, int64_t H, const void *weight_shard,
                      int64_t shard_start, int64_t shard_width, int64_t org_vocab,
                      sga_stat *out_stats, void *workspace, size_t workspace_bytes,
                      sga_stream stream) {
  if (M < 0 || M > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  if (H <= 0 || H % 64 != 0 || H > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  int st = check_shard(shard_start, shard_width, org_vocab);
  if (st != SGA_OK) return st;
  if (M == 0) return SGA_OK;
  if (hidden == nullptr || weight_shard == nullptr || out_stats == nullptr ||
      workspace == nullptr)
    return SGA_ERR_NULL;
  if (misaligned(hidden, 16) || misaligned(weight_shard, 16) || misaligned(out_stats, 8) ||
      misaligned(workspace, 8))
    return SGA_ERR_ALIGN;
  if (workspace_bytes < sga::lmhead_workspace_bytes(M, shard_width)) return SGA_ERR_WORKSPACE;
  DeviceInfo d;
  if ((st = current_device(&d)) != SGA_OK) return st;
  const cudaError_t e = sga::launch_lmhead_argmax(
      hidden, M, H, weight_shard, shard_start, shard_width,
      valid_ids(shard_start, shard_width, org_vocab), out_stats, workspace, d.num_sms, d.err,
      static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return SGA_ERR_UNSUPPORTED;
  return launch_status(e);
}

int sga_lmhead_argmax_fp8(const void *hidden_q, const float *hidden_scale, int64_t M, int64_t H,
                          const void *weight_q, float weight_scale, int64_t shard_start,
                          int64_t shard_width, int64_t org_vocab, sga_stat *out_stats,
                          void *workspace, size_t workspace_bytes, sga_stream stream) {
  if (M < 0 || M > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  if (H <= 0 || H % 128 != 0 || H > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  if (!(weight_scale > 0.0f) || !(weight_scale < 3.4e38f)) return SGA_ERR_SIZE;
  int st = check_shard(shard_start, shard_width, org_vocab);
  if (st != SGA_OK) return st;
  if (M == 0) return SGA_OK;
  if (hidden_q == nullptr || weight_q == nullptr || out_stats == nullptr || workspace == nullptr)
    return SGA_ERR_NULL;
  if (misaligned(hidden_q, 16) || misaligned(weight_q, 16) || misaligned(out_stats, 8) ||
      misaligned(workspace, 8) || misaligned(hidden_scale, 4))
    return SGA_ERR_ALIGN;
  if (workspace_bytes < sga::lmhead_workspace_bytes(M, shard_width)) return SGA_ERR_WORKSPACE;
  DeviceInfo d;
  if ((st = current_device(&d)) != SGA_OK) return st;
  const cudaError_t e = sga::launch_lmhead_argmax(
      hidden_q, M, H, weight_q, shard_start, shard_width,
      valid_ids(shard_start, shard_width, org_vocab), out_stats, workspace, d.num_sms, d.err,
      static_cast<cudaStream_t>(stream), true, hidden_scale, weight_scale);
  if (e == cudaErrorNotSupported) return SGA_ERR_UNSUPPORTED;
  return launch_status(e);
}

// Shared checks of the multi-shard LM-head entry points: the shards (each as
// in sga_lmhead_argmax, ascending, non-overlapping) and their valid ids.
static int check_lm_shards(int num_shards, const int64_t *starts, const int64_t *widths,
                           int64_t org_vocab, int64_t *valids) {
  if (num_shards < 1 || num_shards > sga::kMaxLmShards) return SGA_ERR_SIZE;
  if (starts == nullptr || widths == nullptr) return SGA_ERR_NULL;
  for (int s = 0; s < num_shards; ++s) {
    const int st = check_shard(starts[s], widths[s], org_vocab);
    if (st != SGA_OK) return st;
    if (s > 0 && starts[s] < starts[s - 1] + widths[s - 1]) return SGA_ERR_SHARD;
    valids[s] = valid_ids(starts[s], widths[s], org_vocab);
  }
  return SGA_OK;
}

size_t sga_lmhead_argmax_shards_workspace(int64_t M, int num_shards,
                                          const int64_t *shard_widths) {
  if (M <= 0 || num_shards < 1 || num_shards > sga::kMaxLmShards || shard_widths == nullptr)
    return 0;
  for (int s = 0; s < num_shards; ++s)
    if (shard_widths[s] <= 0) return 0;
  return sga::lmhead_shards_workspace_bytes(M, num_shards, shard_widths);
}

static int lmhead_shards_common(const void *hidden, const float *hidden_scale, int64_t M,
                                int64_t H, const void *weight, bool fp8, float weight_scale,
                                int num_shards, const int64_t *shard_starts,
                                const int64_t *shard_widths, int64_t org_vocab,
                                sga_stat *out_stats, void *workspace, size_t workspace_bytes,
                                sga_stream stream) {
  if (M < 0 || M > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  if (H <= 0 || H % (fp8 ? 128 : 64) != 0 || H > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  if (fp8 && (!(weight_scale > 0.0f) || !(weight_scale < 3.4e38f))) return SGA_ERR_SIZE;
  int64_t valids[sga::kMaxLmShards];
  int st = check_lm_shards(num_shards, shard_starts, shard_widths, org_vocab, valids);
  if (st != SGA_OK) return st;
  if (M == 0) return SGA_OK;
  if (hidden == nullptr || weight == nullptr || out_stats == nullptr || workspace == nullptr)
    return SGA_ERR_NULL;
  if (misaligned(hidden, 16) || misaligned(weight, 16) || misaligned(out_stats, 8) ||
      misaligned(workspace, 8) || misaligned(hidden_scale, 4))
    return SGA_ERR_ALIGN;
  if (workspace_bytes < sga::lmhead_shards_workspace_bytes(M, num_shards, shard_widths))
    return SGA_ERR_WORKSPACE;
  DeviceInfo d;
  if ((st = current_device(&d)) != SGA_OK) return st;
  const cudaError_t e = sga::launch_lmhead_argmax_shards(
      hidden, M, H, weight, num_shards, shard_starts, shard_widths, valids, out_stats, workspace,
      d.num_sms, d.err, static_cast<cudaStream_t>(stream), fp8, fp8 ? hidden_scale : nullptr,
      fp8 ? weight_scale : 1.0f);
  if (e == cudaErrorNotSupported) return SGA_ERR_UNSUPPORTED;
  return launch_status(e);
}

int sga_lmhead_argmax_shards(const void *hidden, int64_t M, int64_t H, const void *weight,
                             int num_shards, const int64_t *shard_starts,
                             const int64_t *shard_widths, int64_t org_vocab,
                             sga_stat *out_stats, void *workspace, size_t workspace_bytes,
                             sga_stream stream) {
  return lmhead_shards_common(hidden, nullptr, M, H, weight, false, 1.0f, num_shards,
                              shard_starts, shard_widths, org_vocab, out_stats, workspace,
                              workspace_bytes, stream);
}

int sga_lmhead_argmax_shards_fp8(const void *hidden_q, const float *hidden_scale, int64_t M,
                                 int64_t H, const void *weight_q, float weight_scale,
                                 int num_shards, const int64_t *shard_starts,
                                 const int64_t *shard_widths, int64_t org_vocab,
                                 sga_stat *out_stats, void *workspace, size_t workspace_bytes,
                                 sga_stream stream) {
  return lmhead_shards_common(hidden_q, hidden_scale, M, H, weight_q, true, weight_scale,
                              num_shards, shard_starts, shard_widths, org_vocab, out_stats,
                              workspace, workspace_bytes, stream);
}

// Same work as sga_lmhead_argmax, with the library's fixed scratch array in
// place of a caller workspace, for callers that cannot allocate device memory.
int sga_lmhead_argmax_noalloc(const void *hidden, int64_t M, int64_t H,
                              const void *weight_shard, int64_t shard_start,
                              int64_t shard_width, int64_t org_vocab, sga_stat *out_stats,
                              sga_stream stream) {
  if (M < 0 || M > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  if (H <= 0 || H % 64 != 0 || H > (int64_t(1) << 20)) return SGA_ERR_SIZE;
  int st = check_shard(shard_start, shard_width, org_vocab);
  if (st != SGA_OK) return st;
  if (M == 0) return SGA_OK;
  if (sga::lmhead_workspace_bytes(M, shard_width) > sga::lmhead_noalloc_scratch_bytes())
    return SGA_ERR_WORKSPACE;
  if (hidden == nullptr || weight_shard == nullptr || out_stats == nullptr) return SGA_ERR_NULL;
  if (misaligned(hidden, 16) || misaligned(weight_shard, 16) || misaligned(out_stats, 8))
    return SGA_ERR_ALIGN;
  DeviceInfo d;
  if ((st = current_device(&d)) != SGA_OK) return st;
  sga_stat *scratch = nullptr;
  if (sga::lmhead_noalloc_scratch(&scratch) != cudaSuccess) return SGA_ERR_CUDA;
  const cudaError_t e = sga::launch_lmhead_argmax(
      hidden, M, H, weight_shard, shard_start, shard_width,
      valid_ids(shard_start, shard_width, org_vocab), out_stats, scratch, d.num_sms, d.err,
      static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return SGA_ERR_UNSUPPORTED;
  return launch_status(e);
}

int sga_selftest_wait_timeout(uint64_t limit_ns, uint64_t *waited_ns, sga_stream stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ull) return SGA_ERR_SIZE;
  if (misaligned(waited_ns, 8)) return SGA_ERR_ALIGN;
  DeviceInfo d;
  const int st = current_device(&d);
  if (st != SGA_OK) return st;
  return launch_status(sga::launch_selftest_timeout(
      limit_ns, d.err, reinterpret_cast<unsigned long long *>(waited_ns),
      static_cast<cudaStream_t>(stream)));
}

int sga_device_error(uint32_t *out_word) {
  if (out_word == nullptr) return SGA_ERR_NULL;
  DeviceInfo d;
  int st = current_device(&d);
  if (st != SGA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return SGA_ERR_CUDA;
  if (cudaMemcpy(out_word, d.err, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SGA_ERR_CUDA;
  return SGA_OK;
}

int sga_clear_device_error(void) {
  DeviceInfo d;
  int st = current_device(&d);
  if (st != SGA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return SGA_ERR_CUDA;
  if (cudaMemset(d.err, 0, sizeof(uint32_t)) != cudaSuccess) return SGA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return SGA_ERR_CUDA;
  return SGA_OK;
}

}  // extern "C"
