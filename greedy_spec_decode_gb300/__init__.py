"""Python binding of libsga.so: vocab-sharded greedy token selection on GB300.

Argument marshalling only.  Each function has the name of the C entry point
it calls (declared in include/sga.h), takes torch CUDA tensors where the C
call takes device pointers, passes data_ptr() values and the current torch
stream, and raises SgaError on a non-zero status.  Every step of the path
runs in the library's CUDA kernels; there is no fallback: if libsga.so has
not been built, every call raises.

Stats tensors are int32 [rows, 2] (8 bytes per row: fp32 value bits, int32
id); ``stat_values``/``stat_ids`` view the two columns.

Method: vLLM PR #34049 (Solution: local argmax per vocab shard, gather of
(max_value, global_index), cross-rank reduce), PR #39419 (draft-to-target
map after the local argmax), PR #62604 (Purpose items 1-2: dim-0 gathered
per-shard stats, one verify kernel; fused get_top_tokens with padding mask
and torch.argmax order).
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsga.so")

SGA_F32, SGA_BF16 = 0, 1
SGA_MAX_K = 15
SGA_MAX_VOCAB = 1 << 24
SGA_DEVERR_K_RANGE, SGA_DEVERR_D2T_RANGE, SGA_DEVERR_TIMEOUT, SGA_DEVERR_LAYOUT = 1, 2, 4, 8

_lib = None


class SgaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({sga_status_string(status)})")


def lib():
    """The loaded libsga.so (ctypes), with argument types set."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m greedy_spec_decode_gb300.build` (or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        sig = {
            "sga_version": ([], i32),
            "sga_status_string": ([i32], ctypes.c_char_p),
            "sga_local_argmax": ([vp, i32, i64, i64, i64, i64, i64, vp, vp], i32),
            "sga_local_argmax_shards": ([vp, i32, i64, i64, i32, vp, vp, i64, vp, vp], i32),
            "sga_block_slots": ([i64, i64, i64, i64], i64),
            "sga_local_argmax_blocks": ([vp, i32, i64, i64, i64, i64, i64, i64, i64, i32, vp,
                                         vp, vp], i32),
            "sga_local_argmax_blocks_shards": ([vp, i32, i64, i64, i32, vp, vp, i64, i64, i64,
                                                i32, vp, vp, vp], i32),
            "sga_shard_reduce": ([vp, i32, i64, vp, vp, vp, i64, vp], i32),
            "sga_greedy_verify": ([vp, i32, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp], i32),
            "sga_greedy_verify_prefill": ([vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                           vp], i32),
            "sga_lmhead_argmax_workspace": ([i64, i64], sz),
            "sga_lmhead_argmax_shards_workspace": ([i64, i32, vp], sz),
            "sga_lmhead_argmax_shards": ([vp, i64, i64, vp, i32, vp, vp, i64, vp, vp, sz, vp], i32),
            "sga_lmhead_argmax_shards_fp8": ([vp, vp, i64, i64, vp, ctypes.c_float, i32, vp, vp,
                                              i64, vp, vp, sz, vp], i32),
            "sga_lmhead_argmax": ([vp, i64, i64, vp, i64, i64, i64, vp, vp, sz, vp], i32),
            "sga_lmhead_argmax_fp8": ([vp, vp, i64, i64, vp, ctypes.c_float, i64, i64, i64, vp,
                                       vp, sz, vp], i32),
            "sga_device_error": ([ctypes.POINTER(ctypes.c_uint32)], i32),
            "sga_clear_device_error": ([], i32),
            "sga_selftest_wait_timeout": ([ctypes.c_uint64, vp, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def sga_version():
    return lib().sga_version()


def sga_status_string(status):
    return lib().sga_status_string(int(status)).decode()


def _check(fn, status):
    if status != 0:
        raise SgaError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SGA_F32
    if t.dtype == torch.bfloat16:
        return SGA_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def new_stats(rows, device="cuda"):
    """An int32 [rows, 2] tensor that holds `rows` stats."""
    return torch.empty((rows, 2), dtype=torch.int32, device=device)


def stat_values(stats):
    return stats[..., 0].view(torch.float32)


def stat_ids(stats):
    return stats[..., 1]


def sga_local_argmax(logits, shard_start, shard_width, org_vocab, out_stats, stream=None):
    """Per-shard argmax.  `logits` is a 2-D CUDA tensor whose column 0 is the
    shard's first id (a column slice of the full matrix, or a per-rank
    buffer), unit stride along the vocab; out_stats receives one stat per row
    (pass a slice of the gathered buffer to emulate all_gather on dim 0)."""
    if logits.dim() != 2 or (logits.size(1) > 1 and logits.stride(1) != 1):
        raise ValueError("logits must be 2-D with unit stride along the vocab")
    rows = logits.size(0)
    ld = logits.stride(0) if rows > 1 else max(logits.stride(0), shard_width)
    _check("sga_local_argmax", lib().sga_local_argmax(
        _ptr(logits), _dtype_code(logits), rows, ld, int(shard_start), int(shard_width),
        int(org_vocab), _ptr(out_stats), _stream(stream)))
    return out_stats


def sga_local_argmax_shards(logits, shards, org_vocab, out_stats, stream=None):
    """Per-shard argmax of several shards in one launch.  `logits` is a 2-D
    CUDA tensor whose column 0 is global id shards[0][0] (unit stride along
    the vocab); shards = [(start, width), ...] ascending; out_stats receives
    len(shards) * rows stats in shard-major (all_gather dim 0) order."""
    if logits.dim() != 2 or (logits.size(1) > 1 and logits.stride(1) != 1):
        raise ValueError("logits must be 2-D with unit stride along the vocab")
    n = len(shards)
    starts = (ctypes.c_int64 * n)(*[int(o) for o, _ in shards])
    widths = (ctypes.c_int64 * n)(*[int(w) for _, w in shards])
    rows = logits.size(0)
    ld = logits.stride(0) if rows > 1 else max(logits.stride(0), logits.size(1))
    _check("sga_local_argmax_shards", lib().sga_local_argmax_shards(
        _ptr(logits), _dtype_code(logits), rows, ld, n, starts, widths, int(org_vocab),
        _ptr(out_stats), _stream(stream)))
    return out_stats


def sga_block_slots(shard_start, shard_width, draft_block, bonus_block=None):
    """Stats per row that sga_local_argmax_blocks writes for one shard."""
    bonus_block = draft_block if bonus_block is None else bonus_block
    n = int(lib().sga_block_slots(int(shard_start), int(shard_width), int(draft_block),
                                  int(bonus_block)))
    _check("sga_block_slots", n if n < 0 else 0)
    return n


def sga_local_argmax_blocks(logits, shard_start, shard_width, org_vocab, draft_block,
                            out_stats, bonus_block=None, cu_num_draft=None, stream=None):
    """Block-granular stats of one shard: for every row, the argmax of each
    fixed global block of ids meeting the shard.  `logits` as for
    sga_local_argmax; out_stats receives sga_block_slots(...) * rows stats,
    piece-major.  With cu_num_draft (int32 CUDA tensor [N + 1]) the bonus row
    of each request uses bonus_block."""
    if logits.dim() != 2 or (logits.size(1) > 1 and logits.stride(1) != 1):
        raise ValueError("logits must be 2-D with unit stride along the vocab")
    bonus_block = draft_block if bonus_block is None else bonus_block
    rows = logits.size(0)
    ld = logits.stride(0) if rows > 1 else max(logits.stride(0), shard_width)
    num_reqs = 0 if cu_num_draft is None else cu_num_draft.numel() - 1
    _check("sga_local_argmax_blocks", lib().sga_local_argmax_blocks(
        _ptr(logits), _dtype_code(logits), rows, ld, int(shard_start), int(shard_width),
        int(org_vocab), int(draft_block), int(bonus_block), int(num_reqs), _ptr(cu_num_draft),
        _ptr(out_stats), _stream(stream)))
    return out_stats


def sga_local_argmax_blocks_shards(logits, shards, org_vocab, draft_block, out_stats,
                                   bonus_block=None, cu_num_draft=None, stream=None):
    """Block-granular stats of several shards in one launch.  `logits` is a
    2-D CUDA tensor whose column 0 is global id shards[0][0]; shards =
    [(start, width), ...] ascending; out_stats receives the shards' slots
    concatenated in shard order (see sga_block_slots), piece-major."""
    if logits.dim() != 2 or (logits.size(1) > 1 and logits.stride(1) != 1):
        raise ValueError("logits must be 2-D with unit stride along the vocab")
    bonus_block = draft_block if bonus_block is None else bonus_block
    n = len(shards)
    starts = (ctypes.c_int64 * n)(*[int(o) for o, _ in shards])
    widths = (ctypes.c_int64 * n)(*[int(w) for _, w in shards])
    rows = logits.size(0)
    ld = logits.stride(0) if rows > 1 else max(logits.stride(0), logits.size(1))
    num_reqs = 0 if cu_num_draft is None else cu_num_draft.numel() - 1
    _check("sga_local_argmax_blocks_shards", lib().sga_local_argmax_blocks_shards(
        _ptr(logits), _dtype_code(logits), rows, ld, n, starts, widths, int(org_vocab),
        int(draft_block), int(bonus_block), int(num_reqs), _ptr(cu_num_draft),
        _ptr(out_stats), _stream(stream)))
    return out_stats


def sga_shard_reduce(stats, num_shards, rows, out_ids, out_vals=None, d2t=None, stream=None):
    """Global argmax per row from the gathered stats [num_shards * rows];
    with d2t (int64 CUDA tensor) the ids are mapped k -> k + d2t[k]."""
    _check("sga_shard_reduce", lib().sga_shard_reduce(
        _ptr(stats), int(num_shards), int(rows), _ptr(out_vals), _ptr(out_ids), _ptr(d2t),
        0 if d2t is None else d2t.numel(), _stream(stream)))
    return out_ids


def sga_greedy_verify(stats, num_shards, cu_num_draft, draft_tokens, max_k, out_sampled,
                      out_num_sampled, out_num_rejected, out_bonus, out_target_ids=None,
                      stream=None):
    """Fused cross-shard reduce + greedy verification (see include/sga.h)."""
    num_reqs = cu_num_draft.numel() - 1
    _check("sga_greedy_verify", lib().sga_greedy_verify(
        _ptr(stats), int(num_shards), int(num_reqs), _ptr(cu_num_draft),
        _ptr(draft_tokens) if draft_tokens is not None and draft_tokens.numel() else None,
        int(max_k), _ptr(out_sampled), _ptr(out_num_sampled), _ptr(out_num_rejected),
        _ptr(out_bonus), _ptr(out_target_ids), _stream(stream)))


def sga_greedy_verify_prefill(stats, num_shards, cu_num_draft, draft_tokens, in_prefill, max_k,
                              out_sampled, out_num_sampled, out_num_rejected, out_bonus,
                              out_target_ids=None, stream=None):
    """sga_greedy_verify where in_prefill (a uint8/bool CUDA tensor [num_reqs],
    or None) marks the requests still in prefill, which emit nothing."""
    num_reqs = cu_num_draft.numel() - 1
    if in_prefill is not None and in_prefill.dtype not in (torch.uint8, torch.bool):
        raise ValueError("in_prefill must be a uint8 or bool tensor")
    _check("sga_greedy_verify_prefill", lib().sga_greedy_verify_prefill(
        _ptr(stats), int(num_shards), int(num_reqs), _ptr(cu_num_draft),
        _ptr(draft_tokens) if draft_tokens is not None and draft_tokens.numel() else None,
        _ptr(in_prefill), int(max_k), _ptr(out_sampled), _ptr(out_num_sampled),
        _ptr(out_num_rejected), _ptr(out_bonus), _ptr(out_target_ids), _stream(stream)))


def sga_lmhead_argmax_workspace(M, shard_width):
    return int(lib().sga_lmhead_argmax_workspace(int(M), int(shard_width)))


def sga_lmhead_argmax(hidden, weight_shard, shard_start, org_vocab, out_stats, workspace,
                      stream=None):
    """Fused LM-head GEMM + per-shard argmax.  hidden: bf16 [M, H] contiguous;
    weight_shard: bf16 [shard_width, H] contiguous; workspace: a CUDA tensor of
    at least sga_lmhead_argmax_workspace(M, shard_width) bytes."""
    if not (hidden.is_contiguous() and weight_shard.is_contiguous()):
        raise ValueError("hidden and weight_shard must be contiguous")
    M, H = hidden.shape
    width = weight_shard.size(0)
    if weight_shard.size(1) != H:
        raise ValueError("hidden and weight_shard must share H")
    nbytes = workspace.numel() * workspace.element_size()
    _check("sga_lmhead_argmax", lib().sga_lmhead_argmax(
        _ptr(hidden), M, H, _ptr(weight_shard), int(shard_start), width, int(org_vocab),
        _ptr(out_stats), _ptr(workspace), nbytes, _stream(stream)))
    return out_stats


def sga_lmhead_argmax_fp8(hidden_q, hidden_scale, weight_q, weight_scale, shard_start,
                          org_vocab, out_stats, workspace, stream=None):
    """Fused fp8 (E4M3) LM-head GEMM + per-shard argmax.  hidden_q: uint8 [M, H]
    codes, hidden_scale: float32 [M] CUDA tensor or None, weight_q: uint8
    [shard_width, H] codes, weight_scale: positive float (see include/sga.h)."""
    if not (hidden_q.is_contiguous() and weight_q.is_contiguous()):
        raise ValueError("hidden_q and weight_q must be contiguous")
    if hidden_q.dtype != torch.uint8 or weight_q.dtype != torch.uint8:
        raise TypeError("fp8 operands are passed as uint8 E4M3 codes")
    M, H = hidden_q.shape
    width = weight_q.size(0)
    if weight_q.size(1) != H:
        raise ValueError("hidden_q and weight_q must share H")
    nbytes = workspace.numel() * workspace.element_size()
    _check("sga_lmhead_argmax_fp8", lib().sga_lmhead_argmax_fp8(
        _ptr(hidden_q), _ptr(hidden_scale), M, H, _ptr(weight_q), float(weight_scale),
        int(shard_start), width, int(org_vocab), _ptr(out_stats), _ptr(workspace), nbytes,
        _stream(stream)))
    return out_stats


def _shard_arrays(shards):
    n = len(shards)
    return (n, (ctypes.c_int64 * n)(*[int(o) for o, _ in shards]),
            (ctypes.c_int64 * n)(*[int(w) for _, w in shards]))


def sga_lmhead_argmax_shards_workspace(M, shards):
    n, _, widths = _shard_arrays(shards)
    return int(lib().sga_lmhead_argmax_shards_workspace(int(M), n, widths))


def sga_lmhead_argmax_shards(hidden, weight, shards, org_vocab, out_stats, workspace,
                             stream=None):
    """Fused LM head + argmax of several shards of one weight buffer in one call:
    weight: bf16 [rows, H] contiguous, row 0 = global id shards[0][0]; shards =
    [(start, width), ...] ascending; out_stats receives len(shards) * M stats,
    shard-major."""
    if not (hidden.is_contiguous() and weight.is_contiguous()):
        raise ValueError("hidden and weight must be contiguous")
    M, H = hidden.shape
    if weight.size(1) != H:
        raise ValueError("hidden and weight must share H")
    n, starts, widths = _shard_arrays(shards)
    if starts[n - 1] - starts[0] + widths[n - 1] > weight.size(0):
        raise ValueError("weight does not span the shards")
    nbytes = workspace.numel() * workspace.element_size()
    _check("sga_lmhead_argmax_shards", lib().sga_lmhead_argmax_shards(
        _ptr(hidden), M, H, _ptr(weight), n, starts, widths, int(org_vocab), _ptr(out_stats),
        _ptr(workspace), nbytes, _stream(stream)))
    return out_stats


def sga_lmhead_argmax_shards_fp8(hidden_q, hidden_scale, weight_q, weight_scale, shards,
                                 org_vocab, out_stats, workspace, stream=None):
    """sga_lmhead_argmax_shards with E4M3 operands (uint8 codes) and one weight
    scale for the whole weight buffer (see include/sga.h)."""
    if not (hidden_q.is_contiguous() and weight_q.is_contiguous()):
        raise ValueError("hidden_q and weight_q must be contiguous")
    if hidden_q.dtype != torch.uint8 or weight_q.dtype != torch.uint8:
        raise TypeError("fp8 operands are passed as uint8 E4M3 codes")
    M, H = hidden_q.shape
    if weight_q.size(1) != H:
        raise ValueError("hidden_q and weight_q must share H")
    n, starts, widths = _shard_arrays(shards)
    if starts[n - 1] - starts[0] + widths[n - 1] > weight_q.size(0):
        raise ValueError("weight_q does not span the shards")
    nbytes = workspace.numel() * workspace.element_size()
    _check("sga_lmhead_argmax_shards_fp8", lib().sga_lmhead_argmax_shards_fp8(
        _ptr(hidden_q), _ptr(hidden_scale), M, H, _ptr(weight_q), float(weight_scale), n,
        starts, widths, int(org_vocab), _ptr(out_stats), _ptr(workspace), nbytes,
        _stream(stream)))
    return out_stats


def sga_device_error():
    """Synchronise the current device and return its error word."""
    w = ctypes.c_uint32(0)
    _check("sga_device_error", lib().sga_device_error(ctypes.byref(w)))
    return w.value


def sga_clear_device_error():
    _check("sga_clear_device_error", lib().sga_clear_device_error())


def sga_selftest_wait_timeout(limit_ns, waited_ns=None, stream=None):
    """Run the bounded-wait self-test kernel (see include/sga.h)."""
    _check("sga_selftest_wait_timeout", lib().sga_selftest_wait_timeout(
        int(limit_ns), _ptr(waited_ns), _stream(stream)))


def sga_lmhead_argmax_noalloc(hidden, weight_shard, shard_start, org_vocab, out_stats,
                              stream=None):
    """sga_lmhead_argmax without a workspace, for callers that cannot allocate
    device memory on their decode path (a server or plugin that owns a
    pre-sized memory pool, or a loop where cudaMalloc would synchronise the
    device).  Partial statistics go to a fixed 4 MiB scratch array inside the
    library, shared by every call on the device: calls that overlap on the
    GPU race.  Rejects sga_lmhead_argmax_workspace(M, width) > 4 MiB with
    SGA_ERR_WORKSPACE.
    The first call on a device resolves the scratch address for that device;
    make it before any stream capture."""
    fn = lib().sga_lmhead_argmax_noalloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [vp, i64, i64, vp, i64, i64, i64, vp, vp]
    fn.restype = ctypes.c_int
    if not (hidden.is_contiguous() and weight_shard.is_contiguous()):
        raise ValueError("hidden and weight_shard must be contiguous")
    M, H = hidden.shape
    if weight_shard.size(1) != H:
        raise ValueError("hidden and weight_shard must share H")
    _check("sga_lmhead_argmax_noalloc", fn(
        _ptr(hidden), M, H, _ptr(weight_shard), int(shard_start), weight_shard.size(0),
        int(org_vocab), _ptr(out_stats), _stream(stream)))
    return out_stats
