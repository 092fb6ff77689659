"""CPU oracle for vocab-sharded greedy token selection (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``greedy_spec_decode_gb300``) never imports it, and this package never imports
the product: the two share nothing but the seeded input generators of
``workloads.py``.

The arithmetic lives in ``sga_oracle.c`` (plain loops, one function per step
of the method, each citing the page section it restates); this module only
marshals numpy arrays into it.  Sources, by page title and section:

* vLLM PR #34049 "[Spec Decode] Reduce TP communication for speculative
  decoding draft token generation", Solution: local argmax per vocab shard,
  gather of (max_value, global_index), reduce to the global argmax.
* vLLM PR #39419 "[SpecDecode] Reduce TP communication for large-vocab draft
  models speculative decoding", review thread "Refactor local argmax code":
  draft-to-target map applied after the local argmax.
* vLLM PR #62604 (sharded greedy verification), Purpose items 1 and 2 and
  Test Plan: dim-0 gathered stats, padding mask, torch.argmax order (lowest
  id on ties, NaN wins), one verify step giving accepted tokens, bonus token
  and sampled/rejected counts.

Pins (``tests/test_oracle_pins.py``, CPU only): an independent set-based brute
force, ``torch.argmax`` as a third opinion on unpadded rows, planted ties /
NaNs / -inf rows with known answers (``tests/golden/``), hand-computed
acceptance cases, shard-count invariance, a grouped brute force of the
block-granular statistics, and for the LM-head logits a numpy fp64 matmul and
exact one-hot weights.
"""
import ctypes

import numpy as np

from . import build as _build

STAT = np.dtype([("v", "<f4"), ("id", "<i4")])
F32, BF16 = 0, 1

_lib = None


def configure(L):
    """Set the ctypes signatures of a loaded oracle library; returns it."""
    i64, vp, cint = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    sig = {
        "oracle_full_argmax": ([vp, cint, i64, i64, i64, i64, vp, vp], None),
        "oracle_shard_argmax": ([vp, cint, i64, i64, i64, i64, i64, vp], None),
        "oracle_shard_reduce": ([vp, cint, i64, vp, vp], None),
        "oracle_greedy_verify": ([vp, cint, cint, vp, vp, cint, vp, vp, vp, vp, vp, vp], cint),
        "oracle_d2t_map": ([vp, i64, vp, i64, vp], cint),
        "oracle_lmhead_logits": ([vp, i64, vp, i64, vp, i64, vp], None),
        "oracle_argmax_f64": ([vp, i64, i64, i64, i64, vp, vp, vp], None),
        "oracle_e4m3_value": ([ctypes.c_uint8], ctypes.c_double),
        "oracle_lmhead_logits_fp8": ([vp, vp, i64, vp, ctypes.c_double, i64, vp, i64, vp], None),
        "oracle_block_count": ([i64, i64, i64], i64),
        "oracle_block_stats": ([vp, cint, i64, i64, i64, i64, i64, i64, i64, cint, vp, vp], i64),
        "oracle_num_threads": ([], cint),
        "oracle_set_num_threads": ([cint], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(_build.build()))
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _dtype_code(x):
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {x.dtype}")


def _row_stride(x):
    if x.ndim != 2 or (x.shape[1] > 1 and x.strides[1] != x.itemsize):
        raise ValueError("logits must be 2-D with unit stride along the vocab")
    return x.strides[0] // x.itemsize


def num_threads():
    return lib().oracle_num_threads()


def set_num_threads(n):
    lib().oracle_set_num_threads(int(n))


def full_argmax(x, org_vocab=None):
    """Argmax of every whole row with the padding mask: (vals f32, ids i32)."""
    ld = _row_stride(x)
    rows, vocab = x.shape
    org = vocab if org_vocab is None else int(org_vocab)
    vals = np.empty(rows, np.float32)
    ids = np.empty(rows, np.int32)
    if rows and vocab:
        lib().oracle_full_argmax(_ptr(x), _dtype_code(x), rows, ld, vocab, org,
                                 _ptr(vals), _ptr(ids))
    return vals, ids


def shard_argmax(x, shard_start, shard_width, org_vocab):
    """Stats of one shard.  x is the full [rows, V] matrix; the shard covers
    global ids [shard_start, shard_start + shard_width)."""
    ld = _row_stride(x)
    rows = x.shape[0]
    if shard_start < 0 or shard_width <= 0 or shard_start + shard_width > x.shape[1]:
        raise ValueError("shard outside the row")
    out = np.zeros(rows, STAT)
    if rows:
        base = x[:, shard_start:]
        lib().oracle_shard_argmax(ctypes.c_void_p(base.ctypes.data), _dtype_code(x), rows,
                                  ld, shard_start, shard_width, int(org_vocab), _ptr(out))
    return out


def gathered_stats(x, shards, org_vocab):
    """Stats of every shard concatenated in shard order (all_gather on dim 0).
    shards: list of (start, width) in ascending order."""
    if x.shape[0] == 0:
        return np.zeros(0, STAT)
    return np.concatenate([shard_argmax(x, o, w, org_vocab) for o, w in shards])


def block_count(shard_start, shard_width, block):
    """Number of fixed global blocks of `block` ids that meet the shard."""
    return int(lib().oracle_block_count(int(shard_start), int(shard_width), int(block)))


def block_slots(shard_start, shard_width, draft_block, bonus_block):
    """Stats slots per row of one shard: the larger of the two block counts."""
    return max(block_count(shard_start, shard_width, draft_block),
               block_count(shard_start, shard_width, bonus_block))


def block_stats(x, shard_start, shard_width, org_vocab, draft_block, bonus_block=None,
                cu_num_draft=None):
    """Block-granular stats of one shard: [n_pieces * rows] entries, piece-major.
    Draft rows use draft_block, the bonus row of each request (given by
    cu_num_draft; None = every row is a draft row) uses bonus_block."""
    ld = _row_stride(x)
    rows = x.shape[0]
    if shard_start < 0 or shard_width <= 0 or shard_start + shard_width > x.shape[1]:
        raise ValueError("shard outside the row")
    bonus_block = draft_block if bonus_block is None else bonus_block
    n = block_slots(shard_start, shard_width, draft_block, bonus_block)
    out = np.zeros(n * rows, STAT)
    cu = None if cu_num_draft is None else np.ascontiguousarray(cu_num_draft, np.int32)
    if rows:
        base = x[:, shard_start:]
        got = lib().oracle_block_stats(
            ctypes.c_void_p(base.ctypes.data), _dtype_code(x), rows, ld, shard_start,
            shard_width, int(org_vocab), int(draft_block), int(bonus_block),
            0 if cu is None else cu.shape[0] - 1, None if cu is None else _ptr(cu), _ptr(out))
        if got != n:
            raise ValueError(f"oracle_block_stats status {got}")
    return out


def gathered_block_stats(x, shards, org_vocab, draft_block, bonus_block=None, cu_num_draft=None):
    """Block stats of every shard concatenated in shard order; returns
    (stats, total pieces per row), ready for shard_reduce / greedy_verify
    with num_shards = total pieces."""
    parts = [block_stats(x, o, w, org_vocab, draft_block, bonus_block, cu_num_draft)
             for o, w in shards]
    rows = x.shape[0]
    total = sum(p.shape[0] for p in parts) // rows if rows else 0
    return (np.concatenate(parts) if rows else np.zeros(0, STAT)), total


def shard_reduce(stats, num_shards, rows):
    stats = np.ascontiguousarray(stats, STAT)
    if stats.shape[0] != num_shards * rows:
        raise ValueError("stats must hold num_shards * rows entries")
    vals = np.empty(rows, np.float32)
    ids = np.empty(rows, np.int32)
    if rows:
        lib().oracle_shard_reduce(_ptr(stats), num_shards, rows, _ptr(vals), _ptr(ids))
    return vals, ids


def greedy_verify(stats, num_shards, cu_num_draft, draft_tokens, max_k, in_prefill=None):
    """Greedy verification from gathered stats.  Returns a dict with
    sampled [N, max_k+1], num_sampled [N], num_rejected [N], bonus [N],
    target_ids [R_tot].  in_prefill (optional, [N], nonzero = the request is
    still in prefill) makes a request emit nothing."""
    stats = np.ascontiguousarray(stats, STAT)
    cu = np.ascontiguousarray(cu_num_draft, np.int32)
    drafts = np.ascontiguousarray(draft_tokens, np.int32)
    n = cu.shape[0] - 1
    total_rows = int(cu[-1]) + n if n > 0 else 0
    if stats.shape[0] != num_shards * total_rows:
        raise ValueError("stats must hold num_shards * (sum K + N) entries")
    out = dict(
        sampled=np.full((n, max_k + 1), -7, np.int32),
        num_sampled=np.full(n, -7, np.int32),
        num_rejected=np.full(n, -7, np.int32),
        bonus=np.full(n, -7, np.int32),
        target_ids=np.full(total_rows, -7, np.int32),
    )
    if n > 0:
        if drafts.size == 0:
            drafts = np.zeros(1, np.int32)
        mask = None
        if in_prefill is not None:
            mask = np.ascontiguousarray(np.asarray(in_prefill) != 0, np.uint8)
            if mask.shape != (n,):
                raise ValueError("in_prefill must hold one flag per request")
        st = lib().oracle_greedy_verify(
            _ptr(stats), num_shards, n, _ptr(cu), _ptr(drafts), max_k,
            None if mask is None else _ptr(mask), _ptr(out["sampled"]), _ptr(out["num_sampled"]), _ptr(out["num_rejected"]),
            _ptr(out["bonus"]), _ptr(out["target_ids"]))
        if st != 0:
            raise ValueError(f"oracle_greedy_verify status {st}")
    return out


def d2t_map(draft_ids, d2t):
    """Draft ids -> target ids, k + d2t[k]."""
    ids = np.ascontiguousarray(draft_ids, np.int32)
    table = np.ascontiguousarray(d2t, np.int64)
    out = np.empty_like(ids)
    if ids.size:
        st = lib().oracle_d2t_map(_ptr(ids), ids.size, _ptr(table), table.size, _ptr(out))
        if st != 0:
            raise ValueError("draft id outside the d2t table")
    return out


def lmhead_logits(hidden_bits, weight_bits, rows_sel):
    """fp64 logits hidden[rows_sel] . weight^T for one weight shard (bf16 bits)."""
    hidden_bits = np.ascontiguousarray(hidden_bits, np.uint16)
    weight_bits = np.ascontiguousarray(weight_bits, np.uint16)
    rows_sel = np.ascontiguousarray(rows_sel, np.int64)
    H = hidden_bits.shape[1]
    if weight_bits.shape[1] != H:
        raise ValueError("hidden and weight must share H")
    w = weight_bits.shape[0]
    out = np.empty((rows_sel.size, w), np.float64)
    if rows_sel.size and w:
        lib().oracle_lmhead_logits(_ptr(hidden_bits), H, _ptr(weight_bits), w,
                                   _ptr(rows_sel), rows_sel.size, _ptr(out))
    return out


def argmax_f64(logits, first, org_vocab):
    """(top1, top2, ids) of fp64 logits rows whose column j is global id first+j."""
    logits = np.ascontiguousarray(logits, np.float64)
    n, w = logits.shape
    top1 = np.empty(n, np.float64)
    top2 = np.empty(n, np.float64)
    ids = np.empty(n, np.int32)
    if n and w:
        lib().oracle_argmax_f64(_ptr(logits), n, w, int(first), int(org_vocab),
                                _ptr(top1), _ptr(top2), _ptr(ids))
    return top1, top2, ids


def lmhead_argmax(hidden_bits, weight_bits, rows_sel, shard_start, org_vocab):
    """Per selected row: (top1, top2, id) of one shard's fp64 logits."""
    logits = lmhead_logits(hidden_bits, weight_bits, rows_sel)
    return argmax_f64(logits, shard_start, org_vocab)


def e4m3_value(code):
    """Exact value of one FP8 E4M3 code (uint8)."""
    return lib().oracle_e4m3_value(int(code))


def lmhead_logits_fp8(hidden_q, hidden_scale, weight_q, weight_scale, rows_sel):
    """fp64 logits of the fp8 LM head for the selected rows: E4M3 codes
    (uint8) of hidden [M, H] and of one weight shard [w, H], a positive fp32
    scale per hidden row and one positive weight scale."""
    hidden_q = np.ascontiguousarray(hidden_q, np.uint8)
    weight_q = np.ascontiguousarray(weight_q, np.uint8)
    scale = np.ascontiguousarray(hidden_scale, np.float32)
    rows_sel = np.ascontiguousarray(rows_sel, np.int64)
    H = hidden_q.shape[1]
    if weight_q.shape[1] != H:
        raise ValueError("hidden and weight must share H")
    w = weight_q.shape[0]
    out = np.empty((rows_sel.size, w), np.float64)
    if rows_sel.size and w:
        lib().oracle_lmhead_logits_fp8(_ptr(hidden_q), _ptr(scale), H, _ptr(weight_q),
                                       float(weight_scale), w, _ptr(rows_sel), rows_sel.size,
                                       _ptr(out))
    return out
