"""Tensor-parallel form of the path: one process per GPU, rank r of a
torch.distributed group holds vocab shard r.

vLLM PR #62604, Purpose item 1: each rank reduces its own vocab shard to
per-row (max, token id) statistics, only those are all-gathered on dim 0, and
one kernel on every rank turns the gathered statistics into the accepted
tokens, the bonus token and the counts; item 2: the draft side's fused
get_top_tokens gathers (max, id) pairs the same way and reduces them.  vLLM
PR #34049, Solution: local argmax, gather of (value, global index), reduce.

Every compute step runs in libsga.so's kernels (sga_local_argmax or the fused
LM head, then sga_greedy_verify_prefill or sga_shard_reduce) on the caller's
current stream; this module only places each rank's statistics in the
gathered buffer and runs the exchange:
  - NCCL (one GPU per rank): an in-place all_gather_into_tensor of the rows x
    8-byte statistics; the collective is ordered after the local kernel and
    before the verify on the current stream.
  - any other backend (gloo): the statistics go through host memory.
The gathered buffer is [world * rows] statistics, rank r's at rows
[r * rows, (r + 1) * rows): byte for byte the single-GPU emulation's
shard-major layout, so every rank's verify sees exactly what one GPU holding
all shards would.
"""
import torch
import torch.distributed as dist

from . import (new_stats, sga_greedy_verify_prefill, sga_lmhead_argmax, sga_local_argmax,
               sga_shard_reduce)


def vocab_shard(vocab, world, rank):
    """(first id, width) of rank's shard of a vocab split over world ranks:
    contiguous ascending shards, the first vocab % world one id wider (the
    uneven split of a vocab-parallel head)."""
    if world < 1 or not 0 <= rank < world or vocab < world:
        raise ValueError("need 0 <= rank < world <= vocab")
    base, extra = divmod(int(vocab), int(world))
    return rank * base + min(rank, extra), base + (1 if rank < extra else 0)


def _group_info(group):
    if not (dist.is_available() and dist.is_initialized()):
        return 0, 1, None
    return dist.get_rank(group), dist.get_world_size(group), dist.get_backend(group)


def gathered_stats_buffer(rows, group=None, device="cuda"):
    """A [world * rows] statistics buffer for the exchange."""
    _, world, _ = _group_info(group)
    return new_stats(world * rows, device=device)


def local_slot(gathered, rows, group=None):
    """This rank's rows of the gathered buffer: where its local kernel writes."""
    rank, _, _ = _group_info(group)
    return gathered[rank * rows:(rank + 1) * rows]


def gather_stats(gathered, rows, group=None):
    """All-gather on dim 0, in place: every rank has written its rows x 8-byte
    statistics to local_slot(gathered, rows); afterwards every rank holds
    all ranks' statistics in rank order.  A group of one rank (or no group)
    exchanges nothing."""
    rank, world, backend = _group_info(group)
    if world == 1:
        return gathered
    out = gathered[:world * rows]
    local = out[rank * rows:(rank + 1) * rows]
    if backend == "nccl":
        dist.all_gather_into_tensor(out, local, group=group)
    else:
        host = local.cpu()
        parts = [torch.empty_like(host) for _ in range(world)]
        dist.all_gather(parts, host, group=group)
        out.copy_(torch.cat(parts))
    return gathered


def tp_greedy_verify(logits_shard, shard_start, org_vocab, cu_num_draft, draft_tokens, max_k,
                     out_sampled, out_num_sampled, out_num_rejected, out_bonus, gathered,
                     out_target_ids=None, in_prefill=None, group=None):
    """Target side on one rank: the local argmax of this rank's shard
    (logits_shard: [rows, shard_width] CUDA tensor whose column 0 is global id
    shard_start), the dim-0 exchange, and the fused verify over every rank's
    statistics.  Every rank gets the same outputs."""
    rows = logits_shard.size(0)
    _, world, _ = _group_info(group)
    sga_local_argmax(logits_shard, shard_start, logits_shard.size(1), org_vocab,
                     local_slot(gathered, rows, group))
    gather_stats(gathered, rows, group)
    sga_greedy_verify_prefill(gathered[:world * rows], world, cu_num_draft, draft_tokens,
                              in_prefill, max_k, out_sampled, out_num_sampled, out_num_rejected,
                              out_bonus, out_target_ids)


def tp_top_tokens(logits_shard, shard_start, org_vocab, out_ids, gathered, out_vals=None,
                  d2t=None, group=None):
    """Draft side on one rank (get_top_tokens from logits): local argmax,
    dim-0 exchange, cross-shard reduce (optionally mapped draft -> target
    ids with d2t)."""
    rows = logits_shard.size(0)
    _, world, _ = _group_info(group)
    sga_local_argmax(logits_shard, shard_start, logits_shard.size(1), org_vocab,
                     local_slot(gathered, rows, group))
    gather_stats(gathered, rows, group)
    sga_shard_reduce(gathered[:world * rows], world, rows, out_ids, out_vals, d2t=d2t)


def tp_lmhead_top_tokens(hidden, weight_shard, shard_start, org_vocab, out_ids, gathered,
                         workspace, out_vals=None, d2t=None, group=None):
    """Draft side on one rank from hidden states: the fused LM head + argmax
    of this rank's weight shard (the logits never leave the tensor cores),
    dim-0 exchange, cross-shard reduce."""
    rows = hidden.size(0)
    _, world, _ = _group_info(group)
    sga_lmhead_argmax(hidden, weight_shard, shard_start, org_vocab,
                      local_slot(gathered, rows, group), workspace)
    gather_stats(gathered, rows, group)
    sga_shard_reduce(gathered[:world * rows], world, rows, out_ids, out_vals, d2t=d2t)
