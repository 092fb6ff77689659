"""Helpers for the GPU parity tests: move seeded host inputs to the device,
run the CUDA path through the binding, and bring results back as numpy."""
import numpy as np
import torch

import greedy_spec_decode_gb300 as sga

STAT = np.dtype([("v", "<f4"), ("id", "<i4")])


def to_device(x):
    """numpy float32 or uint16 (bf16 bits) -> CUDA tensor of the same bytes."""
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def stats_to_numpy(t):
    return t.cpu().numpy().view(STAT).reshape(-1)


def gpu_gathered_stats(x_dev, shards, org_vocab, separate_buffers=False):
    """Run sga_local_argmax for every shard into one gathered buffer."""
    rows = x_dev.size(0)
    stats = sga.new_stats(len(shards) * rows)
    stats.fill_(-12345)
    for s, (o, w) in enumerate(shards):
        src = x_dev[:, o:o + w]
        if separate_buffers:
            src = src.contiguous()
        sga.sga_local_argmax(src, o, w, org_vocab, stats[s * rows:(s + 1) * rows])
    return stats


def gpu_gathered_stats_one_launch(x_dev, shards, org_vocab):
    """All shards in one sga_local_argmax_shards launch."""
    rows = x_dev.size(0)
    stats = sga.new_stats(len(shards) * rows)
    stats.fill_(-12345)
    sga.sga_local_argmax_shards(x_dev[:, shards[0][0]:], shards, org_vocab, stats)
    return stats


def gpu_reduce(stats, num_shards, rows, d2t=None):
    ids = torch.full((rows,), -777, dtype=torch.int32, device="cuda")
    vals = torch.full((rows,), 7.0, dtype=torch.float32, device="cuda")
    sga.sga_shard_reduce(stats, num_shards, rows, ids, vals, d2t=d2t)
    return vals.cpu().numpy(), ids.cpu().numpy()


def gpu_verify(stats, num_shards, cu, drafts, max_k, with_target_ids=True):
    n = len(cu) - 1
    total = int(cu[-1]) + n
    cu_d = torch.from_numpy(np.asarray(cu, np.int32)).cuda()
    dr_d = torch.from_numpy(np.asarray(drafts, np.int32)).cuda()
    out = dict(
        sampled=torch.full((n, max_k + 1), -99, dtype=torch.int32, device="cuda"),
        num_sampled=torch.full((n,), -99, dtype=torch.int32, device="cuda"),
        num_rejected=torch.full((n,), -99, dtype=torch.int32, device="cuda"),
        bonus=torch.full((n,), -99, dtype=torch.int32, device="cuda"),
        target_ids=torch.full((total,), -99, dtype=torch.int32, device="cuda"),
    )
    sga.sga_greedy_verify(stats, num_shards, cu_d, dr_d, max_k, out["sampled"],
                          out["num_sampled"], out["num_rejected"], out["bonus"],
                          out["target_ids"] if with_target_ids else None)
    return {k: v.cpu().numpy() for k, v in out.items()}


def assert_stats_equal(got, exp):
    got = np.asarray(got, STAT)
    exp = np.asarray(exp, STAT)
    assert got.shape == exp.shape
    bad = np.flatnonzero((got["id"] != exp["id"]) |
                         (got["v"].view(np.uint32) != exp["v"].view(np.uint32)))
    assert bad.size == 0, (f"{bad.size} stats differ; first at {bad[:5]}: "
                           f"got {got[bad[:5]]}, expected {exp[bad[:5]]}")
