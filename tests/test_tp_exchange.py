"""The tensor-parallel form of the path (greedy_spec_decode_gb300.tp): rank r
of a process group holds vocab shard r, computes its statistics, the ranks
all-gather them on dim 0, and every rank reduces or verifies the gathered
buffer (vLLM PR #62604, Purpose items 1-2; vLLM PR #34049, Solution).

CPU (gloo, world 2 and 3): the shard split, and that the exchange puts every
rank's statistics where the single-GPU emulation does -- each rank's local
statistics come from the oracle, and after the exchange every rank must hold
exactly the oracle's gathered statistics of the whole matrix.

GPU (gloo over the host, world 3, all ranks on cuda:0): the whole rank-local
path through libsga.so -- local argmax or fused LM head of the rank's own
shard, the exchange, verify or reduce -- on every rank, bit-exact with the
oracle (the LM head within its tolerance).  The ranks' kernels never wait on
one another: the exchange runs on the host between launches, so they can
share one GPU.  The NCCL path of gather_stats (one GPU per rank) needs more
GPUs than a test box has.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    for p in (ROOT, os.path.join(ROOT, "tests")):
        if p not in sys.path:
            sys.path.insert(0, p)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    return dist


def test_vocab_shard_split():
    from greedy_spec_decode_gb300 import tp
    for vocab in (7, 1000, 151936, 152064, 200064, 202048):
        for world in range(1, min(9, vocab + 1)):
            shards = [tp.vocab_shard(vocab, world, r) for r in range(world)]
            assert shards[0][0] == 0 and sum(w for _, w in shards) == vocab
            assert all(a[0] + a[1] == b[0] for a, b in zip(shards, shards[1:]))
            assert max(w for _, w in shards) - min(w for _, w in shards) <= 1
            assert [w for _, w in shards] == sorted((w for _, w in shards), reverse=True)
    assert tp.vocab_shard(202048, 3, 0) == (0, 67350)
    assert tp.vocab_shard(202048, 3, 2) == (134699, 67349)
    with pytest.raises(ValueError):
        tp.vocab_shard(10, 3, 3)


def _cpu_worker(rank, world, port, out_dir):
    dist = _init(rank, world, port)
    import oracle as orc
    import workloads as w
    from greedy_spec_decode_gb300 import tp
    rows, vocab, org = 37, 1003, 990
    x = w.discrete_logits(55, rows, vocab, "bf16", p_nan=0.01)
    start, width = tp.vocab_shard(vocab, world, rank)
    gathered = tp.gathered_stats_buffer(rows, device="cpu")
    gathered.fill_(-1)
    mine = orc.shard_argmax(x, start, width, org)   # x is the full matrix
    tp.local_slot(gathered, rows).copy_(torch.from_numpy(mine.view(np.int32).reshape(-1, 2)))
    tp.gather_stats(gathered, rows)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"), gathered.numpy())
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gather_puts_every_rank_in_the_shard_major_layout(tmp_path, world):
    mp.start_processes(_cpu_worker, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    from greedy_spec_decode_gb300 import tp
    rows, vocab, org = 37, 1003, 990
    x = wl.discrete_logits(55, rows, vocab, "bf16", p_nan=0.01)
    shards = [tp.vocab_shard(vocab, world, r) for r in range(world)]
    exp = oracle.gathered_stats(x, shards, org).view(np.int32).reshape(-1, 2)
    for r in range(world):
        got = np.load(tmp_path / f"rank{r}.npy")
        assert (got == exp).all(), r
    # the gathered statistics reduce to the unsharded argmax
    _, ids = oracle.shard_reduce(exp.reshape(-1).view(oracle.STAT), world, rows)
    _, full = oracle.full_argmax(x, org)
    assert (ids == full).all()


# ------------------------------------------------------------------ GPU path

LM = dict(M=40, H=256, vocab=3001)


def _gpu_worker(rank, world, port, out_dir):
    dist = _init(rank, world, port)
    torch.cuda.set_device(0)
    import workloads as w
    import greedy_spec_decode_gb300 as sga
    from greedy_spec_decode_gb300 import tp
    res = {}
    i32 = dict(dtype=torch.int32, device="cuda")
    # target side: a reduced large-verify batch (32 requests x 16 rows)
    c = w.large_verify(rows_limit=512)
    rows, vocab, k = c["logits"].shape[0], c["logits"].shape[1], c["k"]
    start, width = tp.vocab_shard(vocab, world, rank)
    x = torch.from_numpy(np.ascontiguousarray(c["logits"][:, start:start + width]).view(np.int16))
    x = x.view(torch.bfloat16).cuda()
    n = c["cu_num_draft"].size - 1
    drafts = np.load(os.path.join(out_dir, "drafts.npy"))
    mask = np.load(os.path.join(out_dir, "mask.npy"))
    gathered = tp.gathered_stats_buffer(rows)
    outs = [torch.full((n, k + 1), -9, **i32)] + [torch.full((n,), -9, **i32) for _ in range(3)]
    tids = torch.full((rows,), -9, **i32)
    tp.tp_greedy_verify(x, start, c["org_vocab"], torch.from_numpy(c["cu_num_draft"]).cuda(),
                        torch.from_numpy(drafts).cuda(), k, *outs, gathered, out_target_ids=tids,
                        in_prefill=torch.from_numpy(mask).cuda())
    res.update(verify_stats=gathered.cpu().numpy(), sampled=outs[0].cpu().numpy(),
               num_sampled=outs[1].cpu().numpy(), num_rejected=outs[2].cpu().numpy(),
               bonus=outs[3].cpu().numpy(), target_ids=tids.cpu().numpy())
    # draft side from logits: the padded draft vocabulary
    d = w.draft_top_tokens()
    dv = d["logits"].shape[1]
    s0, sw = tp.vocab_shard(dv, world, rank)
    xd = torch.from_numpy(np.ascontiguousarray(d["logits"][:, s0:s0 + sw]).view(np.int16))
    xd = xd.view(torch.bfloat16).cuda()
    g2 = tp.gathered_stats_buffer(xd.size(0))
    ids = torch.full((xd.size(0),), -9, **i32)
    tp.tp_top_tokens(xd, s0, d["org_vocab"], ids, g2)
    res.update(top_stats=g2.cpu().numpy(), top_ids=ids.cpu().numpy())
    # draft side from hidden states: the fused LM head of the rank's weight rows
    hid = w.normal_matrix(71, LM["M"], LM["H"], 1.0)
    wt = w.normal_matrix(72, LM["vocab"], LM["H"], 1.0 / np.sqrt(LM["H"]))
    l0, lw = tp.vocab_shard(LM["vocab"], world, rank)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    ws = torch.empty(sga.sga_lmhead_argmax_workspace(LM["M"], lw), dtype=torch.uint8, device="cuda")
    g3 = tp.gathered_stats_buffer(LM["M"])
    lids = torch.full((LM["M"],), -9, **i32)
    lvals = torch.full((LM["M"],), 7.0, dtype=torch.float32, device="cuda")
    tp.tp_lmhead_top_tokens(to_dev(hid), to_dev(wt[l0:l0 + lw]), l0, LM["vocab"], lids, g3, ws,
                            out_vals=lvals)
    res.update(lm_ids=lids.cpu().numpy(), lm_vals=lvals.cpu().numpy())
    res["device_error"] = np.array([sga.sga_device_error()])
    np.savez(os.path.join(out_dir, f"gpu_rank{rank}.npz"), **res)
    dist.destroy_process_group()


@pytest.mark.gpu
def test_three_ranks_on_one_gpu_match_the_oracle(sga_lib, tmp_path):
    from greedy_spec_decode_gb300 import tp
    world = 3
    c = wl.large_verify(rows_limit=512)
    x, org, k, cu = c["logits"], c["org_vocab"], c["k"], c["cu_num_draft"]
    shards = [tp.vocab_shard(x.shape[1], world, r) for r in range(world)]
    exp_stats = oracle.gathered_stats(x, shards, org)
    _, t = oracle.shard_reduce(exp_stats, world, x.shape[0])
    drafts = wl.compose_drafts(t, cu, c["flags"], c["rand_ids"])
    mask = (np.arange(cu.size - 1) % 5 == 3).astype(np.uint8)
    np.save(tmp_path / "drafts.npy", drafts)
    np.save(tmp_path / "mask.npy", mask)
    mp.start_processes(_gpu_worker, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    exp = oracle.greedy_verify(exp_stats, world, cu, drafts, k, in_prefill=mask)
    d = wl.draft_top_tokens()
    dshards = [tp.vocab_shard(d["logits"].shape[1], world, r) for r in range(world)]
    d_stats = oracle.gathered_stats(d["logits"], dshards, d["org_vocab"])
    _, d_ids = oracle.full_argmax(d["logits"], d["org_vocab"])
    hid = wl.normal_matrix(71, LM["M"], LM["H"], 1.0)
    wt = wl.normal_matrix(72, LM["vocab"], LM["H"], 1.0 / np.sqrt(LM["H"]))
    logits = oracle.lmhead_logits(hid, wt, np.arange(LM["M"]))
    top1, top2, lm_ids = oracle.argmax_f64(logits, 0, LM["vocab"])
    for r in range(world):
        got = np.load(tmp_path / f"gpu_rank{r}.npz")
        assert int(got["device_error"][0]) == 0
        assert (got["verify_stats"] == exp_stats.view(np.int32).reshape(-1, 2)).all(), r
        for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
            assert (got[key] == exp[key]).all(), (r, key)
        assert (got["top_stats"] == d_stats.view(np.int32).reshape(-1, 2)).all(), r
        assert (got["top_ids"] == d_ids).all(), r
        sure = top1 - top2 > 1e-2
        assert (got["lm_ids"][sure] == lm_ids[sure]).all(), r
        assert (np.abs(got["lm_vals"] - top1) <= np.maximum(1e-2 * np.abs(top1), 1e-3)).all(), r
