"""The hot path inside a CUDA graph.

Serving engines replay decode steps from captured CUDA graphs (the pages'
benchmarks run vLLM with full CUDA graphs, vLLM PR #34049 Test Plan).  The
entry points enqueue kernels only (no synchronisation, no allocation), so a
step can be captured once and replayed on new inputs copied into the same
buffers.  These tests capture (a) the one-launch shard argmax + fused verify
and (b) the fused LM-head argmax of two shards + shard reduce (at a GEMM size
and at both decode sizes), replay them on fresh inputs and check parity with
the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def test_captured_verify_step_replays_on_new_inputs(sga_lib):
    n, k, vocab = 40, 5, 50257
    shards = wl.even_shards(vocab, 3)
    rows = n * (k + 1)
    x_dev = torch.empty((rows, vocab), dtype=torch.bfloat16, device="cuda")
    stats = sga_lib.new_stats(3 * rows)
    cu = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    drafts = torch.empty(n * k, dtype=torch.int32, device="cuda")
    out = dict(sampled=torch.empty((n, k + 1), dtype=torch.int32, device="cuda"),
               ns=torch.empty(n, dtype=torch.int32, device="cuda"),
               nr=torch.empty(n, dtype=torch.int32, device="cuda"),
               bonus=torch.empty(n, dtype=torch.int32, device="cuda"))

    def step():
        sga_lib.sga_local_argmax_shards(x_dev, shards, vocab, stats)
        sga_lib.sga_greedy_verify(stats, 3, cu, drafts, k, out["sampled"], out["ns"],
                                  out["nr"], out["bonus"])

    cu_np, flags, rand = wl.draft_plan(9, n, k, 0.7, vocab)
    cu.copy_(torch.from_numpy(cu_np))
    x_dev.copy_(gh.to_device(wl.normal_matrix(1, rows, vocab, 3.0)))
    drafts.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                   # warm up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (11, 12):
        x = wl.normal_matrix(seed, rows, vocab, 3.0)
        st = oracle.gathered_stats(x, shards, vocab)
        _, t = oracle.shard_reduce(st, 3, rows)
        d = wl.compose_drafts(t, cu_np, flags, rand)
        x_dev.copy_(gh.to_device(x))
        drafts.copy_(torch.from_numpy(d))
        graph.replay()
        torch.cuda.synchronize()
        exp = oracle.greedy_verify(st, 3, cu_np, d, k)
        assert (out["sampled"].cpu().numpy() == exp["sampled"]).all()
        assert (out["ns"].cpu().numpy() == exp["num_sampled"]).all()
        assert (out["nr"].cpu().numpy() == exp["num_rejected"]).all()
        assert (out["bonus"].cpu().numpy() == exp["bonus"]).all()
        gh.assert_stats_equal(gh.stats_to_numpy(stats), st)
    assert sga_lib.sga_device_error() == 0


@pytest.mark.parametrize("M", [300, 100, 16])   # 2-SM GEMM, CTA-pair and one-CTA decode kernels
def test_captured_lmhead_step_replays_on_new_inputs(sga_lib, M):
    H, vocab = 512, 6000
    shards = wl.even_shards(vocab, 2)
    w_np = wl.normal_matrix(3, vocab, H, 1.0 / np.sqrt(H))
    w = gh.to_device(w_np)
    h = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    stats = sga_lib.new_stats(2 * M)
    ws = torch.empty(max(sga_lib.sga_lmhead_argmax_workspace(M, wd) for _, wd in shards),
                     dtype=torch.uint8, device="cuda")
    ids = torch.empty(M, dtype=torch.int32, device="cuda")
    views = [w[o:o + wd] for o, wd in shards]

    def step():
        for s, (o, wd) in enumerate(shards):
            sga_lib.sga_lmhead_argmax(h, views[s], o, vocab, stats[s * M:(s + 1) * M], ws)
        sga_lib.sga_shard_reduce(stats, 2, M, ids)

    h.copy_(gh.to_device(wl.normal_matrix(4, M, H, 1.0)))
    step()                                       # first call resolves per-device facts
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (21, 22):
        h_np = wl.normal_matrix(seed, M, H, 1.0)
        h.copy_(gh.to_device(h_np))
        graph.replay()
        torch.cuda.synchronize()
        rows = np.arange(0, M, 7)
        logits = oracle.lmhead_logits(h_np, w_np, rows)
        top1, top2, exp_ids = oracle.argmax_f64(logits, 0, vocab)
        got = ids.cpu().numpy()[rows]
        sure = top1 - top2 > 1e-2
        assert (got[sure] == exp_ids[sure]).all()
    assert sga_lib.sga_device_error() == 0
