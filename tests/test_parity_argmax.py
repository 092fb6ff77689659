"""GPU parity of sga_local_argmax + sga_shard_reduce against the CPU oracle.

Bit-exact: every stat (value bits and global id) and every reduced id must
equal the oracle's.  Coverage follows the pages' test plan (vLLM PR #62604,
Test Plan: TP 1/2/3/4/8 emulated in one process with stats concatenated in
rank order; vocab 1000 / 50257 / 200064; shards narrower than a block; fp32 /
bf16; ties and planted cross-shard ties; unaligned padding; NaN rows; empty
batch; all -inf rows), plus odd row strides, per-rank buffers and row counts
that select 1..8 CTAs per row.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

import gpu_helpers as gh  # noqa: E402


def run_and_compare(x, shards, org_vocab, separate_buffers=False, x_dev=None):
    rows = x.shape[0]
    if x_dev is None:
        x_dev = gh.to_device(x)
    stats = gh.gpu_gathered_stats(x_dev, shards, org_vocab, separate_buffers)
    exp = oracle.gathered_stats(x, shards, org_vocab)
    gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)
    if len(shards) <= 64 and not separate_buffers:
        one = gh.gpu_gathered_stats_one_launch(x_dev, shards, org_vocab)
        gh.assert_stats_equal(gh.stats_to_numpy(one), exp)
    vals, ids = gh.gpu_reduce(stats, len(shards), rows)
    evals, eids = oracle.shard_reduce(exp, len(shards), rows)
    fvals, fids = oracle.full_argmax(x, org_vocab)
    assert (ids == eids).all() and (ids == fids).all()
    assert (vals.view(np.uint32) == evals.view(np.uint32)).all()
    return ids


def test_tiny_workload(sga_lib):
    c = wl.tiny_sharded_argmax()
    ids = run_and_compare(c["logits"], c["shards"], c["org_vocab"])
    assert ids[3] == 137 and ids[5] == 777 and ids[6] == 0


def test_draft_top_tokens_workload(sga_lib):
    c = wl.draft_top_tokens()
    ids = run_and_compare(c["logits"], c["shards"], c["org_vocab"])
    assert (ids < c["org_vocab"]).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vocab", [1000, 50257, 200064, 40960])
@pytest.mark.parametrize("num_shards", [1, 2, 3, 4, 8])
def test_sweep_discrete_values(sga_lib, dtype, vocab, num_shards):
    rows = 5 if vocab > 100000 else 19
    x = wl.discrete_logits(vocab + num_shards, rows, vocab, dtype, p_nan=2e-5, p_inf=1e-4)
    shards = wl.random_shards(vocab * 7 + num_shards, vocab, num_shards)
    for org in (vocab, vocab - 97):
        run_and_compare(x, shards, org)


@pytest.mark.parametrize("rows", [1, 3, 64, 700])
def test_row_counts_select_cluster_sizes(sga_lib, rows):
    x = wl.normal_matrix(rows, rows, 76032 + 13, 2.0)
    run_and_compare(x, wl.even_shards(x.shape[1], 2), x.shape[1] - 40)


def test_all_inf_nan_rows_and_all_padding_shard(sga_lib):
    x = wl.normal_matrix(9, 12, 4099, 1.0, dtype="f32")
    x[0, :] = -np.inf
    x[1, :] = np.nan
    x[2, 4000:] = np.nan          # NaN only in padding
    x[3, ::7] = np.inf            # +inf ties
    x[4, :] = 0.0
    x[4, ::2] = -0.0              # +-0 ties
    x[5, 1000:3000] = -np.inf
    x[5, 2999] = np.nan
    shards = [(0, 1000), (1000, 2000), (3000, 999), (3999, 100)]   # last shard all padding
    run_and_compare(x, shards, 3999)
    xb = wl.discrete_logits(10, 12, 4099, "bf16", p_nan=0.001, p_inf=0.01)
    xb[0, :] = wl.BF16_NEG_INF
    run_and_compare(xb, shards, 3999)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_odd_row_stride_and_misaligned_starts(sga_lib, dtype):
    vocab, pad = 30011, 5
    full = wl.discrete_logits(21, 33, vocab + pad, dtype, p_nan=1e-4)
    x_dev = gh.to_device(full)[:, :vocab]          # row stride vocab + 5
    x = np.ascontiguousarray(full[:, :vocab])
    shards = wl.random_shards(3, vocab, 3)
    run_and_compare(x, shards, vocab - 3, x_dev=x_dev)
    run_and_compare(x, shards, vocab - 3, separate_buffers=True, x_dev=x_dev)


def test_shards_narrower_than_a_vector(sga_lib):
    x = wl.discrete_logits(5, 40, 64, "bf16", p_nan=0.05)
    shards = [(i, 1) for i in range(8)] + [(8, 3), (11, 5), (16, 48)]
    run_and_compare(x, shards, 60)


def test_empty_batch(sga_lib):
    x_dev = torch.empty((0, 100), dtype=torch.bfloat16, device="cuda")
    stats = sga_lib.new_stats(0)
    sga_lib.sga_local_argmax(x_dev, 0, 100, 100, stats)
    ids = torch.empty(0, dtype=torch.int32, device="cuda")
    sga_lib.sga_shard_reduce(stats, 1, 0, ids)
    torch.cuda.synchronize()


def test_d2t_map_in_reduce(sga_lib):
    x = wl.normal_matrix(4, 50, 40960, 2.0)
    shards = wl.even_shards(40960, 2)
    rng = np.random.default_rng(0)
    d2t = np.sort(rng.choice(150000, 40960, replace=False)) - np.arange(40960)
    stats = gh.gpu_gathered_stats(gh.to_device(x), shards, 40960)
    d2t_dev = torch.from_numpy(d2t.astype(np.int64)).cuda()
    _, ids = gh.gpu_reduce(stats, 2, 50, d2t=d2t_dev)
    _, eids = oracle.shard_reduce(oracle.gathered_stats(x, shards, 40960), 2, 50)
    assert (ids == oracle.d2t_map(eids, d2t)).all()
    assert sga_lib.sga_device_error() & sga_lib.SGA_DEVERR_D2T_RANGE == 0


def test_large_verify_workload_all_rows(sga_lib):
    c = wl.large_verify()
    ids = run_and_compare(c["logits"], c["shards"], c["org_vocab"])
    for r in range(0, 4096, 100):
        assert ids[r] == c["shards"][1 + (r // 100) % 2][0] - 1


def test_one_launch_rejects_overlapping_shards(sga_lib):
    x_dev = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    stats = sga_lib.new_stats(8)
    with pytest.raises(sga_lib.SgaError):
        sga_lib.sga_local_argmax_shards(x_dev, [(0, 60), (50, 50)], 100, stats)
    with pytest.raises(sga_lib.SgaError):
        sga_lib.sga_local_argmax_shards(x_dev, [(0, 60), (60, 50)], 110, stats)


def test_one_launch_subset_of_shards_with_gap(sga_lib):
    # a GPU holding shards 1 and 3 of 4: columns are global ids minus the first start
    x = wl.discrete_logits(77, 9, 4000, "bf16", p_nan=1e-3)
    shards = wl.even_shards(4000, 4)
    held = [shards[1], shards[3]]
    x_dev = gh.to_device(x)
    one = gh.gpu_gathered_stats_one_launch(x_dev, held, 3990)
    exp = np.concatenate([oracle.shard_argmax(x, o, w, 3990) for o, w in held])
    gh.assert_stats_equal(gh.stats_to_numpy(one), exp)


def block_pieces(shards, block):
    """Intersections of the shards with global blocks [k*block, (k+1)*block)."""
    pieces = []
    for o, w in shards:
        start = o
        while start < o + w:
            end = min(o + w, (start // block + 1) * block)
            pieces.append((start, end - start))
            start = end
    return pieces


@pytest.mark.parametrize("block", [8192, 1024])
def test_block_granular_stats_on_global_boundaries(sga_lib, block):
    # per-block statistics on global block boundaries, also across shard edges
    # (vLLM PR #62604, Purpose item 1): every block stat is the oracle's, and
    # the reduce over blocks is the unsharded argmax
    c = wl.large_verify(rows_limit=160)
    x = c["logits"]
    pieces = block_pieces(c["shards"], block)
    x_dev = gh.to_device(x)
    stats = sga_lib.new_stats(len(pieces) * x.shape[0])
    for k in range(0, len(pieces), 64):
        part = pieces[k:k + 64]
        sga_lib.sga_local_argmax_shards(x_dev[:, part[0][0]:], part, c["org_vocab"],
                                        stats[k * x.shape[0]:(k + len(part)) * x.shape[0]])
    exp = oracle.gathered_stats(x, pieces, c["org_vocab"])
    gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)
    _, ids = gh.gpu_reduce(stats, len(pieces), x.shape[0])
    _, full = oracle.full_argmax(x, c["org_vocab"])
    assert (ids == full).all()
