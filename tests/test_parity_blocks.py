"""GPU parity of sga_local_argmax_blocks: block-granular shard statistics on
fixed global block boundaries (vLLM PR #62604, Purpose item 1: per-block
(max, token id) statistics, 8192 ids for draft positions and 1024 for the
bonus position, boundaries kept across shard edges), bit-exact against the
oracle; and the gathered block statistics through the reduce and the fused
verify, which must give exactly what per-shard statistics give.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh
import greedy_spec_decode_gb300 as sga

pytestmark = pytest.mark.gpu


def gpu_block_stats(x_dev, shards, org, draft_block, bonus_block, cu_np):
    """Every shard's block stats into one gathered buffer; returns (stats,
    slots per row)."""
    rows = x_dev.size(0)
    slots = [sga.sga_block_slots(o, w, draft_block, bonus_block) for o, w in shards]
    stats = sga.new_stats(sum(slots) * rows)
    stats.fill_(-12345)
    cu_d = None if cu_np is None else torch.from_numpy(np.asarray(cu_np, np.int32)).cuda()
    off = 0
    for (o, w), n in zip(shards, slots):
        sga.sga_local_argmax_blocks(x_dev[:, o:o + w], o, w, org, draft_block,
                                    stats[off * rows:(off + n) * rows], bonus_block=bonus_block,
                                    cu_num_draft=cu_d)
        off += n
    return stats, sum(slots)


def gpu_block_stats_one_launch(x_dev, shards, org, draft_block, bonus_block, cu_np):
    """All shards' block stats with one sga_local_argmax_blocks_shards launch."""
    rows = x_dev.size(0)
    n = sum(sga.sga_block_slots(o, w, draft_block, bonus_block) for o, w in shards)
    stats = sga.new_stats(n * rows)
    stats.fill_(-12345)
    cu_d = None if cu_np is None else torch.from_numpy(np.asarray(cu_np, np.int32)).cuda()
    sga.sga_local_argmax_blocks_shards(x_dev[:, shards[0][0]:], shards, org, draft_block, stats,
                                       bonus_block=bonus_block, cu_num_draft=cu_d)
    return stats, n


def random_layout(rng, max_k, n):
    ks = rng.integers(0, max_k + 1, n)
    return np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("vocab,num_shards,blocks", [
    (700, 3, (64, 16)), (700, 3, (16, 64)), (5000, 2, (1024, 256)), (1000, 4, (24, 7)),
    (333, 2, (1, 1)), (20000, 3, (8192, 1024)), (4097, 5, (1 << 20, 8)),
])
def test_block_stats_bit_exact(sga_lib, dtype, vocab, num_shards, blocks):
    rng = np.random.default_rng(vocab + num_shards)
    cu = random_layout(rng, 5, 9)
    rows = int(cu[-1]) + 9
    pad = 3                                              # row stride vocab + 3 elements
    full = wl.discrete_logits(vocab * 7 + num_shards, rows, vocab + pad, dtype,
                              p_nan=0.003, p_inf=0.01)
    x = np.ascontiguousarray(full[:, :vocab])
    x_dev = gh.to_device(full)[:, :vocab]
    shards = wl.random_shards(vocab, vocab, num_shards)
    db, bb = blocks
    for org in (vocab, vocab - 13):
        for use_cu in (True, False):
            c = cu if use_cu else None
            stats, n = gpu_block_stats(x_dev, shards, org, db, bb, c)
            exp, n_exp = oracle.gathered_block_stats(x, shards, org, db, bb, c)
            assert n == n_exp
            gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)
            one, n_one = gpu_block_stats_one_launch(x_dev, shards, org, db, bb, c)
            assert n_one == n_exp
            gh.assert_stats_equal(gh.stats_to_numpy(one), exp)
            _, ids = gh.gpu_reduce(stats, n, rows)
            assert (ids == oracle.full_argmax(x, org)[1]).all()


def test_all_padding_pieces_inf_and_nan_rows(sga_lib):
    vocab = 3000
    x = wl.normal_matrix(8, 6, vocab, 2.0)
    x[0, :] = wl.BF16_NEG_INF                           # all -inf row
    x[1, 1500] = wl.BF16_NAN                            # NaN in the middle
    x[1, 2990] = wl.BF16_NAN                            # ... and in padding
    x[2, 2995] = wl.bf16_const(np.inf)                  # +inf only in padding
    x[3, 1023:1025] = wl.bf16_const(50.0)               # tie across a 1024-block edge
    shards = [(0, 1100), (1100, 1900)]
    x_dev = gh.to_device(x)
    for org in (2900, 2040):                            # 2040: block [2048, 3000) all padding
        stats, n = gpu_block_stats(x_dev, shards, org, 1024, 1024, None)
        exp, _ = oracle.gathered_block_stats(x, shards, org, 1024)
        gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)
        _, ids = gh.gpu_reduce(stats, n, 6)
        assert ids[0] == 0 and ids[1] == 1500 and ids[3] == 1023
        assert ids[2] == oracle.full_argmax(x, org)[1][2]


def test_requests_without_drafts_and_single_row(sga_lib):
    x = wl.discrete_logits(9, 5, 2100, "bf16")
    cu = np.array([0, 0, 2, 2], np.int32)                # K = 0, 2, 0: rows 0, 1-3, 4
    shards = wl.even_shards(2100, 2)
    stats, n = gpu_block_stats(gh.to_device(x), shards, 2100, 512, 64, cu)
    exp, _ = oracle.gathered_block_stats(x, shards, 2100, 512, 64, cu)
    gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)
    one = x[:1]
    stats, n = gpu_block_stats(gh.to_device(one), shards, 2100, 512, 64, np.array([0, 0], np.int32))
    exp, _ = oracle.gathered_block_stats(one, shards, 2100, 512, 64, np.array([0, 0], np.int32))
    gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)


def test_empty_batch(sga_lib):
    x_dev = torch.empty((0, 100), dtype=torch.bfloat16, device="cuda")
    stats = sga.new_stats(1)
    stats.fill_(-3)
    sga.sga_local_argmax_blocks(x_dev, 0, 100, 100, 16, stats)
    torch.cuda.synchronize()
    assert (stats.cpu() == -3).all()


def test_verify_sample_block_stats_match_shard_stats(sga_lib):
    # the verify-size workload (24 requests x (3 + 1) rows x 200064 bf16, 4
    # shards) with the pages' block sizes: the verify outputs from the
    # gathered block stats equal the oracle's from per-shard stats
    c = wl.greedy_verify_small()
    x, shards, org, cu = c["logits"], c["shards"], c["org_vocab"], c["cu_num_draft"]
    stats, n = gpu_block_stats(gh.to_device(x), shards, org, 8192, 1024, cu)
    exp, _ = oracle.gathered_block_stats(x, shards, org, 8192, 1024, cu)
    gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)
    shard_stats = oracle.gathered_stats(x, shards, org)
    _, t = oracle.shard_reduce(shard_stats, len(shards), x.shape[0])
    drafts = wl.compose_drafts(t, cu, c["flags"], c["rand_ids"])
    got = gh.gpu_verify(stats, n, cu, drafts, c["k"])
    ref = oracle.greedy_verify(shard_stats, len(shards), cu, drafts, c["k"])
    for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
        assert (got[key] == ref[key]).all(), key


def test_large_verify_full_size_block_stats(sga_lib):
    # 4096 rows x 202048 bf16, 3 uneven shards, blocks 8192 / 1024: every
    # stat of every row against the oracle (per-shard launches and the
    # one-launch form), and the verify from the block stats against the
    # oracle's verify from per-shard stats
    c = wl.large_verify()
    x, shards, org, cu = c["logits"], c["shards"], c["org_vocab"], c["cu_num_draft"]
    rows = x.shape[0]
    stats, n = gpu_block_stats(gh.to_device(x), shards, org, 8192, 1024, cu)
    slots = [oracle.block_slots(o, w, 8192, 1024) for o, w in shards]
    exp_all, _ = oracle.gathered_block_stats(x, shards, org, 8192, 1024, cu)   # every row
    gh.assert_stats_equal(gh.stats_to_numpy(stats), exp_all)
    one, _ = gpu_block_stats_one_launch(gh.to_device(x), shards, org, 8192, 1024, cu)
    gh.assert_stats_equal(gh.stats_to_numpy(one), exp_all)
    shard_stats = oracle.gathered_stats(x, shards, org)
    _, t = oracle.shard_reduce(shard_stats, 3, rows)
    drafts = wl.compose_drafts(t, cu, c["flags"], c["rand_ids"])
    got = gh.gpu_verify(stats, n, cu, drafts, c["k"])
    ref = oracle.greedy_verify(shard_stats, 3, cu, drafts, c["k"])
    for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
        assert (got[key] == ref[key]).all(), key
    assert n == sum(slots) == 66 + 67 + 67
    for r in range(0, rows, 100):                       # planted cross-edge ties
        assert got["target_ids"][r] == shards[1 + (r // 100) % 2][0] - 1
    assert sga_lib.sga_device_error() == 0


def test_request_layout_past_the_rows_sets_error_word(sga_lib):
    # cu_num_draft names 3 + 6 drafts (11 rows) but the logits hold 5 rows:
    # request 1 is skipped and flagged, request 0 (rows 0..3) is still right
    sga_lib.sga_clear_device_error()
    x = wl.discrete_logits(12, 5, 900, "bf16")
    cu = np.array([0, 3, 9], np.int32)
    stats = sga.new_stats(sga.sga_block_slots(0, 900, 256, 64) * 5)
    stats.fill_(-12345)
    sga.sga_local_argmax_blocks(gh.to_device(x), 0, 900, 900, 256, stats, bonus_block=64,
                                cu_num_draft=torch.from_numpy(cu).cuda())
    assert sga_lib.sga_device_error() & sga_lib.SGA_DEVERR_LAYOUT
    n = sga.sga_block_slots(0, 900, 256, 64)
    got = gh.stats_to_numpy(stats).reshape(n, 5)[:, :4].reshape(-1)
    exp = oracle.block_stats(x[:4], 0, 900, 900, 256, 64, np.array([0, 3], np.int32))
    gh.assert_stats_equal(got, exp)
    sga_lib.sga_clear_device_error()
    assert sga_lib.sga_device_error() == 0


@pytest.mark.parametrize("layout", ["uniform_0_15", "skewed", "all_zero"])
def test_many_requests_variable_k(sga_lib, layout):
    # 256 requests: the flat piece numbering of the one-launch kernel spans
    # many requests per CTA and many CTAs per request; every request's rows,
    # its bonus row's block size and the empty slots must land where the
    # oracle puts them (per-shard launches and the one launch alike)
    rng = np.random.default_rng(91)
    if layout == "uniform_0_15":
        ks = rng.integers(0, 16, 256)
    elif layout == "skewed":
        ks = np.concatenate([np.full(40, 15), np.zeros(216, np.int64)])
        rng.shuffle(ks)
    else:
        ks = np.zeros(256, np.int64)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    rows = int(cu[-1]) + 256
    vocab, org = 6000, 5990
    x = wl.discrete_logits(92, rows, vocab, "bf16", p_nan=0.001, p_inf=0.01)
    x_dev = gh.to_device(x)
    shards = [(0, 2001), (2001, 1999), (4000, 2000)]
    exp, n_exp = oracle.gathered_block_stats(x, shards, org, 512, 128, cu)
    one, n_one = gpu_block_stats_one_launch(x_dev, shards, org, 512, 128, cu)
    per, n_per = gpu_block_stats(x_dev, shards, org, 512, 128, cu)
    assert n_one == n_per == n_exp
    gh.assert_stats_equal(gh.stats_to_numpy(one), exp)
    gh.assert_stats_equal(gh.stats_to_numpy(per), exp)
    assert sga_lib.sga_device_error() == 0


def test_decreasing_request_layout_sets_error_word(sga_lib):
    # request 1 ends before it starts (cu 5 -> 3): the launch flags the
    # layout and stays inside the buffers; the error word clears again
    sga_lib.sga_clear_device_error()
    x = wl.discrete_logits(13, 12, 900, "f32")
    cu = np.array([0, 5, 3, 8], np.int32)
    for n_shards in (1, 2):
        shards = [(0, 900)] if n_shards == 1 else [(0, 300), (300, 600)]
        n = sum(sga.sga_block_slots(o, w, 256, 64) for o, w in shards)
        stats = sga.new_stats(n * 12)
        sga.sga_local_argmax_blocks_shards(gh.to_device(x), shards, 900, 256, stats,
                                           bonus_block=64, cu_num_draft=torch.from_numpy(cu).cuda())
        assert sga_lib.sga_device_error() & sga_lib.SGA_DEVERR_LAYOUT
        sga_lib.sga_clear_device_error()
    assert sga_lib.sga_device_error() == 0


def test_one_launch_large_verify_and_subset_of_shards(sga_lib):
    # the large-verify shards in one launch (sampled requests against the
    # oracle, the verify against per-shard launches), and a GPU holding shards
    # 1 and 3 of 4 (a gap between them)
    c = wl.large_verify(rows_limit=640)
    x, shards, org, cu = c["logits"], c["shards"], c["org_vocab"], c["cu_num_draft"]
    x_dev = gh.to_device(x)
    one, n = gpu_block_stats_one_launch(x_dev, shards, org, 8192, 1024, cu)
    per, n_per = gpu_block_stats(x_dev, shards, org, 8192, 1024, cu)
    assert n == n_per == 200
    gh.assert_stats_equal(gh.stats_to_numpy(one), gh.stats_to_numpy(per))
    exp, _ = oracle.gathered_block_stats(x[:16], shards, org, 8192, 1024, cu[:2] - cu[0])
    gh.assert_stats_equal(gh.stats_to_numpy(one).reshape(n, -1)[:, :16].reshape(-1), exp)
    y = wl.discrete_logits(77, 9, 4000, "bf16", p_nan=1e-3)
    quarters = wl.even_shards(4000, 4)
    held = [quarters[1], quarters[3]]
    got, m = gpu_block_stats_one_launch(gh.to_device(y), held, 3990, 256, 64, None)
    exp, m_exp = oracle.gathered_block_stats(y, held, 3990, 256, 64)
    assert m == m_exp
    gh.assert_stats_equal(gh.stats_to_numpy(got), exp)
