"""Randomised parity sweep (fixed seeds) of the one-launch shard argmax, the
reduce and the fused verify, of block-granular statistics (both entry points)
feeding the verify, and of the fused LM head (bf16 and fp8), against the
oracle.

Every case draws its own shape: rows, vocabulary, number and widths of shards,
dtype, row-stride padding, org_vocab (padding), value distribution (normal or
tie-heavy with +-inf, NaN, +-0), requests with 0..max_k drafts and
placeholder drafts.  Bit-exact for the argmax and verify outputs; the LM head
within the tolerance of tests/test_parity_lmhead.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh
import test_parity_lmhead as lm

pytestmark = pytest.mark.gpu


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    vocab = int(rng.choice([7, 64, 513, 4097, 32000, 50257, 99991]))
    num_shards = int(rng.integers(1, min(8, vocab) + 1))
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    max_k = int(rng.choice([1, 3, 5, 15]))
    n = int(rng.integers(1, 40))
    ks = rng.integers(0, max_k + 1, n)
    pad = int(rng.integers(0, 9))
    org = int(vocab if rng.random() < 0.5 else rng.integers(1, vocab + 1))
    tie_heavy = rng.random() < 0.5
    return rng, vocab, num_shards, dtype, max_k, ks, pad, org, tie_heavy


@pytest.mark.parametrize("seed", range(24))
def test_random_argmax_reduce_verify(sga_lib, seed):
    rng, vocab, num_shards, dtype, max_k, ks, pad, org, tie_heavy = draw_case(seed)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    rows = int(cu[-1]) + len(ks)
    width = vocab + pad
    if tie_heavy:
        full = wl.discrete_logits(seed, rows, width, dtype, p_nan=0.003, p_inf=0.01)
    else:
        full = wl.normal_matrix(seed, rows, width, 3.0, dtype=dtype)
    x = np.ascontiguousarray(full[:, :vocab])
    x_dev = gh.to_device(full)[:, :vocab]                 # row stride vocab + pad
    shards = wl.random_shards(seed, vocab, num_shards)

    stats = gh.gpu_gathered_stats_one_launch(x_dev, shards, org)
    exp = oracle.gathered_stats(x, shards, org)
    gh.assert_stats_equal(gh.stats_to_numpy(stats), exp)

    _, t = oracle.shard_reduce(exp, num_shards, rows)
    _, full_ids = oracle.full_argmax(x, org)
    assert (t == full_ids).all()
    _, ids = gh.gpu_reduce(stats, num_shards, rows)
    assert (ids == t).all()

    flags = rng.random(int(cu[-1])) < 0.7
    rand = rng.integers(-1, vocab, int(cu[-1])).astype(np.int32)
    drafts = wl.compose_drafts(t, cu, flags, rand)
    got = gh.gpu_verify(stats, num_shards, cu, drafts, max_k)
    ref = oracle.greedy_verify(exp, num_shards, cu, drafts, max_k)
    for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
        assert (got[key] == ref[key]).all(), key


@pytest.mark.parametrize("seed", range(6))
def test_random_lmhead(sga_lib, seed):
    rng = np.random.default_rng(2000 + seed)
    M = int(rng.choice([1, 7, 128, 129, 255, 256, 300, 640]))
    H = int(64 * rng.integers(1, 9))
    vocab = int(rng.integers(1, 3000))
    num_shards = int(rng.integers(1, min(4, vocab) + 1))
    org = int(vocab if rng.random() < 0.5 else rng.integers(1, vocab + 1))
    hidden = wl.normal_matrix(seed, M, H, 1.0)
    weight = wl.normal_matrix(seed + 77, vocab, H, 1.0 / np.sqrt(H))
    shards = wl.random_shards(seed, vocab, num_shards)
    st, v, i = lm.run_gpu(hidden, weight, shards, org)
    rows = np.arange(M) if M <= 300 else np.arange(0, M, 3)
    lm.check_rows(rows, hidden, weight, shards, org, st, v, i)


@pytest.mark.parametrize("seed", range(16))
def test_random_block_stats(sga_lib, seed):
    # block-granular statistics with random vocab, shards, block sizes (nested
    # or not), request layouts with 0..K drafts, padding and row strides; both
    # entry points (per shard and one launch), then the wide or narrow verify
    import test_parity_blocks as tb
    rng = np.random.default_rng(3000 + seed)
    vocab = int(rng.choice([97, 1000, 4099, 20000, 50257]))
    num_shards = int(rng.integers(1, min(6, vocab) + 1))
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    n = int(rng.integers(1, 20))
    max_k = int(rng.choice([1, 3, 7, 15]))
    ks = rng.integers(0, max_k + 1, n)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    rows = int(cu[-1]) + n
    db = int(rng.choice([1, 7, 64, 1024, 8192]))
    bb = int(rng.choice([1, 16, 1024, 3000]))
    if vocab // min(db, bb) * num_shards > 3000:   # keep the slots under the verify's limit
        db, bb = max(db, 64), max(bb, 64)
    pad = int(rng.integers(0, 5))
    org = int(vocab if rng.random() < 0.5 else rng.integers(1, vocab + 1))
    full = wl.discrete_logits(seed + 50, rows, vocab + pad, dtype, p_nan=0.002, p_inf=0.01)
    x = np.ascontiguousarray(full[:, :vocab])
    x_dev = gh.to_device(full)[:, :vocab]
    shards = wl.random_shards(seed, vocab, num_shards)
    exp, n_exp = oracle.gathered_block_stats(x, shards, org, db, bb, cu)
    per, n_per = tb.gpu_block_stats(x_dev, shards, org, db, bb, cu)
    one, n_one = tb.gpu_block_stats_one_launch(x_dev, shards, org, db, bb, cu)
    assert n_per == n_one == n_exp
    gh.assert_stats_equal(gh.stats_to_numpy(per), exp)
    gh.assert_stats_equal(gh.stats_to_numpy(one), exp)
    _, t = oracle.shard_reduce(oracle.gathered_stats(x, shards, org), num_shards, rows)
    drafts = wl.compose_drafts(t, cu, rng.random(int(cu[-1])) < 0.7,
                               rng.integers(-1, vocab, int(cu[-1])).astype(np.int32))
    got = gh.gpu_verify(one, n_exp, cu, drafts, max_k)
    ref = oracle.greedy_verify(exp, n_exp, cu, drafts, max_k)
    for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
        assert (got[key] == ref[key]).all(), key
    assert (ref["target_ids"] == t).all()


@pytest.mark.parametrize("seed", range(6))
def test_random_lmhead_fp8(sga_lib, seed):
    import test_parity_lmhead_fp8 as f8
    rng = np.random.default_rng(4000 + seed)
    M = int(rng.choice([1, 5, 16, 33, 64, 100, 129, 300]))
    H = int(128 * rng.integers(1, 5))
    vocab = int(rng.integers(1, 3000))
    num_shards = int(rng.integers(1, min(4, vocab) + 1))
    org = int(vocab if rng.random() < 0.5 else rng.integers(1, vocab + 1))
    hq, hs, wq, w_scale = f8.make(M, H, vocab, 4000 + seed)
    shards = wl.random_shards(seed, vocab, num_shards)
    st, v, i = f8.run_gpu(sga_lib, hq, hs, wq, w_scale, shards, org)
    rows = np.arange(M) if M <= 130 else np.arange(0, M, 3)
    f8.check(rows, hq, hs, wq, w_scale, shards, org, st, v, i)
