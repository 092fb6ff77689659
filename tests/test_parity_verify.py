"""GPU parity of sga_greedy_verify (fused cross-shard reduce + greedy
acceptance) against the CPU oracle: accepted tokens, bonus token,
num_sampled / num_rejected and per-row target ids, all bit-exact.

Coverage follows vLLM PR #62604, Test Plan: TP 2/3/4/8 emulated in one
process, compared with the full-logits result; K = 1/3/5 (and 15);
placeholder drafts; planted cross-shard ties; plus variable K per request,
requests with no drafts, max_k larger than every K, and the error word for a
request whose K exceeds max_k.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def check_verify(stats_dev, stats_np, num_shards, cu, drafts, max_k):
    got = gh.gpu_verify(stats_dev, num_shards, cu, drafts, max_k)
    exp = oracle.greedy_verify(stats_np, num_shards, cu, drafts, max_k)
    for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
        assert (got[key] == exp[key]).all(), key
    ns, nr = got["num_sampled"], got["num_rejected"]
    assert (ns + nr == np.diff(cu) + 1).all()
    return got


def run_workload(c):
    x = c["logits"]
    x_dev = gh.to_device(x)
    stats_dev = gh.gpu_gathered_stats(x_dev, c["shards"], c["org_vocab"])
    stats_np = oracle.gathered_stats(x, c["shards"], c["org_vocab"])
    gh.assert_stats_equal(gh.stats_to_numpy(stats_dev), stats_np)
    _, t = oracle.full_argmax(x, c["org_vocab"])
    drafts = wl.compose_drafts(t, c["cu_num_draft"], c["flags"], c["rand_ids"])
    return check_verify(stats_dev, stats_np, len(c["shards"]), c["cu_num_draft"], drafts, c["k"])


def test_greedy_verify_workload(sga_lib):
    got = run_workload(wl.greedy_verify_small())
    assert 0 < got["num_rejected"].sum() < 24 * 3


def test_large_verify_workload(sga_lib):
    got = run_workload(wl.large_verify())
    assert got["num_sampled"].max() > 1


def random_stats(rng, rows, num_shards, vocab):
    """Gathered stats of random logits rows (the oracle computes them)."""
    x = wl.discrete_logits(int(rng.integers(1 << 30)), rows, vocab, "bf16", p_nan=0.002)
    shards = wl.random_shards(int(rng.integers(1 << 30)), vocab, num_shards)
    return oracle.gathered_stats(x, shards, vocab), x, shards


@pytest.mark.parametrize("num_shards", [1, 2, 3, 4, 8, 16, 17, 40, 257])
def test_random_variable_k_and_placeholders(sga_lib, num_shards):
    # up to 16 entries per row: 16 lanes per request; above: a warp per row
    rng = np.random.default_rng(num_shards)
    for trial in range(6):
        n = int(rng.integers(1, 300))
        max_k = int(rng.choice([1, 3, 5, 15]))
        ks = rng.integers(0, max_k + 1, n)
        cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
        total = int(cu[-1]) + n
        stats_np, _, _ = random_stats(rng, total, num_shards, 257)
        _, t = oracle.shard_reduce(stats_np, num_shards, total)
        flags = rng.random(int(cu[-1])) < 0.85
        rand = rng.integers(-1, 257, int(cu[-1])).astype(np.int32)   # -1 = placeholder
        drafts = wl.compose_drafts(t, cu, flags, rand)
        stats_dev = torch.from_numpy(stats_np.view(np.int32).reshape(-1, 2).copy()).cuda()
        check_verify(stats_dev, stats_np, num_shards, cu, drafts, max_k)


@pytest.mark.parametrize("num_shards", [2, 20])
def test_target_ids_optional(sga_lib, num_shards):
    rng = np.random.default_rng(5)
    cu = np.array([0, 3, 6], np.int32)
    stats_np, _, _ = random_stats(rng, 8, num_shards, 100)
    stats_dev = torch.from_numpy(stats_np.view(np.int32).reshape(-1, 2).copy()).cuda()
    got = gh.gpu_verify(stats_dev, num_shards, cu, np.zeros(6, np.int32), 3, with_target_ids=False)
    exp = oracle.greedy_verify(stats_np, num_shards, cu, np.zeros(6, np.int32), 3)
    assert (got["sampled"] == exp["sampled"]).all()
    assert (got["target_ids"] == -99).all()   # untouched


@pytest.mark.parametrize("num_shards", [1, 33])
def test_k_above_max_k_sets_error_word(sga_lib, num_shards):
    sga_lib.sga_clear_device_error()
    rng = np.random.default_rng(6)
    cu = np.array([0, 2, 6, 7], np.int32)   # request 1 has K = 4 > max_k = 3
    stats_np, _, _ = random_stats(rng, 10, num_shards, 50)
    stats_dev = torch.from_numpy(stats_np.view(np.int32).reshape(-1, 2).copy()).cuda()
    got = gh.gpu_verify(stats_dev, num_shards, cu, np.zeros(7, np.int32), 3)
    assert sga_lib.sga_device_error() & sga_lib.SGA_DEVERR_K_RANGE
    assert got["num_sampled"][1] == 0 and got["bonus"][1] == -1 and (got["sampled"][1] == -1).all()
    assert got["num_sampled"][0] >= 1 and got["num_sampled"][2] >= 1
    sga_lib.sga_clear_device_error()
    assert sga_lib.sga_device_error() == 0


@pytest.mark.parametrize("num_shards", [1, 3, 8, 16, 17, 40, 200, 257])
def test_shard_reduce_bit_exact_narrow_and_wide(sga_lib, num_shards):
    # the cross-shard reduce on its own, over statistics with NaNs, infinities,
    # signed zeros and ties: the thread-per-row kernel up to 16 entries per
    # row, the 32-streams-per-row kernel above; values bitwise, ids exact,
    # then the draft-to-target map applied to the same winners
    rng = np.random.default_rng(100 + num_shards)
    for rows in (1, 15, 16, 17, 333):
        stats_np, _, _ = random_stats(rng, rows, num_shards, 300)
        stats_dev = torch.from_numpy(stats_np.view(np.int32).reshape(-1, 2).copy()).cuda()
        vals, ids = gh.gpu_reduce(stats_dev, num_shards, rows)
        evals, eids = oracle.shard_reduce(stats_np, num_shards, rows)
        assert (ids == eids).all()
        assert (vals.view(np.uint32) == np.asarray(evals, np.float32).view(np.uint32)).all()
        d2t = (rng.integers(0, 50, 300) + np.arange(300) * 3).astype(np.int64) - np.arange(300)
        _, mapped = gh.gpu_reduce(stats_dev, num_shards, rows,
                                  d2t=torch.from_numpy(d2t).cuda())
        assert (mapped == oracle.d2t_map(eids, d2t)).all()
    assert sga_lib.sga_device_error() == 0


@pytest.mark.parametrize("num_shards", [4, 40])
def test_shard_reduce_d2t_out_of_range_sets_error_word(sga_lib, num_shards):
    # winners outside the draft-to-target table: the id is left unmapped and
    # the error word says so (thread-per-row and wide kernels alike)
    sga_lib.sga_clear_device_error()
    rng = np.random.default_rng(7)
    stats_np, _, _ = random_stats(rng, 40, num_shards, 300)
    stats_dev = torch.from_numpy(stats_np.view(np.int32).reshape(-1, 2).copy()).cuda()
    _, eids = oracle.shard_reduce(stats_np, num_shards, 40)
    assert (eids >= 10).any()
    short = torch.zeros(10, dtype=torch.int64, device="cuda")
    _, ids = gh.gpu_reduce(stats_dev, num_shards, 40, d2t=short)
    assert sga_lib.sga_device_error() & sga_lib.SGA_DEVERR_D2T_RANGE
    assert (ids == eids).all()   # a zero table maps every id to itself
    sga_lib.sga_clear_device_error()
    assert sga_lib.sga_device_error() == 0


def gpu_verify_prefill(stats_dev, num_shards, cu, drafts, max_k, mask):
    import greedy_spec_decode_gb300 as sga
    n = len(cu) - 1
    total = int(cu[-1]) + n
    i32 = dict(dtype=torch.int32, device="cuda")
    out = dict(sampled=torch.full((n, max_k + 1), -99, **i32),
               num_sampled=torch.full((n,), -99, **i32), num_rejected=torch.full((n,), -99, **i32),
               bonus=torch.full((n,), -99, **i32), target_ids=torch.full((total,), -99, **i32))
    sga.sga_greedy_verify_prefill(
        stats_dev, num_shards, torch.from_numpy(np.asarray(cu, np.int32)).cuda(),
        torch.from_numpy(np.asarray(drafts, np.int32)).cuda(),
        torch.from_numpy(np.asarray(mask, np.uint8)).cuda(), max_k, out["sampled"],
        out["num_sampled"], out["num_rejected"], out["bonus"], out["target_ids"])
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("num_shards", [1, 3, 40])
def test_prefill_hand_cases(sga_lib, num_shards):
    # the hand-computed batch of tests/golden/verify_prefill_cases.txt; 40
    # entries per row runs the wide kernel
    import test_oracle_pins as pins
    cu, drafts, t, max_k, mask, exp = pins.prefill_batch()
    st = pins.stats_for_targets(t, num_shards)
    got = gpu_verify_prefill(torch.from_numpy(st.view(np.int32).reshape(-1, 2).copy()).cuda(),
                             num_shards, cu, drafts, max_k, mask)
    for i, (samp, ns, nr, b) in enumerate(exp):
        assert list(got["sampled"][i]) == samp, i
        assert (got["num_sampled"][i], got["num_rejected"][i], got["bonus"][i]) == (ns, nr, b), i
    assert (got["target_ids"] == t).all()
    assert sga_lib.sga_device_error() == 0


@pytest.mark.parametrize("num_shards,n_reqs", [(2, 1), (3, 37), (8, 256), (24, 33), (200, 9)])
def test_prefill_mask_random_matches_oracle(sga_lib, num_shards, n_reqs):
    rng = np.random.default_rng(num_shards * 1000 + n_reqs)
    max_k = int(rng.integers(1, 16))
    ks = rng.integers(0, max_k + 1, n_reqs)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    rows = int(cu[-1]) + n_reqs
    st, x, shards = random_stats(rng, rows, num_shards, max(4 * num_shards, 300))
    _, t = oracle.full_argmax(x, x.shape[1])
    flags = rng.random(int(cu[-1])) < 0.7
    drafts = wl.compose_drafts(t, cu, flags, rng.integers(-1, x.shape[1], int(cu[-1])).astype(np.int32))
    mask = (rng.random(n_reqs) < 0.3).astype(np.uint8)
    dev = torch.from_numpy(st.view(np.int32).reshape(-1, 2).copy()).cuda()
    got = gpu_verify_prefill(dev, num_shards, cu, drafts, max_k, mask)
    exp = oracle.greedy_verify(st, num_shards, cu, drafts, max_k, in_prefill=mask)
    for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
        assert (got[key] == exp[key]).all(), key
    # an all-zero mask is the plain entry point's result
    none = gpu_verify_prefill(dev, num_shards, cu, drafts, max_k, np.zeros(n_reqs, np.uint8))
    plain = gh.gpu_verify(dev, num_shards, cu, drafts, max_k)
    for key in plain:
        assert (none[key] == plain[key]).all(), key
    assert sga_lib.sga_device_error() == 0
