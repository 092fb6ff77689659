"""Pins of the CPU oracle to things other than itself (CPU only).

* an independent, set-based brute force of the argmax rule (written in pure
  Python, not as a scan), on tie-heavy tiny inputs with +-0, +-inf, NaN and
  padding, for several shardings;
* torch.argmax on CPU as a library third opinion for unpadded rows;
* planted rows with answers fixed by the rule (tests/golden/tiny_planted.txt)
  and by construction (padding spikes, exact cross-shard-edge ties);
* hand-computed greedy acceptance cases (tests/golden/verify_hand_cases.txt)
  and an independent prefix-length brute force of the acceptance rule;
* the LM-head logits against numpy's fp64 matmul and exact one-hot weights.

Rules restated from vLLM PR #62604 (Purpose items 1-2, Test Plan) and
PR #34049 (Solution).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits32(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def as_f32(x):
    return wl.bf16_bits_to_f32(x) if x.dtype == np.uint16 else x


def brute_argmax_row(vals, first, org_vocab):
    """Set-based reading of 'lowest id on ties, NaN wins' over ids
    first .. first+len-1 with ids >= org_vocab masked: returns (id, f32 value)."""
    ids = list(range(first, first + len(vals)))
    live = [(i, float(v)) for i, v in zip(ids, vals) if i < org_vocab]
    nan_ids = [i for i, v in live if math.isnan(v)]
    if nan_ids:
        i = min(nan_ids)
        return i, vals[i - first]
    if not live or all(v == -math.inf for _, v in live):
        return first, np.float32(-np.inf)
    top = max(v for _, v in live)
    i = min(i for i, v in live if v == top)
    return i, vals[i - first]


def check_against_brute(x, shards, org_vocab):
    xf = as_f32(x)
    vals, ids = oracle.full_argmax(x, org_vocab)
    stats = oracle.gathered_stats(x, shards, org_vocab)
    rvals, rids = oracle.shard_reduce(stats, len(shards), x.shape[0])
    for r in range(x.shape[0]):
        bi, bv = brute_argmax_row(xf[r], 0, org_vocab)
        assert ids[r] == bi and rids[r] == bi, (r, ids[r], rids[r], bi)
        assert bits32(vals[r]) == bits32(bv) == bits32(rvals[r])
        for s, (o, w) in enumerate(shards):
            si, sv = brute_argmax_row(xf[r, o:o + w], o, org_vocab)
            st = stats[s * x.shape[0] + r]
            assert st["id"] == si and bits32(st["v"]) == bits32(sv), (r, s)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("num_shards", [1, 2, 3, 4, 8])
def test_argmax_matches_set_brute_force(dtype, num_shards):
    for seed in range(6):
        vocab = 37 + 7 * seed
        x = wl.discrete_logits(100 * num_shards + seed, 12, vocab, dtype)
        shards = wl.random_shards(seed, vocab, num_shards)
        for org in (vocab, vocab - 5, 3, 0 if num_shards == 1 else shards[-1][0]):
            check_against_brute(x, shards, max(org, 0) if org > 0 else 1)


def test_shard_narrower_than_vector_and_single_ids():
    x = wl.discrete_logits(5, 16, 20, "bf16", p_nan=0.1)
    shards = [(i, 1) for i in range(20)]
    check_against_brute(x, shards, 17)


def test_all_padding_shard_reports_its_first_id():
    x = wl.discrete_logits(6, 4, 30, "f32", p_nan=0.0, p_inf=0.0)
    st = oracle.shard_argmax(x, 20, 10, org_vocab=20)
    assert (st["id"] == 20).all() and np.isneginf(st["v"]).all()


def test_nan_and_inf_only_in_padding_never_win():
    x = np.zeros((2, 10), np.float32)
    x[:, 8] = np.nan
    x[:, 9] = np.inf
    x[1, 3] = 1.0
    _, ids = oracle.full_argmax(x, org_vocab=8)
    assert list(ids) == [0, 3]


def test_plus_minus_zero_tie_keeps_lowest_id_and_its_bits():
    x = np.array([[-0.0, 0.0, -1.0], [-1.0, 0.0, -0.0]], np.float32)
    vals, ids = oracle.full_argmax(x)
    assert list(ids) == [0, 1]
    assert bits32(vals[0]) == 0x80000000 and bits32(vals[1]) == 0


def test_nan_payload_and_first_nan_across_shards():
    x = np.zeros((1, 8), np.uint16)
    x[0, 5] = 0x7FC1  # NaN with a payload, shard 1
    x[0, 6] = 0x7FC0
    x[0, 2] = 0x4000  # 2.0 in shard 0
    st = oracle.gathered_stats(x, [(0, 4), (4, 4)], 8)
    vals, ids = oracle.shard_reduce(st, 2, 1)
    assert ids[0] == 5 and bits32(vals[0]) == 0x7FC10000


def test_torch_argmax_third_opinion_unpadded():
    for seed in range(4):
        x = wl.normal_matrix(seed, 9, 333, 1.0, dtype="f32")
        x[seed, 17 + seed] = np.nan
        x[(seed + 1) % 9, 3] = x[(seed + 1) % 9, 300] = 99.0
        for shards in (wl.even_shards(333, 3), wl.random_shards(seed, 333, 5)):
            st = oracle.gathered_stats(x, shards, 333)
            _, rids = oracle.shard_reduce(st, len(shards), 9)
            ref = torch.argmax(torch.from_numpy(x), dim=1).numpy()
            assert (rids == ref).all()


def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([c.strip() for c in line.split("|")])
    return rows


def test_tiny_workload_planted_rows():
    c = wl.tiny_sharded_argmax()
    x = c["logits"]
    st = oracle.gathered_stats(x, c["shards"], c["org_vocab"])
    vals, ids = oracle.shard_reduce(st, 2, x.shape[0])
    table = read_table("tiny_planted.txt")
    assert len(table) == 3
    for row, eid, ev in table:
        r, eid, ev = int(row), int(eid), float(ev)
        assert ids[r] == eid
        if math.isnan(ev):
            assert math.isnan(vals[r])
        else:
            assert vals[r] == ev
    check_against_brute(x, c["shards"], c["org_vocab"])


def test_draft_workload_padding_spikes_ignored():
    c = wl.draft_top_tokens()
    x = c["logits"][:8]
    vals, ids = oracle.full_argmax(x, c["org_vocab"])
    assert (ids < c["org_vocab"]).all() and not np.isnan(vals).any()
    assert (vals < 100.0).all()
    st = oracle.gathered_stats(x, c["shards"], c["org_vocab"])
    _, rids = oracle.shard_reduce(st, 2, 8)
    assert (rids == ids).all()
    # without the mask the planted NaN (id 152000) would win rows r % 4 == 0,
    # since a NaN beats every number; the mask is what keeps them in-vocabulary
    _, raw = oracle.full_argmax(x, x.shape[1])
    assert raw[0] == 152000 and raw[4] == 152000 and raw[1] < c["org_vocab"]


def test_large_verify_sample_planted_edge_ties():
    c = wl.large_verify(rows_limit=208)
    x = c["logits"]
    st = oracle.gathered_stats(x, c["shards"], c["org_vocab"])
    vals, ids = oracle.shard_reduce(st, 3, x.shape[0])
    for r in range(0, x.shape[0], 100):
        s = 1 + (r // 100) % 2
        o = c["shards"][s][0]
        assert ids[r] == o - 1 and vals[r] == wl.LARGE_TIE_VALUE
    full_vals, full_ids = oracle.full_argmax(x, c["org_vocab"])
    assert (full_ids == ids).all() and (bits32(full_vals) == bits32(vals)).all()


def stats_for_targets(t, num_shards=1, seed=0):
    """Gathered stats whose global argmax per row is t[row]: shard 0 holds
    the winner with value 1.0, the other shards hold lower values."""
    rows = len(t)
    st = np.zeros(num_shards * rows, oracle.STAT)
    rng = np.random.default_rng(seed)
    for s in range(num_shards):
        st["v"][s * rows:(s + 1) * rows] = 1.0 if s == 0 else 0.5
        st["id"][s * rows:(s + 1) * rows] = t if s == 0 else rng.integers(10**6, 2 * 10**6, rows)
    return st


def test_verify_hand_cases():
    for k, drafts, t, sampled, ns, nr, bonus in read_table("verify_hand_cases.txt"):
        k = int(k)
        drafts = [int(v) for v in drafts.split()]
        t = np.array([int(v) for v in t.split()], np.int32)
        exp = [int(v) for v in sampled.split()]
        for num_shards in (1, 3):
            st = stats_for_targets(t, num_shards)
            out = oracle.greedy_verify(st, num_shards, np.array([0, k], np.int32),
                                       np.array(drafts, np.int32), max_k=k)
            assert list(out["sampled"][0]) == exp
            assert out["num_sampled"][0] == int(ns) and out["num_rejected"][0] == int(nr)
            assert out["bonus"][0] == int(bonus)
            assert (out["target_ids"] == t).all()


def prefill_batch():
    """The hand cases of verify_prefill_cases.txt as one batch: (cu, drafts,
    t, max_k, in_prefill, expected per request)."""
    table = read_table("verify_prefill_cases.txt")
    ks = [int(r[1]) for r in table]
    max_k = max(ks)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    drafts = np.array([int(v) for r in table for v in r[2].split()], np.int32)
    t = np.array([int(v) for r in table for v in r[3].split()], np.int32)
    mask = np.array([int(r[0]) for r in table], np.uint8)
    exp = []
    for r in table:
        samp = [int(v) for v in r[4].split()]
        exp.append((samp + [-1] * (max_k + 1 - len(samp)), int(r[5]), int(r[6]), int(r[7])))
    return cu, drafts, t, max_k, mask, exp


def test_verify_prefill_hand_cases():
    cu, drafts, t, max_k, mask, exp = prefill_batch()
    assert len(t) == int(cu[-1]) + len(exp)
    for num_shards in (1, 3):
        st = stats_for_targets(t, num_shards)
        out = oracle.greedy_verify(st, num_shards, cu, drafts, max_k, in_prefill=mask)
        for i, (samp, ns, nr, b) in enumerate(exp):
            assert list(out["sampled"][i]) == samp, i
            assert (out["num_sampled"][i], out["num_rejected"][i], out["bonus"][i]) == (ns, nr, b), i
        assert (out["target_ids"] == t).all()
        # without the mask the same batch follows the greedy rule everywhere
        plain = oracle.greedy_verify(st, num_shards, cu, drafts, max_k)
        for i, (samp, ns, nr, b) in enumerate(brute_verify(t, cu, drafts, max_k)):
            assert list(plain["sampled"][i]) == samp
            assert (plain["num_sampled"][i], plain["num_rejected"][i], plain["bonus"][i]) == (ns, nr, b)


def brute_verify(t, cu, drafts, max_k):
    """Prefix-length reading of greedy acceptance, written independently."""
    res = []
    for i in range(len(cu) - 1):
        k = cu[i + 1] - cu[i]
        rows = t[cu[i] + i: cu[i + 1] + i + 1]
        d = drafts[cu[i]:cu[i + 1]]
        a = next((j for j in range(k) if d[j] != rows[j]), k)
        emitted = list(rows[:a + 1])
        res.append((emitted + [-1] * (max_k + 1 - len(emitted)), a + 1, k - a, emitted[-1]))
    return res


def test_verify_random_variable_k_matches_brute_force():
    rng = np.random.default_rng(11)
    for trial in range(40):
        n = int(rng.integers(1, 9))
        max_k = int(rng.integers(1, 16))
        ks = rng.integers(0, max_k + 1, n)
        cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
        t = rng.integers(0, 5, int(cu[-1]) + n).astype(np.int32)
        flags = rng.random(int(cu[-1])) < 0.8
        drafts = wl.compose_drafts(t, cu, flags, rng.integers(-1, 5, int(cu[-1])).astype(np.int32))
        num_shards = int(rng.integers(1, 5))
        st = stats_for_targets(t, num_shards, trial)
        out = oracle.greedy_verify(st, num_shards, cu, drafts, max_k)
        for i, (samp, ns, nr, b) in enumerate(brute_verify(t, cu, drafts, max_k)):
            assert list(out["sampled"][i]) == samp
            assert (out["num_sampled"][i], out["num_rejected"][i], out["bonus"][i]) == (ns, nr, b)
            assert out["num_sampled"][i] + out["num_rejected"][i] == ks[i] + 1


def test_verify_reduces_stats_across_shards_first():
    # the winner of row 0 lives in shard 1 (higher value), of row 1 in shard 0 (tie)
    st = np.zeros(4, oracle.STAT)
    st[0] = (1.0, 3)
    st[1] = (2.0, 4)
    st[2] = (5.0, 12)
    st[3] = (2.0, 14)
    out = oracle.greedy_verify(st, 2, np.array([0, 1], np.int32), np.array([12], np.int32), 1)
    assert list(out["target_ids"]) == [12, 4]
    assert list(out["sampled"][0]) == [12, 4] and out["bonus"][0] == 4


def test_d2t_map_hand_case():
    # draft vocab of 4 ids mapped into a larger target vocab: target = k + d2t[k]
    d2t = np.array([0, 9, 20, 96], np.int64)
    assert list(oracle.d2t_map(np.array([0, 1, 2, 3, 1], np.int32), d2t)) == [0, 10, 22, 99, 10]
    with pytest.raises(ValueError):
        oracle.d2t_map(np.array([4], np.int32), d2t)


def test_lmhead_logits_match_numpy_fp64_matmul():
    h = wl.normal_matrix(1, 6, 96, 1.0)
    w = wl.normal_matrix(2, 50, 96, 0.02)
    rows = np.array([0, 5, 2], np.int64)
    got = oracle.lmhead_logits(h, w, rows)
    ref = wl.bf16_bits_to_f32(h[rows]).astype(np.float64) @ wl.bf16_bits_to_f32(w).astype(np.float64).T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)


def test_lmhead_one_hot_weight_is_exact_column_pick():
    H, V = 64, 40
    h = wl.normal_matrix(3, 4, H, 1.0)
    perm = np.random.default_rng(0).permutation(H)[:V]
    w = np.zeros((V, H), np.uint16)
    w[np.arange(V), perm] = wl.bf16_const(1.0)
    got = oracle.lmhead_logits(h, w, np.arange(4))
    assert (got == wl.bf16_bits_to_f32(h)[:, perm].astype(np.float64)).all()
    # a transposed operand would pick rows of hidden, not columns: shapes differ, so check one row
    top1, top2, ids = oracle.lmhead_argmax(h, w, np.arange(4), shard_start=100, org_vocab=100 + V - 3)
    for r in range(4):
        row = wl.bf16_bits_to_f32(h[r])[perm][:V - 3].astype(np.float64)
        j = int(np.flatnonzero(row == row.max())[0])
        assert ids[r] == 100 + j and top1[r] == row.max()
        assert top2[r] == np.sort(np.delete(row, j))[-1]


def test_e4m3_decode_matches_torch_float8_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(c) for c in codes])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert (both_nan | (got == ref)).all()
    assert np.isnan(got).sum() == 2                          # 0x7F and 0xFF
    assert (np.signbit(got[128:]) | np.isnan(got[128:])).all()  # -0 included


def test_lmhead_fp8_logits_match_numpy_with_scales():
    rng = np.random.default_rng(3)
    hq = rng.integers(0, 256, (5, 128), dtype=np.uint8)
    hq[hq & 0x7F == 0x7F] = 0x3C                       # no NaN codes
    wq = rng.integers(0, 256, (37, 128), dtype=np.uint8)
    wq[wq & 0x7F == 0x7F] = 0x41
    hs = rng.uniform(0.01, 2.0, 5).astype(np.float32)
    ws = 0.0037
    rows = np.array([4, 0, 2], np.int64)
    got = oracle.lmhead_logits_fp8(hq, hs, wq, ws, rows)
    dec = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).double().numpy()
    ref = (dec(hq[rows]) @ dec(wq).T) * hs[rows, None].astype(np.float64) * ws
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-300)


def test_e4m3_quantizer_of_the_generators_matches_torch():
    x = np.random.default_rng(4).standard_normal(50000).astype(np.float32) * 60
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (wl.f32_to_e4m3(x) == ref).all()


def brute_block_stats(xf, shard, org_vocab, row_blocks):
    """Independent reading of block-granular stats: group the shard's ids by
    their global block id // B (B of that row), in ascending block order,
    and take the set-based argmax of each group.  Returns, per row, the
    list of (id, value) of its pieces."""
    o, w = shard
    res = []
    for r, B in enumerate(row_blocks):
        groups = {}
        for i in range(o, o + w):
            groups.setdefault(i // B, []).append(i)
        res.append([brute_argmax_row(xf[r, ids[0]:ids[-1] + 1], ids[0], org_vocab)
                    for _, ids in sorted(groups.items())])
    return res


def row_blocks_of(rows, cu, draft_block, bonus_block):
    blocks = [draft_block] * rows
    if cu is not None:
        for i in range(len(cu) - 1):
            blocks[cu[i + 1] + i] = bonus_block
    return blocks


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_block_stats_match_grouped_brute_force(dtype):
    rng = np.random.default_rng(21)
    for trial in range(16):
        n = int(rng.integers(1, 5))
        ks = rng.integers(0, 4, n)
        cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
        rows = int(cu[-1]) + n
        vocab = int(rng.integers(20, 90))
        x = wl.discrete_logits(300 + trial, rows, vocab, dtype, p_nan=0.02)
        xf = as_f32(x)
        shards = wl.random_shards(trial, vocab, int(rng.integers(1, 5)))
        draft_block, bonus_block = [(8, 2), (4, 16), (16, 16), (1, 4), (32, 8), (128, 1),
                                    (3, 2), (5, 7)][trial % 8]
        use_cu = trial % 3 != 0
        blocks = row_blocks_of(rows, cu if use_cu else None, draft_block, bonus_block)
        for org in (vocab, vocab - 7, shards[-1][0] + 1):
            for o, w in shards:
                st = oracle.block_stats(x, o, w, org, draft_block, bonus_block,
                                        cu if use_cu else None)
                n_pieces = max(len({i // B for i in range(o, o + w)})
                               for B in (draft_block, bonus_block))
                assert st.shape[0] == n_pieces * rows
                exp = brute_block_stats(xf, (o, w), org, blocks)
                for r in range(rows):
                    for p in range(n_pieces):
                        got = st[p * rows + r]
                        if p < len(exp[r]):
                            assert got["id"] == exp[r][p][0], (trial, o, w, r, p)
                            assert bits32(got["v"]) == bits32(exp[r][p][1])
                        else:
                            assert got["id"] == o + w - 1 and got["v"] == -np.inf


def test_block_stats_reduce_to_the_full_argmax_and_to_shard_stats():
    # the reduction over all pieces of all shards is the unsharded argmax for
    # every block size; one block wider than the vocab gives the shard stats
    x = wl.discrete_logits(7, 40, 700, "bf16", p_nan=0.003, p_inf=0.01)
    cu = np.array([0, 3, 3, 10, 25, 35], np.int32)          # 35 drafts + 5 bonus rows
    for shards in (wl.even_shards(700, 3), wl.random_shards(4, 700, 5), [(0, 700)]):
        for org in (700, 613):
            _, full_ids = oracle.full_argmax(x, org)
            for db, bb in ((8192, 1024), (64, 16), (16, 64), (1, 1), (256, 256), (24, 7)):
                st, n = oracle.gathered_block_stats(x, shards, org, db, bb, cu)
                assert n == sum(max(oracle.block_count(o, w, db), oracle.block_count(o, w, bb))
                                for o, w in shards)
                _, ids = oracle.shard_reduce(st, n, 40)
                assert (ids == full_ids).all(), (db, bb, org)
            st, n = oracle.gathered_block_stats(x, shards, org, 1 << 20)
            assert n == len(shards)
            sh = oracle.gathered_stats(x, shards, org)
            assert (st["id"] == sh["id"]).all() and (bits32(st["v"]) == bits32(sh["v"])).all()


def test_block_pieces_follow_global_boundaries_across_shard_edges():
    # shard [5, 15) with 4-id blocks: pieces [5,8), [8,12), [12,15); the
    # second shard [15, 21) starts inside block [12,16), which it shares
    vals = np.arange(21, dtype=np.float32)[::-1].copy()   # strictly decreasing
    x = vals[None, :]
    assert oracle.block_count(5, 10, 4) == 3 and oracle.block_count(15, 6, 4) == 3
    assert oracle.block_count(2, 2, 3) == 2 and oracle.block_count(2, 2, 2) == 1
    assert oracle.block_slots(2, 2, 2, 3) == 2
    assert list(oracle.block_stats(x, 5, 10, 21, 4)["id"]) == [5, 8, 12]
    assert list(oracle.block_stats(x, 15, 6, 21, 4)["id"]) == [15, 16, 20]
    assert list(oracle.block_stats(x, 15, 6, 18, 4)["id"]) == [15, 16, 20]
    st = oracle.block_stats(x, 15, 6, 18, 4)
    assert st["v"][0] == 5.0 and st["v"][1] == 4.0 and st["v"][2] == -np.inf
