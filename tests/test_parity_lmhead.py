"""GPU parity of sga_lmhead_argmax (tcgen05 GEMM + argmax epilogue) against
the CPU oracle's fp64 logits.

The GPU accumulates in fp32 in its own order, so parity is within tolerance:
where the oracle's top-1 minus top-2 logit gap exceeds GAP, the GPU id must
equal the oracle's; elsewhere the GPU id must be a valid near-winner (its
oracle logit within GAP of the top-1).  The GPU value must be within REL of
the oracle's top-1 (relative, with an absolute floor ABS).  vLLM PR #62604,
Purpose item 2 (fused get_top_tokens: same result as torch.argmax on the
logits) with the LM head of the Purpose paragraph.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh

pytestmark = pytest.mark.gpu

GAP = 1e-2
REL = 1e-2
ABS = 1e-3


def run_gpu(hidden, weight, shards, org_vocab):
    h = gh.to_device(hidden)
    w = gh.to_device(weight)
    M = hidden.shape[0]
    stats = torch.full((len(shards) * M, 2), -5, dtype=torch.int32, device="cuda")
    ws_bytes = max(sga_ws(M, wd) for _, wd in shards)
    ws = torch.empty(max(ws_bytes, 8), dtype=torch.uint8, device="cuda")
    import greedy_spec_decode_gb300 as sga
    for s, (o, wd) in enumerate(shards):
        sga.sga_lmhead_argmax(h, w[o:o + wd], o, org_vocab, stats[s * M:(s + 1) * M], ws)
    ids = torch.empty(M, dtype=torch.int32, device="cuda")
    vals = torch.empty(M, dtype=torch.float32, device="cuda")
    sga.sga_shard_reduce(stats, len(shards), M, ids, vals)
    assert sga.sga_device_error() == 0
    return gh.stats_to_numpy(stats), vals.cpu().numpy(), ids.cpu().numpy()


def sga_ws(M, width):
    import greedy_spec_decode_gb300 as sga
    return sga.sga_lmhead_argmax_workspace(M, width)


def check_rows(rows, hidden, weight, shards, org_vocab, gpu_stats, gpu_vals, gpu_ids):
    M = hidden.shape[0]
    vocab = weight.shape[0]
    logits = oracle.lmhead_logits(hidden, weight, rows)          # [n, vocab] fp64
    top1, top2, ids = oracle.argmax_f64(logits, 0, org_vocab)
    checked = excluded = 0
    for q, r in enumerate(rows):
        gi, gv = int(gpu_ids[r]), float(gpu_vals[r])
        assert 0 <= gi < vocab
        if top1[q] == -np.inf:                         # every id padded
            assert gv == -np.inf
            continue
        assert gi < org_vocab
        if top1[q] - top2[q] > GAP:
            assert gi == ids[q], (r, gi, ids[q], top1[q], top2[q])
            checked += 1
        else:
            assert logits[q, gi] >= top1[q] - GAP, (r, gi, logits[q, gi], top1[q])
            excluded += 1
        assert abs(gv - top1[q]) <= max(REL * abs(top1[q]), ABS), (r, gv, top1[q])
        for s, (o, wd) in enumerate(shards):
            st = gpu_stats[s * M + r]
            s1, s2, sid = oracle.argmax_f64(logits[q:q + 1, o:o + wd], o, org_vocab)
            if s1[0] == -np.inf:
                assert st["id"] == o and st["v"] == -np.inf
                continue
            if s1[0] - s2[0] > GAP:
                assert st["id"] == sid[0], (r, s, st, sid[0])
            assert abs(float(st["v"]) - s1[0]) <= max(REL * abs(s1[0]), ABS)
    return checked, excluded


@pytest.mark.parametrize("M,H,vocab,num_shards", [
    (1, 64, 300, 1), (100, 128, 1000, 2), (128, 512, 5000, 3), (300, 256, 2311, 4),
    (257, 64, 256, 1), (513, 1024, 4099, 2),
    # decode-size batches (one to a few dozen rows against a large head), and
    # the CTA-pair kernel with a single K block (H = 64: a partial stage)
    (1, 4096, 20000, 2), (16, 4096, 20000, 2), (64, 1024, 30011, 3), (96, 64, 3000, 2),
])
def test_small_shapes(sga_lib, M, H, vocab, num_shards):
    hidden = wl.normal_matrix(M + H, M, H, 1.0)
    weight = wl.normal_matrix(vocab + H, vocab, H, 1.0 / np.sqrt(H))
    shards = wl.random_shards(M + vocab, vocab, num_shards) if num_shards > 1 else [(0, vocab)]
    for org in (vocab, vocab - 37 if vocab > 40 else vocab):
        st, v, i = run_gpu(hidden, weight, shards, org)
        check_rows(np.arange(M), hidden, weight, shards, org, st, v, i)


@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 31, 32, 33, 48, 63, 64, 65, 96, 127, 128, 129])
def test_decode_sizes_around_kernel_boundaries(sga_lib, M):
    # M <= 64 runs the swapped-operand decode kernel with N = 16, 32 or 64
    # hidden columns; 65..128 its CTA-pair form (N = 128, 64 hidden rows in
    # each CTA of the pair); 129 is the first size of the 2-SM GEMM kernel.
    # A ragged vocab (not a multiple of 128 or 256), 3 uneven shards, and
    # padding.
    H, vocab = 256, 4099
    hidden = wl.normal_matrix(900 + M, M, H, 1.0)
    weight = wl.normal_matrix(901 + M, vocab, H, 1.0 / np.sqrt(H))
    shards = wl.random_shards(M, vocab, 3)
    for org in (vocab, shards[1][0] + 5):
        st, v, i = run_gpu(hidden, weight, shards, org)
        check_rows(np.arange(M), hidden, weight, shards, org, st, v, i)


@pytest.mark.parametrize("M,H", [(8, 192), (40, 64), (3, 320)])
def test_decode_sizes_odd_number_of_k_blocks(sga_lib, M, H):
    # H / 64 odd: the last pipeline stage of a two-K-block ring holds one block
    vocab = 1500
    hidden = wl.normal_matrix(40 + M, M, H, 1.0)
    weight = wl.normal_matrix(41 + M, vocab, H, 1.0 / np.sqrt(H))
    shards = wl.even_shards(vocab, 2)
    st, v, i = run_gpu(hidden, weight, shards, vocab)
    check_rows(np.arange(M), hidden, weight, shards, vocab, st, v, i)


def test_decode_size_vocab_narrower_than_a_tile(sga_lib):
    # one shard of 100 ids: a single 256-id tile, one CTA, 156 ids of zero fill
    M, H, vocab = 9, 128, 100
    hidden = wl.normal_matrix(31, M, H, 1.0)
    weight = wl.normal_matrix(32, vocab, H, 1.0 / np.sqrt(H))
    st, v, i = run_gpu(hidden, weight, [(0, vocab)], vocab)
    check_rows(np.arange(M), hidden, weight, [(0, vocab)], vocab, st, v, i)


@pytest.mark.parametrize("M", [130, 100, 40, 20, 5])
def test_all_padding_shard_and_exact_one_hot(sga_lib, M):
    # one-hot weights: logit[r][j] = hidden[r][perm[j]] exactly, so ties and
    # values are exact and the id must follow torch.argmax order (M <= 128:
    # decode kernels, where ties are resolved across lanes, warps and CTAs)
    H, vocab = 128, 600
    hidden = wl.normal_matrix(7, M, H, 1.0)
    perm = np.random.default_rng(1).integers(0, H, vocab)
    weight = np.zeros((vocab, H), np.uint16)
    weight[np.arange(vocab), perm] = wl.bf16_const(1.0)
    shards = [(0, 256), (256, 300), (556, 44)]
    org = 556                                         # last shard all padding
    st, v, i = run_gpu(hidden, weight, shards, org)
    hf = wl.bf16_bits_to_f32(hidden)
    for r in range(M):
        row = hf[r, perm[:org]]
        j = int(np.flatnonzero(row == row.max())[0])
        assert i[r] == j and v[r] == row.max()
        assert st[2 * M + r]["id"] == 556 and st[2 * M + r]["v"] == -np.inf


@pytest.mark.parametrize("M_req,K,H,vocab,num_shards", [(6, 3, 256, 5000, 3), (40, 1, 128, 3001, 2)])
def test_lmhead_stats_feed_greedy_verify(sga_lib, M_req, K, H, vocab, num_shards):
    # the whole target side from hidden states: fused LM-head argmax per shard
    # (stats gathered shard-major) -> fused greedy verify.  Each row gets a
    # planted winner (its weight row is the row's own hidden vector, so its
    # logit |h|^2 ~ H beats every other by a wide margin); the expected
    # tokens are then exact and the verify outputs must match the oracle's
    import greedy_spec_decode_gb300 as sga
    rows = M_req * (K + 1)
    rng = np.random.default_rng(rows + vocab)
    hidden = wl.normal_matrix(rows + 1, rows, H, 1.0)
    weight = wl.normal_matrix(rows + 2, vocab, H, 1.0 / np.sqrt(H))
    planted = rng.choice(vocab, rows, replace=False).astype(np.int32)
    weight[planted] = hidden
    shards = wl.random_shards(rows, vocab, num_shards)
    st, _, ids = run_gpu(hidden, weight, shards, vocab)
    logits = oracle.lmhead_logits(hidden, weight, np.arange(rows))
    top1, top2, exp_ids = oracle.argmax_f64(logits, 0, vocab)
    assert (top1 - top2 > 1.0).all() and (exp_ids == planted).all()
    assert (ids == planted).all()
    cu = np.arange(M_req + 1, dtype=np.int32) * K
    flags = rng.random(M_req * K) < 0.7
    drafts = wl.compose_drafts(planted, cu, flags, rng.integers(0, vocab, M_req * K).astype(np.int32))
    stats_dev = torch.from_numpy(st.view(np.int32).reshape(-1, 2).copy()).cuda()
    got = gh.gpu_verify(stats_dev, num_shards, cu, drafts, K)
    oracle_stats = np.zeros(num_shards * rows, oracle.STAT)
    for s, (o, w) in enumerate(shards):
        s1, _, sid = oracle.argmax_f64(logits[:, o:o + w], o, vocab)
        oracle_stats["v"][s * rows:(s + 1) * rows] = s1
        oracle_stats["id"][s * rows:(s + 1) * rows] = sid
    ref = oracle.greedy_verify(oracle_stats, num_shards, cu, drafts, K)
    for key in ("sampled", "num_sampled", "num_rejected", "bonus", "target_ids"):
        assert (got[key] == ref[key]).all(), key
    assert sga.sga_device_error() == 0
