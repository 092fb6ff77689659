"""GPU parity of sga_lmhead_argmax_shards / _fp8: the LM head over several vocab
shards of one weight buffer in one call (at decode sizes one launch of the
decode-size kernel, whose CTAs also merge the shards' statistics; from M =
129 one 2-SM GEMM launch and one finalize for every shard).  Each tile's
accumulation is the same as in one call per shard and the per-row merge uses
the total (value, id) order, so the statistics must be bit-identical to
num_shards sga_lmhead_argmax calls; sampled rows are also checked against the
oracle's fp64 logits within the LM-head tolerance.  vLLM PR #62604, Purpose
(vocab-parallel LM head), item 2 (fused get_top_tokens).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh
import test_parity_lmhead as lm
import test_parity_lmhead_fp8 as f8

pytestmark = pytest.mark.gpu


def one_call(sga, h, w, shards, org_vocab, fp8=False, hs=None, w_scale=1.0):
    """All shards through one sga_lmhead_argmax_shards[_fp8] call; w spans
    [shards[0][0], last end)."""
    M = h.shape[0]
    stats = torch.full((len(shards) * M, 2), -5, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(8, sga.sga_lmhead_argmax_shards_workspace(M, shards)),
                     dtype=torch.uint8, device="cuda")
    if fp8:
        sga.sga_lmhead_argmax_shards_fp8(h, hs, w, w_scale, shards, org_vocab, stats, ws)
    else:
        sga.sga_lmhead_argmax_shards(h, w, shards, org_vocab, stats, ws)
    assert sga.sga_device_error() == 0
    return gh.stats_to_numpy(stats)


@pytest.mark.parametrize("M", [1, 7, 16, 17, 32, 33, 64, 65, 96, 128, 200, 513])
@pytest.mark.parametrize("layout", ["uneven3", "gap", "padded", "eight", "single"])
def test_bf16_one_call_equals_per_shard_calls(sga_lib, M, layout):
    H = 256
    if layout == "uneven3":
        vocab, org, shards = 10000, 10000, [(0, 3334), (3334, 3333), (6667, 3333)]
    elif layout == "gap":          # a GPU holding shards 0 and 2 of three
        vocab, org, shards = 9000, 9000, [(0, 3000), (6000, 3000)]
    elif layout == "padded":       # the last shard past org_vocab, the one before it partly
        vocab, org, shards = 6144, 3500, [(0, 2048), (2048, 2048), (4096, 2048)]
    elif layout == "eight":
        vocab, org, shards = 16384, 16000, wl.even_shards(16384, 8)
    else:
        vocab, org, shards = 5000, 4990, [(0, 5000)]
    hidden = wl.normal_matrix(M + 11, M, H, 1.0)
    weight = wl.normal_matrix(M + 12, vocab, H, 1.0 / np.sqrt(H))
    per, vals, ids = lm.run_gpu(hidden, weight, shards, org)
    o0, end = shards[0][0], shards[-1][0] + shards[-1][1]
    one = one_call(sga_lib, gh.to_device(hidden), gh.to_device(weight)[o0:end], shards, org)
    gh.assert_stats_equal(one, per)
    if layout != "gap":   # (the oracle's full-vocab argmax would see the ids between shards)
        rows = np.arange(M) if M <= 20 else np.arange(0, M, 7)
        lm.check_rows(rows, hidden, weight, shards, org, per, vals, ids)


@pytest.mark.parametrize("M", [1, 16, 40, 64, 100, 300])
def test_fp8_one_call_equals_per_shard_calls(sga_lib, M):
    H, vocab = 256, 12288
    shards = [(0, 4096), (4096, 4096), (8192, 4096)]
    org = 12200
    hq, hs, wq, w_scale = f8.make(M, H, vocab, 900 + M)
    per, vals, ids = f8.run_gpu(sga_lib, hq, hs, wq, w_scale, shards, org)
    hs_d = torch.from_numpy(np.ascontiguousarray(hs, np.float32)).cuda()
    one = one_call(sga_lib, f8.u8(hq), f8.u8(wq), shards, org, fp8=True, hs=hs_d,
                   w_scale=w_scale)
    gh.assert_stats_equal(one, per)
    f8.check(np.arange(0, M, 5), hq, hs, wq, w_scale, shards, org, per, vals, ids)


def test_fused_lmhead_decode_shape_every_shard_in_one_launch(sga_lib):
    # the fused LM-head weight (151936 x 4096, 2 and 8 shards) at M = 16,
    # against the per-shard calls bit for bit
    c = wl.fused_lmhead(m=16)
    h = torch.from_numpy(c["hidden"].view(np.int16)).view(torch.bfloat16).cuda()
    w = torch.from_numpy(c["weight"].view(np.int16)).view(torch.bfloat16).cuda()
    for shards in (c["shards"], wl.even_shards(151936, 8)):
        M = 16
        per = torch.full((len(shards) * M, 2), -5, dtype=torch.int32, device="cuda")
        ws = torch.empty(max(sga_lib.sga_lmhead_argmax_workspace(M, wd) for _, wd in shards),
                         dtype=torch.uint8, device="cuda")
        for s, (o, wd) in enumerate(shards):
            sga_lib.sga_lmhead_argmax(h, w[o:o + wd], o, c["org_vocab"], per[s * M:(s + 1) * M], ws)
        one = one_call(sga_lib, h, w, shards, c["org_vocab"])
        gh.assert_stats_equal(one, gh.stats_to_numpy(per))


@pytest.mark.parametrize("M", [1, 16, 64, 100, 130, 300])
@pytest.mark.parametrize("case", ["sixty_four_narrow", "padding_after_first", "tiny_widths"])
def test_one_call_edge_layouts(sga_lib, M, case):
    # the epilogue's per-shard flushes where most CTAs hold tiles of few or no
    # shards: 64 narrow shards (the most one call takes), every shard but the
    # first past org_vocab (no tiles at all), shards narrower than a tile
    H = 128
    if case == "sixty_four_narrow":
        vocab, org = 64 * 300, 64 * 300 - 7
        shards = wl.even_shards(vocab, 64)
    elif case == "padding_after_first":
        vocab, org = 4000, 900
        shards = [(0, 1000), (1000, 1000), (2000, 1000), (3000, 1000)]
    else:
        vocab, org = 500, 500
        shards = [(0, 3), (3, 1), (4, 100), (104, 5), (109, 391)]
    hidden = wl.normal_matrix(M + 31, M, H, 1.0)
    weight = wl.normal_matrix(M + 32, vocab, H, 1.0 / np.sqrt(H))
    per, vals, ids = lm.run_gpu(hidden, weight, shards, org)
    one = one_call(sga_lib, gh.to_device(hidden), gh.to_device(weight), shards, org)
    gh.assert_stats_equal(one, per)
    lm.check_rows(np.arange(0, M, 5), hidden, weight, shards, org, per, vals, ids)


def test_decode_merge_slots_come_back_clean(sga_lib):
    # The decode-size kernel merges its CTAs' winners in one of 32 library-
    # owned slots per call, taken in turn, which the last CTA clears.  Run 80
    # calls in a row (every slot at least twice) over shapes with different
    # shard and row counts -- including an all-padding shard, whose slot keys
    # are never set -- and check each against the per-shard calls' statistics,
    # themselves checked against the oracle: a key a call left behind would
    # change a later result.
    H = 128
    cases = []
    for n in range(8):
        M = [1, 5, 16, 17, 33, 64, 2, 40][n]
        vocab = 900 + 37 * n
        shards = wl.random_shards(n + 101, vocab, 1 + n % 3)
        # even n with several shards: the last shard all padding
        org = vocab - (shards[-1][1] if n % 2 == 0 and len(shards) > 1 else 0)
        hidden = wl.normal_matrix(n + 201, M, H, 1.0)
        weight = wl.normal_matrix(n + 301, vocab, H, 1.0 / np.sqrt(H))
        st, v, i = lm.run_gpu(hidden, weight, shards, org)
        lm.check_rows(np.arange(M), hidden, weight, shards, org, st, v, i)
        cases.append((gh.to_device(hidden), gh.to_device(weight), shards, org, st))
    for k in range(80):
        h, w, sh, org, ref = cases[k % len(cases)]
        gh.assert_stats_equal(one_call(sga_lib, h, w, sh, org), ref)
    assert sga_lib.sga_device_error() == 0


def test_decode_calls_on_concurrent_streams(sga_lib):
    # Decode-size calls issued on four streams at once: each call takes its
    # own merge slot (keys, ticket and tile counter), so calls whose launches
    # overlap on the GPU must not disturb one another.  Every output is
    # compared bit for bit with the same call run alone (itself checked
    # against the oracle on every row).
    H = 512
    cases = []
    for n in range(4):
        M = [16, 3, 48, 100][n]   # one-CTA kernel (N = 16, 16, 64) and CTA pairs
        vocab = 24000 + 1000 * n
        shards = wl.random_shards(n + 401, vocab, 2 + n)
        org = vocab - 37 * n
        hidden = wl.normal_matrix(n + 501, M, H, 1.0)
        weight = wl.normal_matrix(n + 601, vocab, H, 1.0 / np.sqrt(H))
        st, v, i = lm.run_gpu(hidden, weight, shards, org)
        lm.check_rows(np.arange(M), hidden, weight, shards, org, st, v, i)
        h, w = gh.to_device(hidden), gh.to_device(weight)
        ws = torch.empty(max(8, sga_lib.sga_lmhead_argmax_shards_workspace(M, shards)),
                         dtype=torch.uint8, device="cuda")
        cases.append((h, w, shards, org, ws, st))
    streams = [torch.cuda.Stream() for _ in range(4)]
    calls = []
    for k in range(24):
        h, w, sh, org, _, ref = cases[k % len(cases)]
        # each call gets its own (unused at decode sizes) workspace and output,
        # filled on the default stream before the side streams start
        ws = torch.empty(max(8, sga_lib.sga_lmhead_argmax_shards_workspace(h.shape[0], sh)),
                         dtype=torch.uint8, device="cuda")
        out = torch.full((len(sh) * h.shape[0], 2), -5, dtype=torch.int32, device="cuda")
        calls.append((h, w, sh, org, ws, out, ref))
    start = torch.cuda.Event()
    start.record()
    for s in streams:
        s.wait_event(start)
    for k, (h, w, sh, org, ws, out, _) in enumerate(calls):
        sga_lib.sga_lmhead_argmax_shards(h, w, sh, org, out, ws, stream=streams[k % len(streams)])
    for s in streams:
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert sga_lib.sga_device_error() == 0
    for h, w, sh, org, ws, out, ref in calls:
        gh.assert_stats_equal(gh.stats_to_numpy(out), ref)
