"""GPU parity of sga_lmhead_argmax_fp8 (E4M3 operands, tcgen05 kind::f8f6f4)
against the oracle's exact fp64 logits of the decoded codes times the scales.

Same tolerance as the bf16 LM head: ids equal where the oracle's top-1 minus
top-2 gap exceeds GAP (elsewhere a near-winner), values within REL (ABS floor).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh

pytestmark = pytest.mark.gpu

GAP, REL, ABS = 1e-2, 1e-2, 1e-3


def u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def run_gpu(sga, hq, hs, wq, w_scale, shards, org_vocab):
    M = hq.shape[0]
    h = u8(hq)
    w = u8(wq)
    hs_d = None if hs is None else torch.from_numpy(np.ascontiguousarray(hs, np.float32)).cuda()
    stats = torch.full((len(shards) * M, 2), -5, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(8, max(sga.sga_lmhead_argmax_workspace(M, wd) for _, wd in shards)),
                     dtype=torch.uint8, device="cuda")
    for s, (o, wd) in enumerate(shards):
        sga.sga_lmhead_argmax_fp8(h, hs_d, w[o:o + wd], w_scale, o, org_vocab,
                                  stats[s * M:(s + 1) * M], ws)
    ids = torch.empty(M, dtype=torch.int32, device="cuda")
    vals = torch.empty(M, dtype=torch.float32, device="cuda")
    sga.sga_shard_reduce(stats, len(shards), M, ids, vals)
    assert sga.sga_device_error() == 0
    return gh.stats_to_numpy(stats), vals.cpu().numpy(), ids.cpu().numpy()


def check(rows, hq, hs, wq, w_scale, shards, org_vocab, st, vals, ids):
    M = hq.shape[0]
    scale = np.ones(M, np.float32) if hs is None else hs
    logits = oracle.lmhead_logits_fp8(hq, scale, wq, w_scale, rows)
    top1, top2, exp_ids = oracle.argmax_f64(logits, 0, org_vocab)
    checked = 0
    for q, r in enumerate(rows):
        gi, gv = int(ids[r]), float(vals[r])
        if np.isnan(top1[q]):
            assert gi == exp_ids[q] and np.isnan(gv)
            continue
        if top1[q] - top2[q] > GAP:
            assert gi == exp_ids[q], (r, gi, exp_ids[q], top1[q], top2[q])
            checked += 1
        else:
            assert logits[q, gi] >= top1[q] - GAP
        assert abs(gv - top1[q]) <= max(REL * abs(top1[q]), ABS), (r, gv, top1[q])
        for s, (o, wd) in enumerate(shards):
            sv = st[s * M + r]
            s1, s2, sid = oracle.argmax_f64(logits[q:q + 1, o:o + wd], o, org_vocab)
            if s1[0] == -np.inf:
                assert sv["id"] == o and sv["v"] == -np.inf
                continue
            if s1[0] - s2[0] > GAP:
                assert sv["id"] == sid[0]
            assert abs(float(sv["v"]) - s1[0]) <= max(REL * abs(s1[0]), ABS)
    return checked


def make(M, H, vocab, seed):
    hq, hs = wl.quantize_rows_e4m3(wl.normal_matrix(seed, M, H, 1.0, dtype="f32"))
    wq, w_scale = wl.quantize_tensor_e4m3(
        wl.normal_matrix(seed + 1, vocab, H, 1.0 / np.sqrt(H), dtype="f32"))
    return hq, hs, wq, float(w_scale)


@pytest.mark.parametrize("M,H,vocab,num_shards", [
    (1, 128, 300, 1), (100, 256, 1000, 2), (128, 512, 5000, 3), (300, 256, 2311, 4),
    (513, 1024, 4099, 2), (16, 4096, 20000, 2),
    # decode kernel with 16, 32 and 64 hidden columns, and its CTA-pair form
    (7, 256, 3001, 3), (33, 512, 3001, 2), (64, 256, 1000, 3), (5, 384, 2000, 2),
    (65, 384, 3001, 3), (127, 128, 4099, 2),
])
def test_small_shapes(sga_lib, M, H, vocab, num_shards):
    hq, hs, wq, w_scale = make(M, H, vocab, M + H + vocab)
    shards = wl.random_shards(M + vocab, vocab, num_shards) if num_shards > 1 else [(0, vocab)]
    for org in (vocab, vocab - 29):
        st, v, i = run_gpu(sga_lib, hq, hs, wq, w_scale, shards, org)
        check(np.arange(M), hq, hs, wq, w_scale, shards, org, st, v, i)


@pytest.mark.parametrize("M", [200, 100, 40, 12])
def test_no_row_scales_and_nan_code(sga_lib, M):
    H, vocab = 256, 700
    hq, _, wq, w_scale = make(M, H, vocab, 9)
    wq = wq.copy()
    wq[333, 17] = 0x7F                                 # E4M3 NaN in weight row 333
    shards = [(0, 300), (300, 400)]
    st, v, i = run_gpu(sga_lib, hq, None, wq, w_scale, shards, vocab)
    assert (i == 333).all() and np.isnan(v).all()      # the NaN logit wins every row
    st, v, i = run_gpu(sga_lib, hq, None, wq, w_scale, shards, 333)   # ...unless padded
    check(np.arange(0, M, 3), hq, None, wq, w_scale, shards, 333, st, v, i)
