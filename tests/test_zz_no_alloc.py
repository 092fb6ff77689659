"""GPU test of sga_lmhead_argmax_noalloc, the LM-head argmax entry point that
allocates nothing.

Some callers cannot give the library a workspace: a serving process or
framework plugin whose device memory pool is sized once at start-up and which
may not call cudaMalloc afterwards, or a decode loop where an allocation would
synchronise the device.  For them the library keeps the partial statistics in
a fixed scratch array of its own.

The test calls that entry point through the C ABI on several shapes in a row
-- 2-SM GEMM sizes first, then decode sizes (M <= 128, whose kernels merge
in library-owned memory and leave the scratch alone) -- so that each call
finds the previous call's leftovers in the shared scratch.  Each result
must equal the workspace entry point sga_lmhead_argmax bit for bit (the same
kernels run), and must agree with the CPU oracle's fp64 logits under the
LM-head tolerance (ids equal where the oracle's top-1 minus top-2 exceeds
1e-2, else a near-winner; values within 1e-2 relative).  One call goes through
the Python wrapper.  A call needing more than the 4 MiB scratch is refused.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

GAP, REL, ABS = 1e-2, 1e-2, 1e-3

# (M, H, shard width, shard start, org_vocab): 2-SM GEMM sizes, then decode sizes
# (one CTA per SM up to M = 64, CTA pairs above)
CASES = [(300, 256, 3000, 1200, 2950), (200, 512, 1500, 0, 1500),
         (16, 256, 2000, 512, 2500), (1, 128, 700, 0, 650), (64, 256, 5000, 100, 5100),
         (100, 256, 3000, 640, 3500)]


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _fn(sga_lib):
    fn = sga_lib.lib().sga_lmhead_argmax_noalloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [vp, i64, i64, vp, i64, i64, i64, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def check_against_oracle(hidden, weight, start, org, vals, ids):
    """Per row: the oracle's argmax over the shard's ids below org_vocab."""
    M = hidden.shape[0]
    logits = oracle.lmhead_logits(hidden, weight, np.arange(M, dtype=np.int64))
    top1, top2, exp = oracle.argmax_f64(logits, start, org)
    for r in range(M):
        gi = int(ids[r])
        assert start <= gi < min(org, start + weight.shape[0]), (r, gi)
        if top1[r] - top2[r] > GAP:
            assert gi == exp[r], (r, gi, exp[r], top1[r], top2[r])
        else:
            assert logits[r, gi - start] >= top1[r] - GAP, (r, gi, top1[r])
        assert abs(float(vals[r]) - top1[r]) <= max(REL * abs(top1[r]), ABS), (r, vals[r], top1[r])


def test_noalloc_matches_workspace_entry_point_and_oracle(sga_lib):
    fn = _fn(sga_lib)
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    for n, (M, H, width, start, org) in enumerate(CASES):
        hidden = wl.normal_matrix(M + 1, M, H, 1.0)
        weight = wl.normal_matrix(width + 2, width, H, 1.0 / np.sqrt(H))
        h, w = _dev(hidden), _dev(weight)
        ref = torch.full((M, 2), -3, dtype=torch.int32, device="cuda")
        ws = torch.empty(sga_lib.sga_lmhead_argmax_workspace(M, width), dtype=torch.uint8,
                         device="cuda")
        sga_lib.sga_lmhead_argmax(h, w, start, org, ref, ws)
        got = torch.full((M, 2), -4, dtype=torch.int32, device="cuda")
        if n == len(CASES) - 1:
            sga_lib.sga_lmhead_argmax_noalloc(h, w, start, org, got)   # the Python wrapper
        else:
            st = fn(vp(h.data_ptr()), M, H, vp(w.data_ptr()), start, width, org,
                    vp(got.data_ptr()), stream)
            assert st == 0, sga_lib.sga_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), (M, H, width)   # same kernels: bit-identical
        check_against_oracle(hidden, weight, start, org, sga_lib.stat_values(got).cpu().numpy(),
                             sga_lib.stat_ids(got).cpu().numpy())
    assert sga_lib.sga_device_error() == 0


def test_noalloc_refuses_more_than_its_scratch(sga_lib):
    fn = _fn(sga_lib)
    vp = ctypes.c_void_p
    fake = vp(0x10000)   # never dereferenced: the size check comes first
    # the limit is sga_lmhead_argmax_workspace(M, width) <= 4 MiB
    assert sga_lib.sga_lmhead_argmax_workspace(8192, 200000) > (4 << 20)
    assert fn(fake, 8192, 4096, fake, 0, 200000, 200000, fake, None) == -7
    # decode sizes count up to 256 partials per row: 64 rows x 256 x 8 B = 128 KiB fits
    assert sga_lib.sga_lmhead_argmax_workspace(64, 200000) <= (4 << 20)
