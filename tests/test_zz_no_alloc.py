"""GPU test of sga_lmhead_argmax_noalloc, the LM-head argmax entry point that
allocates nothing.

Some callers cannot give the library a workspace: a serving process or
framework plugin whose device memory pool is sized once at start-up and which
may not call cudaMalloc afterwards, or a decode loop where an allocation would
synchronise the device.  For them the library keeps the partial statistics in
a fixed scratch array of its own.  This test calls that entry point through
the C ABI twice in a row, with different shapes (so the second call finds the
first call's leftovers in the shared scratch), and checks each result against
the workspace entry point sga_lmhead_argmax with the tolerance the LM-head
parity tests use (ids equal, values within 1e-2 relative).  It also checks
that a call needing more than the 4 MiB scratch is refused.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

REL, ABS = 1e-2, 1e-3


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def test_noalloc_matches_workspace_entry_point_twice(sga_lib):
    L = sga_lib.lib()
    fn = L.sga_lmhead_argmax_noalloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [vp, i64, i64, vp, i64, i64, i64, vp, vp]
    fn.restype = ctypes.c_int
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [(300, 256, 3000, 1200, 2950), (200, 512, 1500, 0, 1500)]
    for M, H, width, start, org in cases:
        hidden = _dev(wl.normal_matrix(M + 1, M, H, 1.0))
        weight = _dev(wl.normal_matrix(width + 2, width, H, 1.0 / np.sqrt(H)))
        ref = torch.full((M, 2), -3, dtype=torch.int32, device="cuda")
        ws = torch.empty(sga_lib.sga_lmhead_argmax_workspace(M, width), dtype=torch.uint8,
                         device="cuda")
        sga_lib.sga_lmhead_argmax(hidden, weight, start, org, ref, ws)
        got = torch.full((M, 2), -4, dtype=torch.int32, device="cuda")
        st = fn(vp(hidden.data_ptr()), M, H, vp(weight.data_ptr()), start, width, org,
                vp(got.data_ptr()), stream)
        assert st == 0, sga_lib.sga_status_string(st)
        torch.cuda.synchronize()
        gv, gi = sga_lib.stat_values(got).cpu().numpy(), sga_lib.stat_ids(got).cpu().numpy()
        rv, ri = sga_lib.stat_values(ref).cpu().numpy(), sga_lib.stat_ids(ref).cpu().numpy()
        assert (gi == ri).all()
        assert (np.abs(gv - rv) <= np.maximum(REL * np.abs(rv), ABS)).all()
        assert ((ri >= start) & (ri < min(org, start + width))).all()
    assert sga_lib.sga_device_error() == 0


def test_noalloc_refuses_more_than_its_scratch(sga_lib):
    fn = sga_lib.lib().sga_lmhead_argmax_noalloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [vp, i64, i64, vp, i64, i64, i64, vp, vp]
    fn.restype = ctypes.c_int
    fake = vp(0x10000)   # never dereferenced: the size check comes first
    # 4096 rows x ceil(200000/256) tiles x 8 bytes = 25.6 MB > 4 MiB
    assert fn(fake, 4096, 4096, fake, 0, 200000, 200000, fake, None) == -7
