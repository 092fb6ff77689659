"""Failure detection without a GPU fault.

Every pipelined kernel in the library waits on mbarriers with a time limit;
when a limit expires the kernel ORs SGA_DEVERR_TIMEOUT into the device error
word and returns, so the CUDA context stays usable.  The self-test entry
point makes exactly such a wait run out (an mbarrier that nothing arrives at)
and the test checks the status and that the device keeps working.  Range
violations inside verify/reduce are covered by the parity tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import gpu_helpers as gh


def test_selftest_rejects_bad_limits_without_a_gpu(sga_lib):
    f = sga_lib.lib().sga_selftest_wait_timeout
    assert f(10, None, None) == -2               # below 1 us
    assert f(2_000_000_000, None, None) == -2    # above 1 s
    assert f(1_000_000, ctypes.c_void_p(0x10004), None) == -6


@pytest.mark.gpu
def test_bounded_wait_expires_sets_error_word_and_context_survives(sga_lib):
    sga_lib.sga_clear_device_error()
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    sga_lib.sga_selftest_wait_timeout(20_000_000, waited)     # 20 ms
    word = sga_lib.sga_device_error()
    assert word & sga_lib.SGA_DEVERR_TIMEOUT
    ns = int(waited.item())
    assert 20_000_000 <= ns < 1_000_000_000
    sga_lib.sga_clear_device_error()
    assert sga_lib.sga_device_error() == 0
    # the context still runs the real path correctly
    c = wl.tiny_sharded_argmax()
    stats = gh.gpu_gathered_stats(gh.to_device(c["logits"]), c["shards"], c["org_vocab"])
    gh.assert_stats_equal(gh.stats_to_numpy(stats),
                          oracle.gathered_stats(c["logits"], c["shards"], c["org_vocab"]))
    assert sga_lib.sga_device_error() == 0
