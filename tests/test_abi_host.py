"""Host-side checks of the C ABI (no GPU needed, no compute call made).

The library must load, export every function include/sga.h declares, and
reject bad arguments with the documented status before touching CUDA.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sga.h")

BAD_F32 = ctypes.c_void_p(0x1002)  # not 4-byte aligned; never dereferenced
FAKE = ctypes.c_void_p(0x10000)    # aligned; never dereferenced


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sga_\w+)\s*\(", text)))


def test_header_declares_the_path(sga_lib):
    names = declared_functions()
    for n in ("sga_local_argmax", "sga_shard_reduce", "sga_greedy_verify", "sga_lmhead_argmax"):
        assert n in names


def test_library_exports_every_declared_symbol(sga_lib):
    L = sga_lib.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(sga_lib):
    assert sga_lib.sga_version() == 100
    texts = {sga_lib.sga_status_string(s) for s in range(0, -12, -1)}
    assert len(texts) == 12 and all(texts)
    assert sga_lib.sga_status_string(-99) == "unknown status"


def test_local_argmax_validation(sga_lib):
    f = sga_lib.lib().sga_local_argmax
    ok = dict(logits=FAKE, dtype=1, rows=4, ld=10, start=0, width=10, org=10, out=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["logits"], a["dtype"], a["rows"], a["ld"], a["start"], a["width"], a["org"],
                 a["out"], None)

    assert call(dtype=7) == -5
    assert call(rows=-1) == -2
    assert call(width=0) == -3
    assert call(start=-1) == -3
    assert call(ld=9) == -3
    assert call(org=0) == -4
    assert call(start=(1 << 24) - 5) == -4
    assert call(rows=0) == 0            # empty batch: nothing enqueued
    assert call(logits=None) == -1
    assert call(out=None) == -1
    assert call(dtype=0, logits=BAD_F32) == -6
    assert call(out=ctypes.c_void_p(0x10004)) == -6


def test_shard_reduce_and_verify_validation(sga_lib):
    L = sga_lib.lib()
    assert L.sga_shard_reduce(FAKE, 0, 4, FAKE, FAKE, None, 0, None) == -2
    assert L.sga_shard_reduce(FAKE, 2, -1, FAKE, FAKE, None, 0, None) == -2
    assert L.sga_shard_reduce(FAKE, 2, 0, FAKE, FAKE, None, 0, None) == 0
    assert L.sga_shard_reduce(None, 2, 4, FAKE, FAKE, None, 0, None) == -1
    assert L.sga_shard_reduce(FAKE, 2, 4, None, ctypes.c_void_p(0x10002), None, 0, None) == -6
    v = L.sga_greedy_verify
    assert v(FAKE, 2, 3, FAKE, FAKE, 0, FAKE, FAKE, FAKE, FAKE, None, None) == -8
    assert v(FAKE, 2, 3, FAKE, FAKE, 16, FAKE, FAKE, FAKE, FAKE, None, None) == -8
    assert v(FAKE, 0, 3, FAKE, FAKE, 3, FAKE, FAKE, FAKE, FAKE, None, None) == -2
    assert v(FAKE, 2, -1, FAKE, FAKE, 3, FAKE, FAKE, FAKE, FAKE, None, None) == -2
    assert v(FAKE, 2, 0, FAKE, FAKE, 3, FAKE, FAKE, FAKE, FAKE, None, None) == 0
    assert v(FAKE, 2, 3, None, FAKE, 3, FAKE, FAKE, FAKE, FAKE, None, None) == -1
    assert v(FAKE, 2, 3, FAKE, FAKE, 3, FAKE, FAKE, FAKE, ctypes.c_void_p(0x10001), None, None) == -6


def test_lmhead_validation(sga_lib):
    L = sga_lib.lib()
    ws = L.sga_lmhead_argmax_workspace(512, 75968)
    assert ws >= 512 * 8
    f = L.sga_lmhead_argmax
    assert f(FAKE, 512, 100, FAKE, 0, 64, 64, FAKE, FAKE, ws, None) == -2   # H % 64
    assert f(FAKE, -1, 64, FAKE, 0, 64, 64, FAKE, FAKE, ws, None) == -2
    assert f(FAKE, 0, 64, FAKE, 0, 64, 64, FAKE, FAKE, ws, None) == 0
    assert f(ctypes.c_void_p(0x10008), 4, 64, FAKE, 0, 64, 64, FAKE, FAKE, ws, None) == -6
    assert f(FAKE, 512, 64, FAKE, 0, 75968, 75968, FAKE, FAKE, ws - 8, None) == -7
    assert f(FAKE, 4, 64, FAKE, 0, 64, 0, FAKE, FAKE, ws, None) == -4


def test_lmhead_shards_validation(sga_lib):
    L = sga_lib.lib()

    def arr(v):
        return (ctypes.c_int64 * len(v))(*v)

    wsf = L.sga_lmhead_argmax_shards_workspace
    assert wsf(16, 2, arr([75968, 75968])) == 2 * 16 * 256 * 8   # decode sizes: one launch
    # M >= 129: one 2-SM launch for both shards, one partial per (shard, row,
    # chunk), at most min(128, tiles of all shards) chunks
    assert wsf(512, 2, arr([75968, 1000])) == 2 * 512 * 128 * 8
    assert wsf(512, 2, arr([256, 300])) == 2 * 512 * 3 * 8          # 1 + 2 tiles
    # 65 <= M <= 128: decode sizes too (one CTA-pair launch), sized as below 65
    assert wsf(100, 2, arr([75968, 1000])) == 2 * 100 * 256 * 8
    assert L.sga_lmhead_argmax_workspace(100, 75968) == 100 * 297 * 8
    assert L.sga_lmhead_argmax_workspace(512, 75968) == 512 * 128 * 8
    assert wsf(16, 0, arr([1])) == 0 and wsf(16, 65, None) == 0 and wsf(16, 1, arr([0])) == 0
    ws = wsf(16, 2, arr([64, 64]))
    f = L.sga_lmhead_argmax_shards

    def call(starts, widths, M=16, H=64, org=128, hidden=FAKE, weight=FAKE, out=FAKE,
             work=FAKE, nbytes=ws):
        return f(hidden, M, H, weight, len(starts), arr(starts), arr(widths), org, out, work,
                 nbytes, None)

    assert call([0, 40], [64, 64]) == -3                        # overlap
    assert call([0, 64], [64, 0]) == -3                         # empty shard
    assert call([0, 64], [64, 64], H=100) == -2                 # H % 64
    assert call([0, 64], [64, 64], M=-1) == -2
    assert call([0, 64], [64, 64], M=0) == 0
    assert call([0, 64], [64, 64], weight=None) == -1
    assert call([0, 64], [64, 64], weight=ctypes.c_void_p(0x10008)) == -6
    assert call([0, 64], [64, 64], nbytes=ws - 8) == -7
    assert call([0, 64], [64, 64], org=0) == -4
    assert f(FAKE, 16, 64, FAKE, 0, None, None, 128, FAKE, FAKE, ws, None) == -2
    assert f(FAKE, 16, 64, FAKE, 65, None, None, 128, FAKE, FAKE, ws, None) == -2
    assert f(FAKE, 16, 64, FAKE, 2, None, None, 128, FAKE, FAKE, ws, None) == -1
    g = L.sga_lmhead_argmax_shards_fp8
    a0, a1 = arr([0, 128]), arr([128, 128])
    assert g(FAKE, None, 16, 128, FAKE, 0.0, 2, a0, a1, 256, FAKE, FAKE, ws, None) == -2
    assert g(FAKE, None, 16, 64, FAKE, 1.0, 2, a0, a1, 256, FAKE, FAKE, ws, None) == -2
    assert g(FAKE, BAD_F32, 16, 128, FAKE, 1.0, 2, a0, a1, 256, FAKE, FAKE, ws, None) == -6


def test_missing_library_fails_loudly(monkeypatch, sga_lib):
    monkeypatch.setattr(sga_lib, "_lib", None)
    monkeypatch.setattr(sga_lib, "LIB_PATH", os.path.join(ROOT, "nonexistent", "libsga.so"))
    with pytest.raises(RuntimeError, match="missing"):
        sga_lib.lib()


def test_local_argmax_shards_validation(sga_lib):
    f = sga_lib.lib().sga_local_argmax_shards

    def call(starts, widths, rows=4, ld=100, org=100, dtype=1, logits=FAKE, out=FAKE):
        n = len(starts)
        st = (ctypes.c_int64 * n)(*starts)
        wd = (ctypes.c_int64 * n)(*widths)
        return f(logits, dtype, rows, ld, n, st, wd, org, out, None)

    assert call([0, 40], [50, 50]) == -3          # overlap
    assert call([0, 50], [50, 60]) == -3          # past ld
    assert call([0, 50], [50, 0]) == -3           # empty shard
    assert call([0], [100], dtype=3) == -5
    assert call([0], [100], rows=-1) == -2
    assert call([0], [100], rows=0) == 0
    assert call([0], [100], logits=None) == -1
    assert f(FAKE, 1, 4, 100, 0, None, None, 100, FAKE, None) == -2
    assert f(FAKE, 1, 4, 100, 65, None, None, 100, FAKE, None) == -2
    assert f(FAKE, 1, 4, 100, 2, None, None, 100, FAKE, None) == -1


def test_fp8_validation(sga_lib):
    f = sga_lib.lib().sga_lmhead_argmax_fp8
    fake = FAKE
    ws = 1 << 20
    assert f(fake, None, 4, 192, fake, 1.0, 0, 64, 64, fake, fake, ws, None) == -2   # H % 128
    assert f(fake, None, 4, 128, fake, 0.0, 0, 64, 64, fake, fake, ws, None) == -2   # scale
    assert f(fake, None, 4, 128, fake, -1.0, 0, 64, 64, fake, fake, ws, None) == -2
    assert f(fake, ctypes.c_void_p(0x10002), 4, 128, fake, 1.0, 0, 64, 64, fake, fake, ws,
             None) == -6


def test_block_slots_and_block_argmax_validation(sga_lib):
    L = sga_lib.lib()
    slots = L.sga_block_slots
    assert slots(0, 67350, 8192, 1024) == 66            # 1024-blocks 0..65
    assert slots(67350, 67349, 8192, 1024) == 67         # blocks 65..131
    assert slots(67350, 67349, 8192, 8192) == 9          # blocks 8..16
    assert slots(2, 2, 2, 3) == 2                        # 3 does not nest in 2
    assert slots(5, 10, 1 << 20, 1 << 20) == 1
    assert slots(0, 10, 0, 4) == -2 and slots(0, 10, 4, (1 << 24) + 1) == -2
    assert slots(-1, 10, 4, 4) == -3 and slots(0, 0, 4, 4) == -3
    assert sga_lib.sga_block_slots(0, 67350, 8192) == 9
    with pytest.raises(sga_lib.SgaError):
        sga_lib.sga_block_slots(0, 10, 0)
    f = L.sga_local_argmax_blocks
    ok = dict(logits=FAKE, dtype=1, rows=4, ld=100, start=0, width=100, org=100, db=16, bb=4,
              n=0, cu=None, out=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["logits"], a["dtype"], a["rows"], a["ld"], a["start"], a["width"], a["org"],
                 a["db"], a["bb"], a["n"], a["cu"], a["out"], None)

    assert call(dtype=2) == -5
    assert call(db=0) == -2 and call(bb=-4) == -2
    assert call(rows=-1) == -2
    assert call(rows=1 << 27) == -2                      # rows * 25 slots > 2^28
    assert call(width=0) == -3 and call(ld=99) == -3
    assert call(org=0) == -4
    assert call(cu=FAKE, n=0) == -2                      # a request layout needs requests
    assert call(rows=0) == 0
    assert call(logits=None) == -1 and call(out=None) == -1
    assert call(dtype=0, logits=BAD_F32) == -6
    assert call(cu=ctypes.c_void_p(0x10002), n=2) == -6


def test_block_shards_validation(sga_lib):
    f = sga_lib.lib().sga_local_argmax_blocks_shards

    def call(starts, widths, rows=4, ld=100, org=100, dtype=1, db=16, bb=4, n=0, cu=None,
             logits=FAKE, out=FAKE):
        k = len(starts)
        st = (ctypes.c_int64 * k)(*starts)
        wd = (ctypes.c_int64 * k)(*widths)
        return f(logits, dtype, rows, ld, k, st, wd, org, db, bb, n, cu, out, None)

    assert call([0, 40], [50, 50]) == -3          # overlap
    assert call([0, 50], [50, 60]) == -3          # past ld
    assert call([0, 50], [50, 0]) == -3           # empty shard
    assert call([0], [100], dtype=3) == -5
    assert call([0], [100], db=0) == -2
    assert call([0, 50], [50, 50], rows=1 << 25) == -2   # rows x slots > 2^28
    assert call([0], [100], cu=FAKE, n=0) == -2
    assert call([0], [100], rows=0) == 0
    assert call([0], [100], logits=None) == -1
    assert f(FAKE, 1, 4, 100, 0, None, None, 100, 16, 4, 0, None, FAKE, None) == -2
    assert f(FAKE, 1, 4, 100, 65, None, None, 100, 16, 4, 0, None, FAKE, None) == -2
    assert f(FAKE, 1, 4, 100, 2, None, None, 100, 16, 4, 0, None, FAKE, None) == -1


def test_valid_call_without_a_gpu_returns_the_cuda_status(sga_lib):
    # every argument valid, but no device: the status is SGA_ERR_CUDA and
    # nothing is dereferenced.  Only where no GPU is visible (with one, the
    # fake pointers would reach a kernel).
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    L = sga_lib.lib()
    assert L.sga_local_argmax(FAKE, 1, 4, 100, 0, 100, 100, FAKE, None) == -9
    assert L.sga_shard_reduce(FAKE, 2, 4, None, FAKE, None, 0, None) == -9
    assert L.sga_lmhead_argmax(FAKE, 4, 64, FAKE, 0, 64, 64, FAKE, FAKE,
                               L.sga_lmhead_argmax_workspace(4, 64), None) == -9
    word = ctypes.c_uint32(7)
    assert L.sga_device_error(ctypes.byref(word)) == -9
