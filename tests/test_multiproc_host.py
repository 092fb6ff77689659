"""World-size-2 checks of the bench's multi-process host logic on CPU (gloo).

Rows are independent, so N GPUs run N replicas with no data-path collective:
the only cross-rank steps are the barrier around the timed region and the max
over ranks of the elapsed time.  These tests run those steps, and the
reference arm (rank 0 alone prints; the other ranks exit without work), as two
gloo processes on 127.0.0.1.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    import workloads as wl

    bench.init_dist(world, "gloo")
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world, "cpu")

    class Args:
        steps, warmup, gpus, workload = 2, 1, world, "large_verify"
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.run_reference(Args, lambda: wl.large_verify(rows_limit=48))
    bench.barrier(world)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got, "rc": rc, "stdout": buf.getvalue()}, f)


def test_two_rank_barrier_max_and_reference_arm(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert all(r["max"] == 2.5 for r in res)
    assert all(r["rc"] == 0 for r in res)
    assert res[1]["stdout"] == ""                      # only rank 0 prints
    line = json.loads(res[0]["stdout"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "rows/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
