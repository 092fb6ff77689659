"""Benchmark of the sharded greedy token-selection hot path on GB300.

One step = one pass of the whole path over one batch: sga_local_argmax for
every vocab shard (tensor-parallel ranks emulated as vocab slices of one
logits matrix, stats written in shard order as all_gather(dim=0) would) and
the fused sga_greedy_verify.  Default workload: 256 requests x (15 drafts + 1
bonus) = 4096 rows x vocab 202048 bf16 N(0,3), 3 uneven shards, 1% planted
cross-shard-edge ties, drafts copying the target w.p. 0.6 (synthetic; the
inputs, 1.66 GB, are larger than the 129 MB L2, so no flush is needed).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload large_verify|lmhead|...] [--tp]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own batch
(rows are independent: weak scaling, no data-path collective); the barrier
and the max-over-ranks time use torch.distributed.  The default line also
carries nested records of the other configurations: the fused LM head
(`lmhead`) and the two L2-resident latency workloads.  --tp runs the
tensor-parallel form instead: rank r holds vocab shard r only and the
statistics are all-gathered (NCCL) every step (strong scaling).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "logit rows/s and achieved HBM GB/s (frac of roofline) for sharded argmax+verify"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["large_verify", "large_verify_blocks", "lmhead",
                                          "lmhead_fp8", "draft_top_tokens", "greedy_verify"],
                   default="large_verify")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--tp", action="store_true",
                   help="tensor-parallel form of the default step: rank r of N holds vocab "
                        "shard r only, statistics all-gathered (NCCL) every step")
    p.add_argument("--no-extra", action="store_true",
                   help="default workload: leave out the nested records of the fused LM head "
                        "and the two small latency workloads")
    p.add_argument("--graph", action="store_true",
                   help="lmhead, draft_top_tokens and greedy_verify workloads: replay each "
                        "step from a CUDA graph and time the whole step (no per-launch events)")
    p.add_argument("--lmhead-rows", type=int, default=512,
                   help="rows (hidden states) of the fused LM-head workload")
    p.add_argument("--lmhead-per-shard", action="store_true",
                   help="lmhead workloads: one sga_lmhead_argmax call per shard (each "
                        "emulated rank its own) instead of every shard through one "
                        "sga_lmhead_argmax_shards call (one decode-size launch for M <= 128)")
    p.add_argument("--lmhead-shards", type=int, default=2,
                   help="vocab shards (emulated TP ranks) of the fused LM-head workload")
    p.add_argument("--lmhead-vocab", type=int, default=151936,
                   help="vocab of the fused LM-head workload (smaller for profiling)")
    p.add_argument("--mixed-k", action="store_true",
                   help="large_verify workloads: 256 requests with K_i uniform in 1..15 "
                        "instead of K = 15 for all")
    p.add_argument("--rows", type=int, default=None,
                   help="keep only the first rows (whole requests) of the workload; "
                        "for small profiling captures")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def source_digest(*rel_paths):
    h = hashlib.sha256()
    for rel in rel_paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(profile_name, kernel_sources, key="dram_bytes_per_launch"):
    """DRAM bytes per launch recorded by an ncu capture in profiles/ (the
    field `key`), or None when the kernel source changed since that capture."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.strip().startswith("- "):
                    k, v = line.strip()[2:].split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("source_digest") != source_digest(*kernel_sources):
            return None
        return float(fields[key])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# process group (torchrun) helpers: barrier and max over ranks only
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the device path (our kernels through the binding)
# ---------------------------------------------------------------------------

class VerifyPath:
    """Device buffers and one step of the large-verify path."""

    def __init__(self, c, torch, sga, blocks=None):
        self.torch, self.sga = torch, sga
        self.rows = c["logits"].shape[0]
        self.shards = c["shards"]
        self.org = c["org_vocab"]
        self.k = c["k"]
        self.cu_host = c["cu_num_draft"]
        self.n = self.cu_host.size - 1
        self.x = torch.from_numpy(c["logits"].view(np.int16)).view(torch.bfloat16).cuda()
        # blocks = (draft_block, bonus_block): block-granular stats, one
        # sga_local_argmax_blocks launch per shard; else one stat per shard
        self.blocks = blocks
        self.slots = ([sga.sga_block_slots(o, w, *blocks) for o, w in self.shards] if blocks
                      else [1] * len(self.shards))
        self.n_stats = sum(self.slots)
        self.stats = sga.new_stats(self.n_stats * self.rows)
        self.cu = torch.from_numpy(self.cu_host).cuda()
        # drafts: copy the target's greedy token where the plan says so; the
        # target tokens come from one untimed pass of the device path
        t = torch.empty(self.rows, dtype=torch.int32, device="cuda")
        self.run_argmax()
        sga.sga_shard_reduce(self.stats, self.n_stats, self.rows, t)
        self.drafts_host = wl.compose_drafts(t.cpu().numpy(), self.cu_host, c["flags"], c["rand_ids"])
        self.drafts = torch.from_numpy(self.drafts_host).cuda()
        i32 = dict(dtype=torch.int32, device="cuda")
        self.sampled = torch.empty((self.n, self.k + 1), **i32)
        self.num_sampled = torch.empty(self.n, **i32)
        self.num_rejected = torch.empty(self.n, **i32)
        self.bonus = torch.empty(self.n, **i32)
        self.launches_per_step = 2
        elt = 2
        self.argmax_bytes = [self.rows * (w * elt + 8 * n) for (_, w), n in zip(self.shards, self.slots)]
        self.step_bytes = (sum(self.argmax_bytes) + 8 * self.n_stats * self.rows
                           + 4 * int(self.cu_host[-1]) + 4 * (self.n + 1)
                           + 4 * self.n * (self.k + 1) + 12 * self.n)

    def run_argmax(self):
        """All shards of this GPU in one launch (sga_local_argmax_shards, or
        sga_local_argmax_blocks_shards for block statistics)."""
        if self.blocks:
            self.sga.sga_local_argmax_blocks_shards(
                self.x, self.shards, self.org, self.blocks[0], self.stats,
                bonus_block=self.blocks[1], cu_num_draft=self.cu)
        else:
            self.sga.sga_local_argmax_shards(self.x, self.shards, self.org, self.stats)

    def run_argmax_per_shard(self):
        """One launch per shard, as separate tensor-parallel ranks would."""
        off = 0
        for (o, w), n in zip(self.shards, self.slots):
            out = self.stats[off * self.rows:(off + n) * self.rows]
            if self.blocks:
                self.sga.sga_local_argmax_blocks(self.x[:, o:o + w], o, w, self.org,
                                                 self.blocks[0], out, bonus_block=self.blocks[1],
                                                 cu_num_draft=self.cu)
            else:
                self.sga.sga_local_argmax(self.x[:, o:o + w], o, w, self.org, out)
            off += n

    def run_verify(self):
        self.sga.sga_greedy_verify(self.stats, self.n_stats, self.cu, self.drafts, self.k,
                                   self.sampled, self.num_sampled, self.num_rejected, self.bonus)

    def step(self):
        self.run_argmax()
        self.run_verify()

    def step_per_shard(self):
        self.run_argmax_per_shard()
        self.run_verify()


GRAPH_STEPS = 10   # steps per captured CUDA graph in the timed loop


def time_device_steps(path, steps, warmup, torch, world, rank):
    """K steps back to back between two events (no event between the
    kernels, so each launch overlaps the previous one's tail through
    programmatic dependent launch).  The steps are replayed from a CUDA graph
    of GRAPH_STEPS steps (the remainder of K launched directly): every
    launch still runs, and the timed loop does not depend on how fast the
    host can submit (eager submission measured the same 225 us step on an
    idle host, and 13 % longer steps on one busy host)."""
    for _ in range(warmup):
        path.step()
    torch.cuda.synchronize()
    g_steps = min(GRAPH_STEPS, steps)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(g_steps):
            path.step()
    graph.replay()   # untimed
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.3)
    start.record()
    for _ in range(steps // g_steps):
        graph.replay()
    for _ in range(steps % g_steps):
        path.step()
    end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    del graph
    return start.elapsed_time(end), clocks


def time_launches(fn, n, torch):
    """n launches of fn, each between its own pair of events on the current
    stream (the events keep launches apart); returns the per-launch
    durations in ms.  Before each pair the stream runs a short GPU-side
    sleep, so the host has enqueued the events and the launch before the
    first event runs: the interval holds the kernel, not host launch
    latency."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    for a, b in ev:
        torch.cuda._sleep(100000)   # ~50 us of GPU time, outside the interval
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def spread(ms_list):
    """median / min / max in microseconds of per-launch durations."""
    us = sorted(t * 1e3 for t in ms_list)
    return {"launches": len(us), "median_us": round(statistics.median(us), 2),
            "min_us": round(us[0], 2), "max_us": round(us[-1], 2)}


def time_per_shard_steps(path, steps, torch):
    """The same step with one argmax launch per shard (emulated ranks)."""
    for _ in range(3):
        path.step_per_shard()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        path.step_per_shard()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


E2E_REPEATS = 3   # e2e loops per figure; the median is reported


def time_e2e(path, c, steps, torch):
    """Same metric through the public API with host buffers: every step
    copies the step's inputs from pinned host memory to the device and reads
    the results back.  Returns the median over E2E_REPEATS loops of `steps`
    steps (the host memory and link are shared with the machine's other
    jobs) and every loop's ms per step."""
    logits_h = torch.from_numpy(c["logits"].view(np.int16)).pin_memory()
    drafts_h = torch.from_numpy(path.drafts_host).pin_memory()
    cu_h = torch.from_numpy(path.cu_host).pin_memory()
    outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory()
              for t in (path.sampled, path.num_sampled, path.num_rejected, path.bonus)]
    x_i16 = path.x.view(torch.int16)

    def one():
        x_i16.copy_(logits_h, non_blocking=True)
        path.drafts.copy_(drafts_h, non_blocking=True)
        path.cu.copy_(cu_h, non_blocking=True)
        path.step()
        for h, d in zip(outs_h, (path.sampled, path.num_sampled, path.num_rejected, path.bonus)):
            h.copy_(d, non_blocking=True)

    one()
    torch.cuda.synchronize()
    loops = []
    for _ in range(E2E_REPEATS):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(steps):
            one()
        end.record()
        torch.cuda.synchronize()
        loops.append(start.elapsed_time(end) / steps)
    h2d = logits_h.numel() * 2 + drafts_h.numel() * 4 + cu_h.numel() * 4
    d2h = sum(h.numel() * 4 for h in outs_h)
    return statistics.median(loops), h2d, d2h, loops


def time_e2e_pipelined(paths, c, steps, torch):
    """The same end-to-end step with two device buffer sets: while step i runs
    on one set (compute stream), step i+1's inputs are copied from pinned
    host memory into the other (copy stream), as a serving loop overlaps the
    next batch's transfer with the current batch.  Every step still copies its
    inputs in and its results out."""
    logits_h = torch.from_numpy(c["logits"].view(np.int16)).pin_memory()
    drafts_h = torch.from_numpy(paths[0].drafts_host).pin_memory()
    cu_h = torch.from_numpy(paths[0].cu_host).pin_memory()
    outs = [(p.sampled, p.num_sampled, p.num_rejected, p.bonus) for p in paths]
    outs_h = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in o] for o in outs]
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    loaded = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(i):
        p = paths[i % 2]
        with torch.cuda.stream(copy_s):
            if i >= 2:
                copy_s.wait_event(freed[i % 2])   # step i-2 is done with this set
            p.x.view(torch.int16).copy_(logits_h, non_blocking=True)
            p.drafts.copy_(drafts_h, non_blocking=True)
            p.cu.copy_(cu_h, non_blocking=True)
            loaded[i % 2].record(copy_s)

    def compute(i):
        p = paths[i % 2]
        with torch.cuda.stream(comp_s):
            comp_s.wait_event(loaded[i % 2])
            p.step()
            for h, d in zip(outs_h[i % 2], outs[i % 2]):
                h.copy_(d, non_blocking=True)
            freed[i % 2].record(comp_s)

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)

    run(2)
    torch.cuda.synchronize()
    loops = []
    for _ in range(E2E_REPEATS):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(copy_s)
        run(steps)
        end.record(comp_s)
        torch.cuda.synchronize()
        loops.append(start.elapsed_time(end) / steps)
    ms = statistics.median(loops)
    h2d = logits_h.numel() * 2 + drafts_h.numel() * 4 + cu_h.numel() * 4
    d2h = sum(h.numel() * 4 for h in outs_h[0])
    # the host link alone: the same logits copy with nothing beside it
    # (median of 3); the pipelined step cannot beat it
    x = paths[0].x.view(torch.int16)
    link = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        x.copy_(logits_h, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        link.append(logits_h.numel() * 2 / (a.elapsed_time(b) * 1e-3) / 1e9)
    return ms, h2d, d2h, statistics.median(link), loops


# ---------------------------------------------------------------------------
# the CPU oracle as a timed baseline (rank 0 only)
# ---------------------------------------------------------------------------

def oracle_verify_step(oracle, x, shards, org, cu, drafts, k, blocks=None):
    if blocks:
        st, n = oracle.gathered_block_stats(x, shards, org, blocks[0], blocks[1], cu)
        return oracle.greedy_verify(st, n, cu, drafts, k)
    st = oracle.gathered_stats(x, shards, org)
    return oracle.greedy_verify(st, len(shards), cu, drafts, k)


def oracle_sample(c, n_reqs):
    """The first n_reqs requests of the workload (whole requests)."""
    cu = c["cu_num_draft"][:n_reqs + 1]
    rows, drafts = int(cu[-1]) + n_reqs, int(cu[-1])
    return c["logits"][:rows], cu, c["flags"][:drafts], c["rand_ids"][:drafts]


def oracle_drafts(oracle, x, shards, org, cu, flags, rand_ids):
    st = oracle.gathered_stats(x, shards, org)
    _, t = oracle.shard_reduce(st, len(shards), x.shape[0])
    return wl.compose_drafts(t, cu, flags, rand_ids)


def cpu_baseline(c, target_seconds, blocks=None):
    import oracle
    x, cu = c["logits"], c["cu_num_draft"]
    shards, org, k = c["shards"], c["org_vocab"], c["k"]
    drafts = oracle_drafts(oracle, x, shards, org, cu, c["flags"], c["rand_ids"])
    reps, t0 = 0, time.perf_counter()
    while True:
        out = oracle_verify_step(oracle, x, shards, org, cu, drafts, k, blocks)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_seconds or reps >= 500:
            break
    rows = x.shape[0]
    cores = oracle.num_threads()
    # the same oracle on one thread, over the first 16 requests (whole
    # requests), for about a fifth of the time
    n1 = min(16, cu.size - 1)
    x1, cu1 = x[:int(cu[n1]) + n1], cu[:n1 + 1]
    d1 = drafts[:int(cu[n1])]
    oracle.set_num_threads(1)
    try:
        reps1, t1 = 0, time.perf_counter()
        while True:
            oracle_verify_step(oracle, x1, shards, org, cu1, d1, k, blocks)
            reps1 += 1
            el1 = time.perf_counter() - t1
            if el1 >= target_seconds / 5 or reps1 >= 500:
                break
    finally:
        oracle.set_num_threads(cores)
    single = {"value": x1.shape[0] * reps1 / el1, "unit": "rows/s", "cores": 1,
              "sample": f"the first {n1} requests ({x1.shape[0]} rows) repeated {reps1} "
                        f"times in {el1:.1f} s"}
    return {"value": rows * reps / el, "unit": "rows/s", "cores": cores,
            "kind": "oracle", "_drafts": drafts, "_outputs": out, "single_thread": single,
            "sample": f"the whole workload ({rows} rows x {x.shape[1]} bf16 logits, "
                      + (f"block statistics {blocks[0]}/{blocks[1]} of {len(shards)} shards"
                         if blocks else f"{len(shards)} shard argmaxes")
                      + f" + verify of {cu.size - 1} requests) repeated {reps} times in "
                      f"{el:.1f} s"}


def run_reference(args, c_builder, blocks=None):
    """--impl reference: the CPU oracle, as it stands, on the host cores, on
    the same workload; each step is a bounded sample of whole requests sized so
    the whole run takes about two minutes at most."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    c = c_builder()
    k = c["k"]
    n_total = c["cu_num_draft"].size - 1
    # calibrate on 16 requests
    x, cu, fl, rd = oracle_sample(c, min(16, n_total))
    d = oracle_drafts(oracle, x, c["shards"], c["org_vocab"], cu, fl, rd)
    t0 = time.perf_counter()
    oracle_verify_step(oracle, x, c["shards"], c["org_vocab"], cu, d, k, blocks)
    per_req = (time.perf_counter() - t0) / min(16, n_total)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_reqs = int(max(1, min(n_total, budget / max(per_req, 1e-9))))
    x, cu, fl, rd = oracle_sample(c, n_reqs)
    d = oracle_drafts(oracle, x, c["shards"], c["org_vocab"], cu, fl, rd)
    for _ in range(args.warmup):
        oracle_verify_step(oracle, x, c["shards"], c["org_vocab"], cu, d, k, blocks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_verify_step(oracle, x, c["shards"], c["org_vocab"], cu, d, k, blocks)
    el = time.perf_counter() - t0
    rows = x.shape[0]
    value = rows * args.steps / el
    stats_kind = (f"block statistics {blocks[0]}/{blocks[1]} of {len(c['shards'])} shards"
                  if blocks else f"{len(c['shards'])} shard argmaxes")
    sample = (f"first {n_reqs} of {n_total} requests ({rows} rows x {x.shape[1]} bf16) per "
              f"step: {stats_kind} + verify")
    name = c["name"] + (f", block stats {blocks[0]}/{blocks[1]} (draft/bonus)" if blocks else "")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": name, "sample_rows_per_step": rows,
                       "workload_requested": args.workload},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


BLOCK_SIZES = (8192, 1024)   # draft / bonus block of the per-block statistics


KERNEL_LAUNCHES = 30   # isolated event-timed launches behind the roofline figure


def run_ours_verify(args, blocks=None):
    import torch
    rank, world = setup_device()
    import greedy_spec_decode_gb300 as sga

    c = (wl.large_verify_mixed_k if args.mixed_k else wl.large_verify)(rows_limit=args.rows)
    if args.rows is not None:
        c["name"] += f" (first {c['logits'].shape[0]} rows)"
    if blocks:
        c["name"] += f", block stats {blocks[0]}/{blocks[1]} (draft/bonus)"
    path = VerifyPath(c, torch, sga, blocks)
    total_ms, clocks = time_device_steps(path, args.steps, args.warmup, torch, world, rank)
    total_ms = max_over_ranks(total_ms, world, "cuda")
    # the dominant kernel alone: KERNEL_LAUNCHES launches, each between its
    # own events; the roofline figure uses their median
    argmax_times = time_launches(path.run_argmax, KERNEL_LAUNCHES, torch)
    verify_times = time_launches(path.run_verify, KERNEL_LAUNCHES, torch)
    argmax_ms = statistics.median(argmax_times)
    verify_ms = statistics.median(verify_times)
    step_ms = total_ms / args.steps
    rows_per_s = world * path.rows / (step_ms * 1e-3)

    pk, pk_src = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK_HBM_GBS))
    argmax_bytes = sum(path.argmax_bytes)
    achieved = argmax_bytes / (argmax_ms * 1e-3) / 1e9
    per_shard_ms = time_per_shard_steps(path, max(20, min(500, args.steps // 4)), torch)
    kernel_src = "blocks.cu" if blocks else "argmax.cu"
    traffic = ncu_traffic("block_argmax_large_verify.md" if blocks
                          else "local_argmax_large_verify.md",
                          ["greedy_spec_decode_gb300/csrc/" + kernel_src,
                           "greedy_spec_decode_gb300/csrc/scan.cuh",
                           "greedy_spec_decode_gb300/csrc/common.cuh"])  # device code only
    # (the block-stats profile records the DRAM bytes of the one-launch step)
    serial_ms, h2d, d2h, serial_loops = time_e2e(path, c, args.e2e_steps, torch)
    serial_ms = max_over_ranks(serial_ms, world, "cuda")
    path2 = VerifyPath(c, torch, sga, blocks)   # the second buffer set of the pipelined loop
    e2e_ms, _, _, link_gbs, e2e_loops = time_e2e_pipelined([path, path2], c, args.e2e_steps,
                                                            torch)
    e2e_ms = max_over_ranks(e2e_ms, world, "cuda")
    del path2

    # parity of the timed outputs is the tests' job; here only a sanity check
    # that the timed launches produced a full set of counts
    ns = path.num_sampled.cpu().numpy()
    assert ((ns >= 1) & (ns <= path.k + 1)).all(), "verify produced invalid counts"
    assert sga.sga_device_error() == 0, "device error word set during the bench"

    line = {
        "metric": METRIC, "value": rows_per_s, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": c["name"], "rows": path.rows, "vocab": int(c["logits"].shape[1]),
                   "shards": [w for _, w in path.shards], "requests": path.n, "k": path.k,
                   "stats_per_row": path.n_stats,
                   "l2": f"inputs ({c['logits'].nbytes / 1e9:.2f} GB) larger than L2 (129 MB); no flush",
                   "parallelism": f"{world} independent replica(s), emulated TP{len(path.shards)} per GPU"},
        "step_timing": (f"K steps between two CUDA events, replayed from CUDA graphs of "
                        f"{min(GRAPH_STEPS, args.steps)} steps (every launch runs; no event "
                        f"between steps)"),
        "step_gbs": path.step_bytes / (step_ms * 1e-3) / 1e9,
        "step_frac_of_hbm": path.step_bytes / (step_ms * 1e-3) / 1e9 / hbm,
        "kernel_us": {("block_argmax_all_shards" if blocks else "local_argmax_all_shards"):
                      spread(argmax_times),
                      "greedy_verify": spread(verify_times),
                      "note": "each kernel timed alone after the timed steps: "
                              f"{KERNEL_LAUNCHES} launches, each between its own CUDA events "
                              "(in the timed steps the verify launch overlaps the argmax tail "
                              "through programmatic dependent launch)"},
        "per_shard_launches": {"ms_per_step": per_shard_ms,
                               "rows_per_s": world * path.rows / (per_shard_ms * 1e-3),
                               "note": "same step with one launch per shard (sga_local_argmax"
                                       + ("_blocks" if blocks else "") + ")"},
        "roofline": {"bound": "hbm",
                     "kernel": ("block_argmax_kernel<bf16> (all shards, one launch)" if blocks
                                else "local_argmax_kernel<bf16> (all shards, one launch)"),
                     "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "timing": f"median of {KERNEL_LAUNCHES} isolated event-timed launches",
                     "peak_source": f"{pk_src} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)"
                     if pk_src == "measured" else "fallback 6.8 TB/s",
                     "bytes_per_launch": argmax_bytes},
        "e2e": {"value": world * path.rows / (e2e_ms * 1e-3), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": "two buffer sets: step i+1's inputs are copied in while step i runs",
                "timing": (f"median of {E2E_REPEATS} loops of {args.e2e_steps} steps (the host "
                           f"memory and link are shared with other jobs on the machine)"),
                "loops_ms_per_step": [round(x, 3) for x in e2e_loops],
                "host_link": {"h2d_gbs": link_gbs,
                              "achieved_gbs": h2d / (e2e_ms * 1e-3) / 1e9,
                              "frac": h2d / (e2e_ms * 1e-3) / 1e9 / link_gbs,
                              "note": "the step's input bytes per e2e step time against one "
                                      "plain copy of the logits from pinned host memory; "
                                      "more streams or a kernel reading the pinned memory "
                                      "directly move no more over this link"},
                "serial": {"value": world * path.rows / (serial_ms * 1e-3),
                           "ms_per_step": serial_ms,
                           "loops_ms_per_step": [round(x, 3) for x in serial_loops],
                           "note": "copy in, step, copy out, one after the other"}},
        "gpu_launches": args.steps * path.launches_per_step,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(c, args.cpu_seconds, blocks)
        # the baseline leg ran the oracle on the whole workload: recheck the
        # timed device outputs against it, bit for bit
        exp, exp_drafts = base.pop("_outputs"), base.pop("_drafts")
        got = {"sampled": path.sampled, "num_sampled": path.num_sampled,
               "num_rejected": path.num_rejected, "bonus": path.bonus}
        same = bool((exp_drafts == path.drafts_host).all()) and all(
            bool((v.cpu().numpy() == exp[key]).all()) for key, v in got.items())
        if not same:
            raise SystemExit("timed outputs differ from the oracle: no number is reported")
        line["parity"] = ("timed outputs (sampled, num_sampled, num_rejected, bonus) and the "
                          "drafts bit-exact with the oracle of the cpu_baseline leg")
        line["cpu_baseline"] = base
    if not args.no_extra and blocks is None and not args.mixed_k:
        del path
        torch.cuda.empty_cache()
        add_extra_records(line, args, rank, world)
    return finish(line, rank, world)


def add_extra_records(line, args, rank, world):
    """The other configurations of the metric, each as a nested record of the
    default line: the fused LM head (512 x 4096 . [151936 x 4096]^T bf16, 2
    shards; tensor roofline), the same head at a decode size (16 rows, bf16
    and fp8, the step replayed from a CUDA graph; HBM roofline) and the two
    L2-resident latency workloads (draft get_top_tokens, small greedy
    verify)."""
    import argparse as ap
    sub = ap.Namespace(**vars(args))
    sub.graph, sub.lmhead_per_shard, sub.e2e_steps = False, False, 5
    sub.lmhead_rows, sub.lmhead_vocab, sub.lmhead_shards = 512, 151936, 2
    sub.steps, sub.warmup, sub.cpu_seconds = 100, 5, min(args.cpu_seconds, 6.0)
    line["lmhead"] = measure_lmhead(sub, False, rank, world)
    sub.graph, sub.lmhead_rows, sub.steps, sub.cpu_seconds = True, 16, 200, min(args.cpu_seconds,
                                                                                  3.0)
    line["lmhead_decode"] = measure_lmhead(sub, False, rank, world)
    line["lmhead_decode_fp8"] = measure_lmhead(sub, True, rank, world)
    sub.graph, sub.steps, sub.cpu_seconds = False, 200, min(args.cpu_seconds, 2.0)
    line["draft_top_tokens"] = measure_small(sub, wl.draft_top_tokens, rank, world)
    line["greedy_verify_small"] = measure_small(sub, wl.greedy_verify_small, rank, world)


def run_ours_tp(args):
    """--tp: the tensor-parallel form of the default step.  Rank r of the N
    ranks holds only vocab shard r of the large-verify logits on its own GPU,
    runs the local argmax of it, all-gathers the 8-byte statistics of its
    rows on dim 0 (NCCL), and runs the fused verify on the gathered buffer.
    The N ranks process ONE batch together (strong scaling): value = rows /
    step time.  The exchange is also timed alone."""
    import torch
    rank, world = setup_device()
    import greedy_spec_decode_gb300 as sga
    from greedy_spec_decode_gb300 import tp

    c = (wl.large_verify_mixed_k if args.mixed_k else wl.large_verify)(rows_limit=args.rows)
    rows, vocab, k = c["logits"].shape[0], c["logits"].shape[1], c["k"]
    org, cu_np = c["org_vocab"], c["cu_num_draft"]
    n = cu_np.size - 1
    start, width = tp.vocab_shard(vocab, world, rank)
    x = torch.from_numpy(np.ascontiguousarray(c["logits"][:, start:start + width]).view(np.int16))
    x = x.view(torch.bfloat16).cuda()
    cu = torch.from_numpy(cu_np).cuda()
    gathered = tp.gathered_stats_buffer(rows)
    i32 = dict(dtype=torch.int32, device="cuda")
    # drafts from one untimed pass of the same path (every rank gets the same)
    t = torch.empty(rows, **i32)
    tp.tp_top_tokens(x, start, org, t, gathered)
    drafts_np = wl.compose_drafts(t.cpu().numpy(), cu_np, c["flags"], c["rand_ids"])
    drafts = torch.from_numpy(drafts_np).cuda()
    outs = [torch.empty((n, k + 1), **i32)] + [torch.empty(n, **i32) for _ in range(3)]

    def step():
        tp.tp_greedy_verify(x, start, org, cu, drafts, k, *outs, gathered)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.3)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    step_ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda") / args.steps
    # the pieces alone: the rank's local argmax, the exchange, the verify
    argmax_times = time_launches(
        lambda: sga.sga_local_argmax(x, start, width, org, tp.local_slot(gathered, rows)),
        KERNEL_LAUNCHES, torch)
    exchange_times = time_launches(lambda: tp.gather_stats(gathered, rows), KERNEL_LAUNCHES, torch)
    verify_times = time_launches(
        lambda: sga.sga_greedy_verify(gathered, world, cu, drafts, k, *outs), KERNEL_LAUNCHES,
        torch)
    argmax_ms = max_over_ranks(statistics.median(argmax_times), world, "cuda")
    exchange_ms = max_over_ranks(statistics.median(exchange_times), world, "cuda")
    assert sga.sga_device_error() == 0, "device error word set during the bench"
    pk, pk_src = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK_HBM_GBS))
    local_bytes = rows * (width * 2 + 8)
    achieved = local_bytes / (statistics.median(argmax_times) * 1e-3) / 1e9

    # end to end: each rank copies its shard of the logits (and the drafts)
    # in from pinned host memory and reads the results back
    x_h = torch.from_numpy(np.ascontiguousarray(c["logits"][:, start:start + width]).view(np.int16))
    x_h = x_h.pin_memory()
    d_h = torch.from_numpy(drafts_np).pin_memory()
    outs_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    x_raw = x.view(torch.int16)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.e2e_steps):
        x_raw.copy_(x_h, non_blocking=True)
        drafts.copy_(d_h, non_blocking=True)
        step()
        for h_, d_ in zip(outs_h, outs):
            h_.copy_(d_, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / args.e2e_steps, world, "cuda")

    line = {
        "metric": METRIC, "value": rows / (step_ms * 1e-3), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": c["name"] + f", as TP{world}", "rows": rows, "vocab": vocab,
                   "shards": [tp.vocab_shard(vocab, world, r)[1] for r in range(world)],
                   "requests": n, "k": k,
                   "l2": f"inputs ({c['logits'].nbytes / 1e9:.2f} GB) larger than L2; no flush",
                   "parallelism": f"TP{world}: rank r holds vocab shard r; per step one "
                                  f"dim-0 all-gather of {rows} x 8 B statistics per rank"},
        "exchange": {"us_per_step": round(exchange_ms * 1e3, 2),
                     "bytes_per_rank": rows * 8, "backend": "none (one rank)" if world == 1
                     else "nccl all_gather_into_tensor",
                     "spread": spread(exchange_times)},
        "kernel_us": {"local_argmax_own_shard": spread(argmax_times),
                      "greedy_verify": spread(verify_times)},
        "roofline": {"bound": "hbm", "kernel": "local_argmax_kernel<bf16> (this rank's shard)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None, "timing": f"median of {KERNEL_LAUNCHES} isolated launches",
                     "peak_source": f"{pk_src} hbm_gbs", "bytes_per_launch": local_bytes},
        "e2e": {"value": rows / (e2e_ms * 1e-3), "unit": "rows/s",
                "h2d_bytes_per_step": x_h.numel() * 2 + d_h.numel() * 4,
                "d2h_bytes_per_step": sum(h_.numel() * 4 for h_ in outs_h),
                "ms_per_step": e2e_ms, "note": "per rank: its logits shard in, the results out"},
        "gpu_launches": args.steps * 2,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        shards = [tp.vocab_shard(vocab, world, r) for r in range(world)]
        t0 = time.perf_counter()
        exp = oracle_verify_step(oracle, c["logits"], shards, org, cu_np, drafts_np, k)
        el = time.perf_counter() - t0
        got = dict(sampled=outs[0], num_sampled=outs[1], num_rejected=outs[2], bonus=outs[3])
        if not all(bool((v.cpu().numpy() == exp[key]).all()) for key, v in got.items()):
            raise SystemExit("TP outputs differ from the oracle: no number is reported")
        line["parity"] = "rank 0's outputs bit-exact with the oracle of the whole batch"
        line["cpu_baseline"] = {"value": rows / el, "unit": "rows/s", "kind": "oracle",
                                "cores": oracle.num_threads(),
                                "sample": f"the whole batch once ({el:.1f} s)"}
    return finish(line, rank, world)


LMHEAD_METRIC = "fused LM-head + argmax rows/s and TFLOP/s (frac of bf16 tensor peak)"
LMHEAD_METRIC_FP8 = "fused fp8 LM-head + argmax rows/s and TFLOP/s (frac of fp8 tensor peak)"


FP8_TO_BF16_NOMINAL = 4.5 / 2.25   # dense tensor peaks, PFLOP/s per GPU


def lmhead_cpu_baseline(c, fp8, gpu_ids, target_seconds):
    """The oracle's fp64 LM-head logits + argmax on a bounded sample of rows
    (whole vocabulary, every shard), timed; the same rows of the device path's
    ids are checked against it within the LM-head tolerance (ids equal where
    the top-1 / top-2 gap exceeds 1e-2, else a near-winner)."""
    import oracle
    M = c["hidden"].shape[0]
    org = c["org_vocab"]
    rows_done, checked, t0 = 0, 0, time.perf_counter()
    while rows_done < M:
        sel = np.arange(rows_done, min(M, rows_done + 2), dtype=np.int64)
        if fp8:
            logits = oracle.lmhead_logits_fp8(c["hidden"], c["hidden_scale"], c["weight"],
                                              c["weight_scale"], sel)
        else:
            logits = oracle.lmhead_logits(c["hidden"], c["weight"], sel)
        top1, top2, exp = oracle.argmax_f64(logits, 0, org)
        for q, r in enumerate(sel):
            g = int(gpu_ids[r])
            ok = g == exp[q] if top1[q] - top2[q] > 1e-2 else logits[q, g] >= top1[q] - 1e-2
            if not ok:
                raise SystemExit(f"LM-head row {r}: device id {g}, oracle {exp[q]}: no number is "
                                 "reported")
            checked += 1
        rows_done += sel.size
        if time.perf_counter() - t0 >= target_seconds:
            break
    el = time.perf_counter() - t0
    base = {"value": rows_done / el, "unit": "rows/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"the first {rows_done} of {M} rows, fp64 logits over all "
                      f"{c['weight'].shape[0]} ids ({el:.1f} s)"}
    return base, (f"ids of {checked} sampled rows within the LM-head tolerance of the oracle "
                  "of the cpu_baseline leg")


DECODE_MAX_M = 128  # the library's decode-size LM-head kernels cover M <= 128


def decode_roofline(weight_bytes, kern_ms, num_shards, fp8, captured_shape=True,
                    one_call=True, M=16):
    """HBM roofline of the decode-size LM-head kernels: the weight is read once
    per step (one launch per shard).  The committed captures are of M = 16
    (one CTA per SM) and, for one call, M = 128 (CTA pairs)."""
    pk, pk_src = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = weight_bytes / (kern_ms * 1e-3) / 1e9
    # the captures are of the default shape (2 x 75968 ids, H = 4096): one
    # launch for both shards (one call), or one shard per launch
    pair = M > 64
    key = ("dram_bytes_per_launch_all_shards" if one_call else "dram_bytes_per_launch") + \
        ("_pair" if pair else "") + ("_fp8" if fp8 else "")
    captured_shape = captured_shape and (one_call or not pair)
    traffic = ncu_traffic("lmhead_decode.md", ["greedy_spec_decode_gb300/csrc/lmhead_decode.cu",
                                               "greedy_spec_decode_gb300/csrc/tcgen05.cuh",
                                               "greedy_spec_decode_gb300/csrc/common.cuh"], key)
    return {"bound": "hbm",
            "kernel": "lmhead_argmax_decode_%skernel<%s>" % ("pair_" if pair else "",
                                                             "fp8" if fp8 else "bf16"),
            "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": traffic if captured_shape else None,
            "traffic_unit": "DRAM bytes per decode launch (%s), %s M = %d capture"
                            % ("every shard" if one_call else "one shard",
                               "fp8" if fp8 else "bf16", 128 if pair else 16),
            "peak_source": f"{pk_src} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)"
            if pk_src == "measured" else "fallback 6.8 TB/s",
            "bytes_per_step": weight_bytes, "launches_per_step": 1 if one_call else num_shards,
            "timing": f"median of {KERNEL_LAUNCHES} isolated event-timed LM-head calls"
                      + ("" if one_call else f" ({num_shards} launches in each interval)")}


def setup_device():
    """Device, process group and the built library (rank 0 builds)."""
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    from greedy_spec_decode_gb300 import build as sga_build
    if rank == 0 or world == 1:
        sga_build.build()
    barrier(world)
    return rank, world


def finish(line, rank, world):
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_ours_lmhead(args, fp8=False):
    """Fused LM-head + argmax: 512 rows, hidden 4096, vocab 151936 in 2 shards;
    one step = sga_lmhead_argmax (or its fp8 variant) per shard +
    sga_shard_reduce."""
    rank, world = setup_device()
    return finish(measure_lmhead(args, fp8, rank, world), rank, world)


def library_gemm_context(hidden, weight, fp8, torch):
    """cuBLAS (bf16) or cuBLASLt (fp8, torch._scaled_mm) on the LM head's GEMM
    shape, writing the logits and taking no argmax, and on an 8192^3 GEMM of
    the same type: context for the fused kernel's tensor roofline (the fp8
    roofline itself is the measured bf16 burst x the nominal fp8 / bf16
    ratio).  Back-to-back calls between two events, median of 3 x 20."""
    def rate(fn, flops):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        res = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(20):
                fn()
            b.record()
            torch.cuda.synchronize()
            res.append(flops / (a.elapsed_time(b) / 20 * 1e-3) / 1e12)
        return statistics.median(res)
    M, H = hidden.shape
    V = weight.shape[0]
    g = torch.Generator(device="cuda").manual_seed(0)
    sq = 8192
    try:
        if fp8:
            one = torch.ones((), dtype=torch.float32, device="cuda")
            h8, w8 = hidden.view(torch.float8_e4m3fn), weight.view(torch.float8_e4m3fn)
            same = rate(lambda: torch._scaled_mm(h8, w8.t(), scale_a=one, scale_b=one,
                                                 out_dtype=torch.bfloat16), 2.0 * M * H * V)
            a = torch.randn(sq, sq, device="cuda", generator=g).to(torch.float8_e4m3fn)
            b = torch.randn(sq, sq, device="cuda", generator=g).to(torch.float8_e4m3fn)
            square = rate(lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one,
                                                   out_dtype=torch.bfloat16), 2.0 * sq ** 3)
            lib = "cuBLASLt via torch._scaled_mm, E4M3 x E4M3 -> bf16"
        else:
            out = torch.empty(M, V, dtype=torch.bfloat16, device="cuda")
            same = rate(lambda: torch.matmul(hidden, weight.t(), out=out), 2.0 * M * H * V)
            del out
            a = torch.randn(sq, sq, device="cuda", generator=g).to(torch.bfloat16)
            b = torch.randn(sq, sq, device="cuda", generator=g).to(torch.bfloat16)
            square = rate(lambda: torch.matmul(a, b.t()), 2.0 * sq ** 3)
            lib = "cuBLAS via torch.matmul, bf16 -> bf16"
        del a, b
        torch.cuda.empty_cache()
    except (RuntimeError, TypeError) as e:
        return {"unavailable": str(e).splitlines()[0][:200]}
    return {"library": lib, "same_shape_tflops": same, "square_8192_tflops": square,
            "note": "the library GEMM writes the logits and takes no argmax; context only"}


def measure_lmhead(args, fp8, rank, world):
    """The fused LM-head step timed on this GPU; returns its JSON record."""
    import torch
    import greedy_spec_decode_gb300 as sga

    if fp8:
        c = wl.fused_lmhead_fp8(m=args.lmhead_rows, vocab=args.lmhead_vocab,
                                num_shards=args.lmhead_shards)
        hidden = torch.from_numpy(c["hidden"]).cuda()
        weight = torch.from_numpy(c["weight"]).cuda()
        hscale = torch.from_numpy(c["hidden_scale"]).cuda()
    else:
        c = wl.fused_lmhead(m=args.lmhead_rows, vocab=args.lmhead_vocab,
                            num_shards=args.lmhead_shards)
        hidden = torch.from_numpy(c["hidden"].view(np.int16)).view(torch.bfloat16).cuda()
        weight = torch.from_numpy(c["weight"].view(np.int16)).view(torch.bfloat16).cuda()
    M, H = hidden.shape
    shards = c["shards"]
    S = len(shards)
    stats = sga.new_stats(S * M)
    one_call = not args.lmhead_per_shard
    ws_bytes = (sga.sga_lmhead_argmax_shards_workspace(M, shards) if one_call else
                max(sga.sga_lmhead_argmax_workspace(M, w) for _, w in shards))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ids = torch.empty(M, dtype=torch.int32, device="cuda")
    w_views = [weight[o:o + w] for o, w in shards]

    def step(ev=None):
        if one_call:
            if ev is not None:
                ev[0].record()
            if fp8:
                sga.sga_lmhead_argmax_shards_fp8(hidden, hscale, weight, c["weight_scale"],
                                                 shards, c["org_vocab"], stats, ws)
            else:
                sga.sga_lmhead_argmax_shards(hidden, weight, shards, c["org_vocab"], stats, ws)
            if ev is not None:
                ev[1].record()
            sga.sga_shard_reduce(stats, S, M, ids)
            return
        for s, (o, w) in enumerate(shards):
            if ev is not None:
                ev[2 * s].record()
            if fp8:
                sga.sga_lmhead_argmax_fp8(hidden, hscale, w_views[s], c["weight_scale"], o,
                                          c["org_vocab"], stats[s * M:(s + 1) * M], ws)
            else:
                sga.sga_lmhead_argmax(hidden, w_views[s], o, c["org_vocab"],
                                      stats[s * M:(s + 1) * M], ws)
            if ev is not None:
                ev[2 * s + 1].record()
        sga.sga_shard_reduce(stats, S, M, ids)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    graph = None
    if args.graph:
        # the whole step replayed from one CUDA graph, as a serving engine
        # replays a decode step: no host submission gaps between launches
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
    barrier(world)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * S)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.3)
    start.record()
    for i in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(ev[i])
    end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    total_ms = max_over_ranks(start.elapsed_time(end), world, "cuda")
    step_ms = total_ms / args.steps
    if graph is not None:
        kern_times = None
        kern_ms = step_ms   # the step as a whole (LM-head launches + finalize + reduce)
    else:
        kern_times = [sum(e[2 * s].elapsed_time(e[2 * s + 1]) for s in range(1 if one_call else S))
                      for e in ev]
        kern_ms = statistics.median(kern_times)
    # M <= 128 runs a decode-size kernel: a weight stream bound by HBM, not
    # by the tensor cores (2 M flops per weight element)
    decode = M <= DECODE_MAX_M
    iso_times = None
    if decode:
        # the decode kernel alone for its roofline: KERNEL_LAUNCHES calls, each
        # between its own events (one launch per call: the CTAs merge in-kernel)
        def lmhead_calls():
            for s, (o, w) in enumerate([(None, None)] if one_call else shards):
                if one_call and fp8:
                    sga.sga_lmhead_argmax_shards_fp8(hidden, hscale, weight, c["weight_scale"],
                                                     shards, c["org_vocab"], stats, ws)
                elif one_call:
                    sga.sga_lmhead_argmax_shards(hidden, weight, shards, c["org_vocab"], stats, ws)
                elif fp8:
                    sga.sga_lmhead_argmax_fp8(hidden, hscale, w_views[s], c["weight_scale"], o,
                                              c["org_vocab"], stats[s * M:(s + 1) * M], ws)
                else:
                    sga.sga_lmhead_argmax(hidden, w_views[s], o, c["org_vocab"],
                                          stats[s * M:(s + 1) * M], ws)
        iso_times = time_launches(lmhead_calls, KERNEL_LAUNCHES, torch)
    flops = 2.0 * M * H * sum(w for _, w in shards)
    pk, pk_src = peaks()
    # the LM-head calls are timed one by one over a short loop: the burst
    # GEMM peak is the roofline; the sustained (power-capped) one is reported
    sustained = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS)))
    peak = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    if fp8:
        peak *= FP8_TO_BF16_NOMINAL
        sustained *= FP8_TO_BF16_NOMINAL
    achieved = flops / (kern_ms * 1e-3) / 1e12
    assert sga.sga_device_error() == 0, "device error word set during the bench"
    weight_bytes = weight.numel() * weight.element_size()

    # end to end: hidden states in from pinned host memory, ids back
    hid_h = (torch.from_numpy(c["hidden"]) if fp8 else
             torch.from_numpy(c["hidden"].view(np.int16))).pin_memory()
    ids_h = torch.empty(M, dtype=torch.int32).pin_memory()
    hid_i16 = hidden if fp8 else hidden.view(torch.int16)
    scale_h = torch.from_numpy(c["hidden_scale"]).pin_memory() if fp8 else None
    h2d_bytes = hid_h.numel() * hid_h.element_size() + (scale_h.numel() * 4 if fp8 else 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.e2e_steps):
        hid_i16.copy_(hid_h, non_blocking=True)
        if fp8:
            hscale.copy_(scale_h, non_blocking=True)
        step()
        ids_h.copy_(ids, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, "cuda")
    lib_ctx = None if decode else library_gemm_context(hidden, weight, fp8, torch)

    line = {
        "metric": LMHEAD_METRIC_FP8 if fp8 else LMHEAD_METRIC,
        "value": world * M / (step_ms * 1e-3), "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8 e4m3 (fp32 accumulate)" if fp8 else "bf16 (fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": c["name"], "M": M, "H": H, "shards": [w for _, w in shards],
                   "l2": "weight (1.24 GB) larger than L2 (129 MB); no flush",
                   "parallelism": f"{world} independent replica(s), emulated TP{S} per GPU"},
        "tflops_step": flops / (step_ms * 1e-3) / 1e12,
        "weight_gbs": weight.numel() * weight.element_size() / (kern_ms * 1e-3) / 1e9,
        "kernel_us": {"lmhead_argmax_per_step": (spread(kern_times) if kern_times is not None
                                                 else round(kern_ms * 1e3, 2)),
                      "reduce_and_gaps": round((step_ms - kern_ms) * 1e3, 2),
                      **({"lmhead_argmax_isolated": spread(iso_times)} if decode else {})},
        "roofline": decode_roofline(weight_bytes, statistics.median(iso_times), S, fp8,
                                    S == 2 and H == 4096 and args.lmhead_vocab == 151936,
                                    one_call, M)
        if decode else
                    {"bound": "tensor",
                     "kernel": "lmhead_argmax_2sm_kernel<fp8>" if fp8 else "lmhead_argmax_2sm_kernel",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": ncu_traffic(
                         "lmhead_fused_fp8.md" if fp8 else "lmhead_fused.md",
                         ["greedy_spec_decode_gb300/csrc/lmhead.cu",
                          "greedy_spec_decode_gb300/csrc/tcgen05.cuh",
                          "greedy_spec_decode_gb300/csrc/common.cuh"]),
                     "traffic_unit": "DRAM bytes per launch of the GEMM kernel",
                     "peak_source": ((f"{pk_src} bf16_tflops (cuBLAS bf16 GEMM, burst)")
                                     if pk_src == "measured" else "fallback 1.9 PFLOP/s")
                                    + (" x 2 (nominal fp8 / bf16 dense ratio)" if fp8 else ""),
                     "timing": (f"median of {len(kern_times)} event-timed LM-head calls"
                                if kern_times is not None else "graph-replayed steps"),
                     "frac_of_sustained": achieved / sustained,
                     "flops_per_step": flops},
        "e2e": {"value": world * M / (e2e_ms * 1e-3), "unit": "rows/s",
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": M * 4,
                "ms_per_step": e2e_ms,
                "note": f"{args.e2e_steps} steps after the timed loop, with the hidden "
                        "states copied in and the ids read back each step; a tensor-bound "
                        "step runs under the power cap, so the clocks of the two loops "
                        "can differ and this figure can exceed `value`"},
        "timing": ("whole step replayed from a CUDA graph" if graph is not None else
                   "CUDA events around each LM-head call (GEMM + finalize)"),
        "calls": ("every shard in one sga_lmhead_argmax_shards call" if one_call else
                  "one sga_lmhead_argmax call per shard (each emulated rank its own)"),
        # one call: decode sizes 1 launch (the CTAs merge in-kernel), else the
        # GEMM + finalize; per shard: the same per call; + the reduce
        "gpu_launches": args.steps * (((1 if M <= DECODE_MAX_M else 2) * (1 if one_call else S))
                                      + 1),
        "clocks": clocks,
    }
    if lib_ctx is not None:
        line["library_gemm"] = lib_ctx
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = lmhead_cpu_baseline(
            c, fp8, ids.cpu().numpy(), args.cpu_seconds)
    return line


def small_cpu_baseline(c, stats, outs, drafts, target_seconds):
    """The oracle on the whole small workload, repeated for about
    target_seconds and timed; the device path's statistics and results are
    checked against it bit for bit (no number on a mismatch)."""
    import oracle
    x, shards, org = c["logits"], c["shards"], c["org_vocab"]
    S, rows = len(shards), c["logits"].shape[0]
    verify = drafts is not None
    reps, t0 = 0, time.perf_counter()
    while True:
        st = oracle.gathered_stats(x, shards, org)
        if verify:
            exp = oracle.greedy_verify(st, S, c["cu_num_draft"], drafts, c["k"])
        else:
            _, exp_ids = oracle.shard_reduce(st, S, rows)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_seconds or reps >= 2000:
            break
    got_st = stats.cpu().numpy().view(oracle.STAT).reshape(-1)
    same = bool((got_st["id"] == st["id"]).all()
                and (got_st["v"].view(np.uint32) == st["v"].view(np.uint32)).all())
    if verify:
        names = ("sampled", "num_sampled", "num_rejected", "bonus")
        same = same and all(bool((o.cpu().numpy() == exp[k]).all()) for k, o in zip(names, outs))
        # the drafts copy the device path's own argmax: they must be the oracle's
        _, t = oracle.shard_reduce(st, S, rows)
        same = same and bool((wl.compose_drafts(t, c["cu_num_draft"], c["flags"],
                                                c["rand_ids"]) == drafts).all())
    else:
        same = same and bool((outs.cpu().numpy() == exp_ids).all())
    if not same:
        raise SystemExit("timed outputs differ from the oracle: no number is reported")
    base = {"value": rows * reps / el, "unit": "rows/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"the whole workload ({rows} rows, {S} shards) repeated {reps} times "
                      f"in {el:.1f} s"}
    return base, ("timed statistics and results bit-exact with the oracle of the "
                  "cpu_baseline leg")


def run_ours_small(args, builder):
    """L2-resident workloads (draft get_top_tokens, small greedy verify): one
    step = the one-launch shard argmax + the reduce (no drafts) or the fused
    verify.  Each timed step follows an L2 flush (a 256 MB write) and is timed
    alone with CUDA events; value = rows / mean step time."""
    rank, world = setup_device()
    return finish(measure_small(args, builder, rank, world), rank, world)


def measure_small(args, builder, rank, world):
    """An L2-resident workload timed on this GPU; returns its JSON record."""
    import torch
    import greedy_spec_decode_gb300 as sga

    c = builder()
    x_np = c["logits"]
    x = (torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16) if x_np.dtype == np.uint16
         else torch.from_numpy(x_np)).cuda()
    rows, shards, org = x.shape[0], c["shards"], c["org_vocab"]
    S = len(shards)
    stats = sga.new_stats(S * rows)
    i32 = dict(dtype=torch.int32, device="cuda")
    verify = "k" in c
    if verify:
        k, cu_np = c["k"], c["cu_num_draft"]
        n = cu_np.size - 1
        cu = torch.from_numpy(cu_np).cuda()
        t = torch.empty(rows, **i32)
        sga.sga_local_argmax_shards(x, shards, org, stats)
        sga.sga_shard_reduce(stats, S, rows, t)
        drafts = torch.from_numpy(wl.compose_drafts(t.cpu().numpy(), cu_np, c["flags"],
                                                    c["rand_ids"])).cuda()
        outs = [torch.empty((n, k + 1), **i32)] + [torch.empty(n, **i32) for _ in range(3)]
    else:
        ids = torch.empty(rows, **i32)

    def step():
        sga.sga_local_argmax_shards(x, shards, org, stats)
        if verify:
            sga.sga_greedy_verify(stats, S, cu, drafts, k, *outs)
        else:
            sga.sga_shard_reduce(stats, S, rows, ids)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    graph = None
    if args.graph:
        # the step replayed from one CUDA graph, as a serving engine replays
        # a decode step
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
    run_step = graph.replay if graph is not None else step
    barrier(world)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.3)
    for a, b in evs:
        flush.zero_()
        a.record()
        run_step()
        b.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    times = [a.elapsed_time(b) for a, b in evs]
    step_ms = max_over_ranks(sum(times) / len(times), world, "cuda")
    elt = x.element_size()
    step_bytes = sum(rows * (w * elt + 8) for _, w in shards)
    pk, pk_src = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK_HBM_GBS))
    assert sga.sga_device_error() == 0
    line = {
        "metric": METRIC, "value": world * rows / (step_ms * 1e-3), "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "us_per_step_min": min(times) * 1e3, "us_per_step_median": sorted(times)[len(times) // 2] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if elt == 2 else "f32", "data": "synthetic",
        "config": {"workload": c["name"], "rows": rows, "shards": [w for _, w in shards],
                   "l2": "inputs fit in L2: 256 MB flush before every timed step",
                   "step": "one-launch shard argmax + " + ("fused verify" if verify else "shard reduce")
                   + (", replayed from a CUDA graph" if graph is not None else "")},
        "step_gbs": step_bytes / (step_ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": step_bytes / (step_ms * 1e-3) / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": step_bytes / (step_ms * 1e-3) / 1e9 / hbm,
                     "traffic": None, "note": "latency-bound at this size; whole step timed"},
        "gpu_launches": args.steps * 2,
        "clocks": clocks,
    }
    # end to end through the same calls with host buffers: logits (and the
    # drafts) in from pinned memory, the step's results back
    logits_h = torch.from_numpy(x_np.view(np.int16) if x_np.dtype == np.uint16 else x_np).pin_memory()
    x_raw = x.view(torch.int16) if x_np.dtype == np.uint16 else x
    outs_d = outs if verify else [ids]
    outs_h = [torch.empty(t_.shape, dtype=t_.dtype).pin_memory() for t_ in outs_d]
    drafts_h = torch.from_numpy(drafts.cpu().numpy()).pin_memory() if verify else None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, args.e2e_steps)
    e0.record()
    for _ in range(e2e_steps):
        x_raw.copy_(logits_h, non_blocking=True)
        if verify:
            drafts.copy_(drafts_h, non_blocking=True)
        step()
        for h_, d_ in zip(outs_h, outs_d):
            h_.copy_(d_, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, "cuda")
    line["e2e"] = {"value": world * rows / (e2e_ms * 1e-3), "unit": "rows/s",
                   "h2d_bytes_per_step": logits_h.numel() * logits_h.element_size()
                   + (drafts_h.numel() * 4 if verify else 0),
                   "d2h_bytes_per_step": sum(h_.numel() * 4 for h_ in outs_h),
                   "ms_per_step": e2e_ms}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = small_cpu_baseline(
            c, stats, outs if verify else ids, drafts.cpu().numpy() if verify else None,
            args.cpu_seconds)
    return line


def main():
    args = parse_args()
    if args.impl == "reference":
        # the oracle's arm is defined for the verify workloads; any other
        # workload is timed on the default one and says so in its config
        return run_reference(args, wl.large_verify_mixed_k if args.mixed_k else wl.large_verify,
                             BLOCK_SIZES if args.workload == "large_verify_blocks" else None)
    if args.tp:
        return run_ours_tp(args)
    if args.workload == "lmhead":
        return run_ours_lmhead(args)
    if args.workload == "lmhead_fp8":
        return run_ours_lmhead(args, fp8=True)
    if args.workload == "draft_top_tokens":
        return run_ours_small(args, wl.draft_top_tokens)
    if args.workload == "greedy_verify":
        return run_ours_small(args, wl.greedy_verify_small)
    if args.workload == "large_verify_blocks":
        return run_ours_verify(args, BLOCK_SIZES)
    return run_ours_verify(args)


if __name__ == "__main__":
    sys.exit(main())
