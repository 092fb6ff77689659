"""The bench's one-line JSON contract on reduced workloads (GPU): every line
carries the metric, the whole-job value, the roofline with its peak source,
the end-to-end figure with its host<->device bytes, the clocks seen, the
launch count and, with the CPU leg on, the oracle baseline and the parity
recheck of the timed outputs."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def check_common(d, unit):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["unit"] == unit and d["value"] > 0 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["scaling"] in ("weak", "strong")
    assert "workload" in d["config"]
    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= d["steps"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_large_verify_line_with_oracle_leg_and_nested_records():
    d = run_bench("--rows", "512", "--steps", "16", "--warmup", "3", "--e2e-steps", "1",
                  "--cpu-seconds", "1")
    check_common(d, "rows/s")
    assert d["roofline"]["unit"] == "GB/s"
    assert d["kernel_us"]["local_argmax_all_shards"]["launches"] >= 20
    k = d["kernel_us"]["local_argmax_all_shards"]
    assert k["min_us"] <= k["median_us"] <= k["max_us"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["single_thread"]["cores"] == 1
    assert "bit-exact" in d["parity"]
    # the other configurations ride along as nested records
    lm = d["lmhead"]
    check_common(lm, "rows/s")
    assert lm["roofline"]["bound"] == "tensor" and lm["roofline"]["unit"] == "TFLOP/s"
    assert lm["config"]["M"] == 512 and lm["config"]["shards"] == [75968, 75968]
    assert lm["cpu_baseline"]["kind"] == "oracle" and "tolerance" in lm["parity"]
    for key in ("lmhead_decode", "lmhead_decode_fp8"):
        dec = d[key]
        check_common(dec, "rows/s")
        assert dec["config"]["M"] == 16 and dec["roofline"]["bound"] == "hbm"
        assert dec["kernel_us"]["lmhead_argmax_isolated"]["launches"] >= 20
        assert "tolerance" in dec["parity"]
    for key in ("draft_top_tokens", "greedy_verify_small"):
        check_common(d[key], "rows/s")
        assert "bit-exact" in d[key]["parity"]


def test_tensor_parallel_line_one_rank():
    d = run_bench("--tp", "--rows", "512", "--steps", "16", "--warmup", "3", "--e2e-steps", "1")
    check_common(d, "rows/s")
    assert d["scaling"] == "strong" and d["exchange"]["bytes_per_rank"] == 512 * 8
    assert "bit-exact" in d["parity"]


def test_block_statistics_line_mixed_k():
    d = run_bench("--workload", "large_verify_blocks", "--mixed-k", "--rows", "400",
                  "--steps", "16", "--warmup", "3", "--e2e-steps", "1", "--cpu-seconds", "1")
    check_common(d, "rows/s")
    assert d["config"]["stats_per_row"] == 200
    assert "bit-exact" in d["parity"]


def test_lmhead_decode_line():
    d = run_bench("--workload", "lmhead", "--lmhead-rows", "4", "--lmhead-vocab", "32768",
                  "--steps", "5", "--warmup", "3", "--e2e-steps", "1", "--cpu-seconds", "1")
    check_common(d, "rows/s")
    assert d["roofline"]["bound"] == "hbm"            # M <= 128: a decode-size kernel
    assert d["roofline"]["traffic"] is None           # not the captured shape
    assert "tolerance" in d["parity"]
