"""Writes the expected statistics of every row of the fused LM-head workload
(512 x 4096 hidden states against a 151936 x 4096 head in 2 vocab shards),
bf16 and fp8, from the CPU oracle alone.

    python tests/golden/make_lmhead_golden.py [bf16|fp8 ...]

Each output file lists, per hidden row, the oracle's fp64 argmax over the
whole vocabulary (id, top-1 logit, largest logit at any other id) and the
same three numbers for each vocab shard.  The tolerance rule of the fused
LM head is applied to the GPU path against these numbers: ids equal where
top-1 minus top-2 exceeds 1e-2, values within 1e-2 relative (vLLM PR #62604,
Purpose: vocab-parallel LM head, item 2: fused get_top_tokens with the same
result as torch.argmax over the logits).

The inputs are the seeded draws of workloads.fused_lmhead /
workloads.fused_lmhead_fp8; a digest of their bytes heads each file so a test
can confirm that it regenerated the same inputs before comparing.  Only the
oracle computes anything here.
"""
import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as wl  # noqa: E402

FILES = {"bf16": "lmhead_workload_bf16.txt", "fp8": "lmhead_workload_fp8.txt"}


def input_digest(c):
    """sha256 (first 16 hex digits) of the workload's input bytes."""
    h = hashlib.sha256()
    for key in ("hidden", "hidden_scale", "weight"):
        if key in c:
            h.update(np.ascontiguousarray(c[key]).tobytes())
    if "weight_scale" in c:
        h.update(np.float32(c["weight_scale"]).tobytes())
    return h.hexdigest()[:16]


def workload(kind):
    return wl.fused_lmhead() if kind == "bf16" else wl.fused_lmhead_fp8()


def oracle_logits(kind, c, rows):
    if kind == "bf16":
        return oracle.lmhead_logits(c["hidden"], c["weight"], rows)
    return oracle.lmhead_logits_fp8(c["hidden"], c["hidden_scale"], c["weight"],
                                    c["weight_scale"], rows)


def write(kind, chunk=8):
    c = workload(kind)
    M = c["hidden"].shape[0]
    shards, org = c["shards"], c["org_vocab"]
    lines = [
        f"# Oracle statistics of every row of the fused LM-head workload ({kind}):",
        f"# {c['name']}.",
        "# Written by tests/golden/make_lmhead_golden.py from the CPU oracle alone",
        "# (fp64 dot products in k order of the exactly widened inputs).",
        "# Source: vLLM PR #62604, Purpose (vocab-parallel LM head) and item 2",
        "# (fused get_top_tokens, same result as torch.argmax on the logits).",
        f"# input_digest: {input_digest(c)}",
        f"# rows: {M}",
        "# shards: " + " ".join(f"{o}:{w}" for o, w in shards),
        f"# org_vocab: {org}",
        "# Columns: row | id top1 top2 (whole vocab) | id top1 top2 of shard 0 | ...",
    ]
    t0 = time.perf_counter()
    for r0 in range(0, M, chunk):
        rows = np.arange(r0, min(M, r0 + chunk), dtype=np.int64)
        logits = oracle_logits(kind, c, rows)
        top1, top2, ids = oracle.argmax_f64(logits, 0, org)
        per_shard = [oracle.argmax_f64(logits[:, o:o + w], o, org) for o, w in shards]
        for q, r in enumerate(rows):
            cols = [f"{int(ids[q])} {float(top1[q])!r} {float(top2[q])!r}"]
            for s1, s2, sid in per_shard:
                cols.append(f"{int(sid[q])} {float(s1[q])!r} {float(s2[q])!r}")
            lines.append(f"{int(r)} | " + " | ".join(cols))
        print(f"{kind}: {rows[-1] + 1}/{M} rows, {time.perf_counter() - t0:.0f} s",
              file=sys.stderr, flush=True)
    with open(os.path.join(HERE, FILES[kind]), "w") as f:
        f.write("\n".join(lines) + "\n")


def read(kind):
    """Parsed golden file: dict(input_digest, shards, org_vocab, rows) where
    rows[r] = ((id, top1, top2), [(id, top1, top2) per shard])."""
    meta, rows = {}, {}
    with open(os.path.join(HERE, FILES[kind])) as f:
        for line in f:
            line = line.strip()
            if line.startswith("#"):
                if ":" in line:
                    k, v = line[1:].split(":", 1)
                    meta[k.strip()] = v.strip()
                continue
            if not line:
                continue
            parts = [p.split() for p in line.split("|")]
            r = int(parts[0][0])
            trip = [(int(p[0]), float(p[1]), float(p[2])) for p in parts[1:]]
            rows[r] = (trip[0], trip[1:])
    shards = [tuple(int(v) for v in s.split(":")) for s in meta["shards"].split()]
    return dict(input_digest=meta["input_digest"], shards=shards,
                org_vocab=int(meta["org_vocab"]), rows=rows)


if __name__ == "__main__":
    for kind in (sys.argv[1:] or ["bf16", "fp8"]):
        write(kind)
