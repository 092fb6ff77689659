"""Seeded synthetic inputs for the sharded greedy token-selection path.

This module only draws numbers and lays them out: it holds none of the
method's arithmetic (no argmax, no comparison, no acceptance rule), so the
CUDA path and the CPU oracle can both be fed from it without sharing any of
the computation they are checked on.

Shapes follow the workloads of the pages (vocabularies 40960 .. 202048,
drafts K = 1 .. 15, 1 .. 256 concurrent requests; vLLM PR #39419 Purpose,
PR #46448 Test, PR #62604 Results and Test Plan).  Logits are normal draws
rounded to bf16 with round-to-nearest-even (or kept fp32); the planted
values (ties, NaNs, padding spikes) are exact constants far outside the
normal range, so their effect is known without computing anything.
"""
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
BF16_NEG_INF = np.uint16(0xFF80)


def f32_to_bf16_bits(f):
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.
    Inputs must be finite (the generators plant NaN/inf as bits directly)."""
    u = np.ascontiguousarray(f, np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_const(x):
    """bf16 bits of an exactly representable constant."""
    return np.uint16(f32_to_bf16_bits(np.array([x], np.float32))[0])


def even_shards(vocab, num_shards):
    """(start, width) of each shard; the first vocab % S shards get one more id,
    as uneven TP splits of a vocab-parallel head do."""
    base, extra = divmod(vocab, num_shards)
    out, start = [], 0
    for s in range(num_shards):
        w = base + (1 if s < extra else 0)
        out.append((start, w))
        start += w
    return out


def _chunk_rng(seed, chunk):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(chunk)])))


def normal_matrix(seed, rows, cols, sigma, dtype="bf16", chunk_rows=64, threads=None):
    """rows x cols draws of N(0, sigma^2): uint16 bf16 bits or float32.
    Rows are drawn in fixed chunks, each from its own seeded stream, so the
    result does not depend on the number of threads."""
    out = np.empty((rows, cols), np.uint16 if dtype == "bf16" else np.float32)
    n_chunks = (rows + chunk_rows - 1) // chunk_rows

    def fill(c):
        r0, r1 = c * chunk_rows, min(rows, (c + 1) * chunk_rows)
        z = _chunk_rng(seed, c).standard_normal((r1 - r0, cols), dtype=np.float32)
        z *= np.float32(sigma)
        out[r0:r1] = f32_to_bf16_bits(z) if dtype == "bf16" else z

    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        nt = threads or min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def draft_plan(seed, num_reqs, k, p_accept, vocab):
    """Per draft position: a Bernoulli(p_accept) flag saying the draft copies
    the target's greedy token, and a uniform id in [0, vocab) used otherwise.
    Every request has k drafts; returns (cu_num_draft, flags, random_ids)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 7919])))
    flags = rng.random(num_reqs * k) < p_accept
    rand_ids = rng.integers(0, vocab, num_reqs * k, dtype=np.int64).astype(np.int32)
    cu = (np.arange(num_reqs + 1, dtype=np.int64) * k).astype(np.int32)
    return cu, flags, rand_ids


def draft_plan_mixed(seed, num_reqs, k_max, p_accept, vocab):
    """As draft_plan, with each request's draft count K_i drawn uniformly from
    1..k_max; returns (cu_num_draft, flags, random_ids)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 7920])))
    ks = rng.integers(1, k_max + 1, num_reqs)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    flags = rng.random(int(cu[-1])) < p_accept
    rand_ids = rng.integers(0, vocab, int(cu[-1]), dtype=np.int64).astype(np.int32)
    return cu, flags, rand_ids


def compose_drafts(target_ids, cu_num_draft, flags, rand_ids):
    """Draft tokens: draft j of request i is the given target token of row
    cu[i] + i + j where its flag is set, else its random id.  target_ids comes
    from whichever side is being fed (the oracle in tests)."""
    cu = np.asarray(cu_num_draft, np.int64)
    n = cu.size - 1
    req = np.repeat(np.arange(n), np.diff(cu))
    pos = np.arange(int(cu[-1])) - np.repeat(cu[:-1], np.diff(cu))
    rows = cu[req] + req + pos
    t = np.asarray(target_ids, np.int32)
    return np.where(flags, t[rows], rand_ids).astype(np.int32)


# --------------------------------------------------------------------------
# The five named workloads.  Each returns a dict: logits (uint16 bf16 bits or
# float32), shards [(start, width)], org_vocab, and for verify workloads the
# draft plan (cu_num_draft, flags, rand_ids, k).
# --------------------------------------------------------------------------

def tiny_sharded_argmax():
    """8 rows x vocab 1000 fp32 N(0,1), 2 shards of 500.  Row 3: equal maxima
    10.0 at ids 137 (shard 0) and 600 (shard 1).  Row 5: one NaN at id 777.
    Row 6: all -inf."""
    x = normal_matrix(1, 8, 1000, 1.0, dtype="f32")
    x[3, 137] = 10.0
    x[3, 600] = 10.0
    x[5, 777] = np.nan
    x[6, :] = -np.inf
    return dict(name="tiny sharded argmax: 8 x 1000 fp32, 2 shards",
                logits=x, shards=even_shards(1000, 2), org_vocab=1000)


def draft_top_tokens():
    """32 rows x padded vocab 152064 bf16 N(0,2), org_vocab 151936, 2 shards
    of 76032.  Rows r % 4 == 0 also get +100 at id 151940 and NaN at 152000,
    both padding."""
    x = normal_matrix(2, 32, 152064, 2.0)
    x[0::4, 151940] = bf16_const(100.0)
    x[0::4, 152000] = BF16_NAN
    return dict(name="draft get_top_tokens: 32 x 152064 bf16 (org 151936), 2 shards",
                logits=x, shards=even_shards(152064, 2), org_vocab=151936)


def greedy_verify_small():
    """24 requests x (K=3 + 1) rows, vocab 200064 bf16 N(0,3), 4 shards;
    drafts copy the target w.p. 0.7."""
    n, k, v = 24, 3, 200064
    x = normal_matrix(3, n * (k + 1), v, 3.0)
    cu, flags, rand_ids = draft_plan(3, n, k, 0.7, v)
    return dict(name="greedy verify: 24 req x (3+1) rows x 200064 bf16, 4 shards",
                logits=x, shards=even_shards(v, 4), org_vocab=v, k=k,
                cu_num_draft=cu, flags=flags, rand_ids=rand_ids)


LARGE_TIE_VALUE = 64.0  # > 21 sigma of N(0, 3): no normal draw reaches it


def plant_edge_ties(x, shards, every=100):
    """Rows r % every == 0 get an exact tie at LARGE_TIE_VALUE on ids
    (o_s - 1, o_s) for shard s = 1 + (r / every) % (S - 1); the lower id,
    which sits in the previous shard, is the expected winner."""
    hi = bf16_const(LARGE_TIE_VALUE)
    for r in range(0, x.shape[0], every):
        s = 1 + (r // every) % (len(shards) - 1)
        o = shards[s][0]
        x[r, o - 1] = hi
        x[r, o] = hi
    return x


def large_verify(rows_limit=None):
    """256 requests x (K=15 + 1) = 4096 rows x vocab 202048 bf16 N(0,3), 3
    uneven shards 67350/67349/67349, 1% of rows with an exact tie across a
    shard edge; drafts copy the target w.p. 0.6.  rows_limit keeps only the
    first requests (whole requests) for a smaller sample of the same recipe."""
    n, k, v = 256, 15, 202048
    if rows_limit is not None:
        n = max(1, min(n, rows_limit // (k + 1)))
    shards = even_shards(v, 3)
    x = normal_matrix(4, n * (k + 1), v, 3.0)
    plant_edge_ties(x, shards)
    cu, flags, rand_ids = draft_plan(4, n, k, 0.6, v)
    return dict(name="large verify: 256 req x (15+1) = 4096 rows x 202048 bf16, 3 uneven shards",
                logits=x, shards=shards, org_vocab=v, k=k,
                cu_num_draft=cu, flags=flags, rand_ids=rand_ids)


def large_verify_mixed_k(rows_limit=None):
    """The large-verify recipe with draft lengths that differ per request: 256
    requests with K_i uniform in 1..15 (about 2300 rows) x vocab 202048 bf16
    N(0,3), 3 uneven shards, 1% edge ties, drafts copy the target w.p. 0.6.
    rows_limit keeps only the first requests (whole requests)."""
    n, k, v = 256, 15, 202048
    cu, flags, rand_ids = draft_plan_mixed(6, n, k, 0.6, v)
    if rows_limit is not None:
        n = max(1, int(np.searchsorted(cu[1:] + np.arange(1, n + 1), rows_limit, "right")))
        cu, flags, rand_ids = cu[:n + 1], flags[:cu[n]], rand_ids[:cu[n]]
    rows = int(cu[-1]) + n
    shards = even_shards(v, 3)
    x = normal_matrix(6, rows, v, 3.0)
    plant_edge_ties(x, shards)
    return dict(name=f"large verify, mixed K: 256 req x (K_i in 1..15, + 1) = {rows} rows x "
                     "202048 bf16, 3 uneven shards",
                logits=x, shards=shards, org_vocab=v, k=k,
                cu_num_draft=cu, flags=flags, rand_ids=rand_ids)


def fused_lmhead(m=512, h=4096, vocab=151936, num_shards=2):
    """hidden m x h bf16 N(0,1) and an LM-head weight vocab x h bf16
    N(0, 0.02), split into num_shards vocab shards."""
    hidden = normal_matrix(5, m, h, 1.0)
    weight = normal_matrix(50005, vocab, h, 0.02, chunk_rows=1024)
    return dict(name=f"fused LM-head + argmax: {m} x {h} . [{vocab} x {h}]^T bf16, "
                     f"{num_shards} shards",
                hidden=hidden, weight=weight, shards=even_shards(vocab, num_shards),
                org_vocab=vocab)


# --------------------------------------------------------------------------
# Small randomized cases for sweeps: values from a short list (so ties, +-0,
# +-inf and NaN occur often), or normal draws.
# --------------------------------------------------------------------------

SPECIAL_VALUES = np.array([-np.inf, -2.0, -1.0, -0.0, 0.0, 1.0, 2.0, 3.0, np.inf, np.nan],
                          np.float32)


def discrete_logits(seed, rows, vocab, dtype="f32", p_nan=0.02, p_inf=0.02, levels=4):
    """Logits drawn from a few levels so that ties are frequent, with some
    +inf, -inf, NaN, +0 and -0 mixed in."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 17])))
    x = rng.integers(-levels, levels, (rows, vocab)).astype(np.float32)
    u = rng.random((rows, vocab))
    x[u < p_nan] = np.nan
    x[(u >= p_nan) & (u < p_nan + p_inf)] = np.inf
    x[(u >= p_nan + p_inf) & (u < p_nan + 2 * p_inf)] = -np.inf
    zero = (x == 0) & (rng.random((rows, vocab)) < 0.5)
    x[zero] = -0.0
    if dtype == "f32":
        return x
    bits = np.empty(x.shape, np.uint16)
    finite = np.isfinite(x)
    bits[finite] = f32_to_bf16_bits(x[finite])
    bits[np.isnan(x)] = BF16_NAN
    bits[x == np.inf] = np.uint16(0x7F80)
    bits[x == -np.inf] = BF16_NEG_INF
    return bits


def random_shards(seed, vocab, num_shards):
    """Ascending shards of random positive widths covering [0, vocab)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 29])))
    if num_shards == 1:
        return [(0, vocab)]
    cuts = np.sort(rng.choice(np.arange(1, vocab), num_shards - 1, replace=False))
    edges = [0] + [int(c) for c in cuts] + [vocab]
    return [(edges[i], edges[i + 1] - edges[i]) for i in range(num_shards)]


# --------------------------------------------------------------------------
# FP8 (OCP E4M3, "e4m3fn") inputs for the fp8 LM head: values are scaled so
# that the largest magnitude maps to 448 (the largest finite E4M3 value) and
# rounded to the nearest code, ties to the even code.
# --------------------------------------------------------------------------

def _e4m3_positive_table():
    codes = np.arange(0x7F, dtype=np.uint8)          # +0 .. 448, NaN (0x7F) excluded
    e = ((codes >> 3) & 0xF).astype(np.int32)
    m = (codes & 0x7).astype(np.float64)
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return codes, v


def f32_to_e4m3(x):
    """Round finite values with |x| <= 448 to E4M3 codes (nearest, ties to even)."""
    codes, v = _e4m3_positive_table()
    a = np.abs(np.asarray(x, np.float64))
    i = np.clip(np.searchsorted(v, a), 1, len(v) - 1)
    lo, hi = v[i - 1], v[i]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & (codes[i] % 2 == 0))
    c = np.where(pick_hi, codes[i], codes[i - 1]).astype(np.uint8)
    c = np.where(a == 0, np.uint8(0), c)
    return (c | (np.signbit(x).astype(np.uint8) << 7)).astype(np.uint8)


def quantize_rows_e4m3(x, threads=None, chunk_rows=1024):
    """Per-row scale s_r = max|x_r| / 448 and codes of x_r / s_r."""
    out = np.empty(x.shape, np.uint8)
    scale = np.empty(x.shape[0], np.float32)

    def work(c):
        r0, r1 = c * chunk_rows, min(x.shape[0], (c + 1) * chunk_rows)
        m = np.abs(x[r0:r1]).max(axis=1).astype(np.float32)
        s = np.where(m > 0, m / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        scale[r0:r1] = s
        out[r0:r1] = f32_to_e4m3(x[r0:r1] / s[:, None])

    n = (x.shape[0] + chunk_rows - 1) // chunk_rows
    with ThreadPoolExecutor(threads or min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(n)))
    return out, scale


def quantize_tensor_e4m3(x, threads=None, chunk_rows=1024):
    """One scale s = max|x| / 448 for the whole tensor, and codes of x / s."""
    s = np.float32(np.abs(x).max() / 448.0) or np.float32(1.0)
    out = np.empty(x.shape, np.uint8)

    def work(c):
        r0, r1 = c * chunk_rows, min(x.shape[0], (c + 1) * chunk_rows)
        out[r0:r1] = f32_to_e4m3(x[r0:r1] / s)

    n = (x.shape[0] + chunk_rows - 1) // chunk_rows
    with ThreadPoolExecutor(threads or min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(n)))
    return out, s


def fused_lmhead_fp8(m=512, h=4096, vocab=151936, num_shards=2):
    """The fused LM-head shapes with E4M3 operands: hidden N(0,1) quantized
    per row, weight N(0, 0.02) quantized per tensor."""
    hq, hs = quantize_rows_e4m3(normal_matrix(5, m, h, 1.0, dtype="f32"))
    wq, ws = quantize_tensor_e4m3(normal_matrix(50005, vocab, h, 0.02, dtype="f32", chunk_rows=1024))
    return dict(name=f"fused LM-head + argmax, fp8 e4m3: {m} x {h} . [{vocab} x {h}]^T, "
                     f"{num_shards} shards",
                hidden=hq, hidden_scale=hs, weight=wq, weight_scale=float(ws),
                shards=even_shards(vocab, num_shards), org_vocab=vocab)
