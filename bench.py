#!/usr/bin/env python3
"""Benchmark of the TurboQuant packed-KV hot path on GB300.

Workload (the long-context 3.5-bit decode): batch 4, 32 query / 8 KV heads,
head_dim 128, context lengths drawn uniform in [65536, 131072] per sequence,
K 3-bit packed at every position, V 4-bit packed with the newest 256 tokens
kept as an fp16 ring.  One step is one pass of the whole hot path for a
decode step: append one new token per sequence (quantize K and V of all
heads, quantizing the V token that leaves the ring) and decode attention of
every query head over the whole cache (query rotation, split-K scoring with
online softmax and V accumulation, merge and inverse rotation).  Lengths grow
by one per step; the cache has head-room for the steps.

Reported: decode-attention algorithmic HBM GB/s (packed K+V+norms, hot fp16 V,
q, out per step) over the timed steps, its fraction of the measured HBM peak,
quantize throughput (Mtokens/s) on the batch 16 x 8192-token x 8-head
append at 3.5 bits, an end-to-end number through the public API with host
buffers, and the CPU oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_10_gb300 import synth  # noqa: E402

METRIC = "packed-KV decode-attn HBM GB/s (% roofline) & quantize Mtokens/s, 1 GB300"
SEED = 5
B, HQ, HKV, D, W = 4, 32, 8, 128, 256
KB, VB = 3, 4
LO, HI = 65536, 131072
QB, QT = 16, 8192  # quantize workload: batch x new tokens (8 KV heads)
FALLBACK_HBM_GBS = 6800.0
# float32 multiply-add peak: 152 SMs x 128 FMA lanes x 2.07 GHz (maximum SM clock)
FP32_FMA_PEAK = 152 * 128 * 2.07e9
WORKLOAD = ("long-context 3.5-bit decode: B4, 32q/8kv heads, d128, L~U[65536,131072] (+1 per step), "
            "K 3-bit packed, V 4-bit packed + 256-token fp16 hot window; step = append 1 token per "
            "sequence (quantize + ring evict) + decode attention of all query heads")


def decode_bytes(lens) -> int:
    """Algorithmic bytes of one decode step: packed K + norms at every
    position, packed V + norms on the cold part, fp16 V on the hot part,
    the fp16 queries and the float32 outputs."""
    total = 0
    for L in lens:
        L = int(L)
        hot = min(W, L)
        total += HKV * (L * (D * KB // 8 + 4) + (L - hot) * (D * VB // 8 + 4) + hot * D * 2)
    return total + len(lens) * HQ * D * (2 + 4)


def max_over_ranks(ms: float, world: int, dist=None, device="cpu") -> float:
    """Duration of the whole job's timed region: the maximum over the ranks
    (every rank runs the same replica workload, so the slowest one ends it)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms: float, world: int) -> float:
    """Whole-job throughput in units x 1e9 per second: `world` replicas each
    processed `units_per_rank` within `ms` milliseconds."""
    return world * units_per_rank / (ms * 1e-3) / 1e9


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# the sources of the long-context decode call (split kernels, dispatch, merge and entry points)
DECODE_SAMPLE = 8  # one timed step in DECODE_SAMPLE has its decode call bracketed by events
DECODE_SOURCES = ("tq_decode_mma.cuh", "tq_decode_split.cuh", "tq_split_plan.h", "tq_decode_dispatch.cuh", "tq_decode.cu")


def profile_traffic():
    """dram bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel sources (DECODE_SOURCES); else None."""
    path = os.path.join(ROOT, "profiles", "decode_long_context.md")
    csrc = os.path.join(ROOT, "bit_kv_cache_10_gb300", "csrc")
    try:
        text = open(path).read()
        src = b"".join(open(os.path.join(csrc, f), "rb").read() for f in DECODE_SOURCES)
        sha = hashlib.sha256(src).hexdigest()[:16]
        m = re.search(r"traffic_bytes_per_step:\s*([0-9]+)", text)
        s = re.search(r"decode_source_sha256_16:\s*([0-9a-f]+)", text)
        if m and s and s.group(1) == sha:
            return int(m.group(1))
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = os.path.join("/tmp", "tq_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> list:
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.out):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    pass
        os.unlink(self.out)
        return rows

    @staticmethod
    def summarize(rows, source):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": source}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "source": source}


# ----------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------

_ROWS: dict = {}


def _oracle_row_cache(lens, b, h, n_tokens):
    """The oracle's view of one (batch, KV head) row of the bench cache,
    restricted to its first n_tokens positions (a bounded sample; the row
    generators are prefix-consistent, so this equals a slice of the full row)."""
    import oracle
    key = (b, h, n_tokens)
    if key not in _ROWS:
        if len(_ROWS) > 64:
            _ROWS.clear()
        kw, kn = synth.packed_row(SEED, synth.STREAM_CODES_K, b, h, n_tokens, D * KB // 32, 12.0)
        vw, vn = synth.packed_row(SEED, synth.STREAM_CODES_V, b, h, n_tokens, D * VB // 32, 30.0)
        ring = synth.kv_fp16(SEED, synth.STREAM_V, B, HKV, W, D,
                             synth.channel_scales(SEED, synth.STREAM_SCALE_V, HKV, D))[b:b + 1, h:h + 1]
        _ROWS[key] = oracle.PackedCache(0, 0, D, KB, VB, kw[None, None], kn[None, None], None, vw[None, None],
                                        vn[None, None], W, ring)
    return _ROWS[key]


def oracle_sample_step(lens, q16, b, h, n_tokens):
    """Oracle decode of the G query heads of one (b, h) row over its first
    n_tokens positions; returns (seconds, algorithmic bytes)."""
    import oracle
    c = _oracle_row_cache(lens, b, h, n_tokens)
    g = HQ // HKV
    t0 = time.perf_counter()
    k, v = oracle.dequantized_kv(c, 0, 0, n_tokens)
    for j in range(g):
        oracle.attention_one(q16[b, h * g + j].astype(np.float64), k, v)
    dt = time.perf_counter() - t0
    hot = min(W, n_tokens)
    nbytes = n_tokens * (D * KB // 8 + 4) + (n_tokens - hot) * (D * VB // 8 + 4) + hot * D * 2 + g * D * 6
    return dt, nbytes


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_task(args):
    """One oracle row in a worker process: (seconds, algorithmic bytes)."""
    lens, q16, b, h, n = args
    return oracle_sample_step(lens, q16, b, h, n)


def _oracle_quant_task(args):
    """Oracle quantize of n token vectors of K and of V of one (batch, KV head)
    of the quantize workload (N(0,1) x lognormal channel scales) in a worker
    process, K at kb and V at vb bits: (seconds, token-heads)."""
    import oracle
    b, h, n = args[:3]
    kb, vb = args[3:] if len(args) > 3 else (KB, VB)
    rows = []
    for stream, scale_stream in ((synth.STREAM_K, synth.STREAM_SCALE_K), (synth.STREAM_V, synth.STREAM_SCALE_V)):
        s = synth.channel_scales(SEED + 2, scale_stream, HKV, D)[h]
        rows.append((synth.row_rng(SEED + 2, stream, b, h).standard_normal((n, D)) * s).astype(np.float16))
    rot = oracle.rotation(0, 0, h, D)
    cbs = (oracle.codebook(D, kb), oracle.codebook(D, vb))  # built (or cached) outside the timed part
    t0 = time.perf_counter()
    for x, bits, cb in zip(rows, (kb, vb), cbs):
        codes, _, _ = oracle.quantize_rows(x, rot, cb)
        oracle.pack(codes, bits)
    return time.perf_counter() - t0, n


def _oracle_plain_task(args):
    """Oracle decode of the 4 query heads of one (batch, KV head) row of a
    plain (no hot window) decode workload of context n: packed K (k_fp16 False)
    or fp16 K drawn N(0,1) x lognormal channel scales, packed 4-bit V.  Returns
    (seconds, algorithmic bytes)."""
    import oracle
    seed, b, h, n, k_fp16 = args
    g = HQ // HKV
    vw, vn = synth.packed_row(seed, synth.STREAM_CODES_V, b, h, n, D * VB // 32, 30.0)
    if k_fp16:
        sk = synth.channel_scales(seed, synth.STREAM_SCALE_K, HKV, D)
        k16 = synth.kv_fp16(seed + b, synth.STREAM_K, 1, HKV, n, D, sk)[:, h:h + 1]
        c = oracle.PackedCache(0, 0, D, 16, VB, None, None, k16, vw[None, None], vn[None, None], 0, None)
        k_bytes = n * D * 2
    else:
        kw, kn = synth.packed_row(seed, synth.STREAM_CODES_K, b, h, n, D * KB // 32, 12.0)
        c = oracle.PackedCache(0, 0, D, KB, VB, kw[None, None], kn[None, None], None, vw[None, None],
                               vn[None, None], 0, None)
        k_bytes = n * (D * KB // 8 + 4)
    q16 = synth.queries_fp16(seed, b + 1, HQ, D)[b]
    t0 = time.perf_counter()
    k, v = oracle.dequantized_kv(c, 0, 0, n)
    for j in range(g):
        oracle.attention_one(q16[h * g + j].astype(np.float64), k, v)
    return time.perf_counter() - t0, k_bytes + n * (D * VB // 8 + 4) + g * D * 6


def oracle_pool():
    """Spawned worker processes, one per host core, each with single-threaded
    BLAS, so that independent (batch, KV head) rows run on all cores."""
    import concurrent.futures
    import multiprocessing
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    n = cpu_cores()
    return concurrent.futures.ProcessPoolExecutor(max_workers=n, mp_context=multiprocessing.get_context("spawn")), n


def pooled_rows(pool, tasks):
    """Runs the row tasks on the pool; returns (wall seconds, algorithmic bytes)."""
    t0 = time.perf_counter()
    nbytes = sum(nb for _, nb in pool.map(_oracle_task, tasks))
    return time.perf_counter() - t0, nbytes


def cpu_baseline(lens, q16, pool, workers, rounds=4):
    """The oracle on all host cores: `rounds` passes over the 32 (batch, KV head)
    rows of the workload at full context, one row per task."""
    tasks = [(lens, q16, b, h, int(lens[b])) for _ in range(rounds) for b in range(B) for h in range(HKV)]
    pooled_rows(pool, tasks[:workers])  # start-up of the workers, untimed
    wall, nbytes = pooled_rows(pool, tasks)
    # quantize: 2048-token slices of (batch, KV head) rows of the quantize workload, K 3-bit and V 4-bit
    qtasks = [(i % QB, (i // QB) % HKV, 2048) for i in range(4 * workers)]
    list(pool.map(_oracle_quant_task, qtasks[:workers]))  # untimed: codebooks built in every worker
    t0 = time.perf_counter()
    token_heads = sum(n for _, n in pool.map(_oracle_quant_task, qtasks))
    qwall = time.perf_counter() - t0
    widths = {}
    for kb, vb in ((3, 3), (4, 4)):
        wt = [t + (kb, vb) for t in qtasks]
        t0 = time.perf_counter()
        th = sum(n for _, n in pool.map(_oracle_quant_task, wt))
        widths["%d" % kb] = {"value": th / HKV / (time.perf_counter() - t0) / 1e6, "unit": "Mtokens/s"}
    # the other decode workloads, every (batch, KV head) row of the Llama-like layer
    # (B1, context 4096) and 2 rows per worker of the asym workload (B8, context 16384)
    plain = {}
    for name, seed, batch, ctx, k_fp16, n_rows in (("llama_layer", SEED + 3, 1, 4096, False, HKV),
                                                   ("asym", SEED + 3, 8, 16384, True, 2 * workers)):
        ptasks = [(seed, (i // HKV) % batch, i % HKV, ctx, k_fp16) for i in range(n_rows)]
        t0 = time.perf_counter()
        pb = sum(nb for _, nb in pool.map(_oracle_plain_task, ptasks))
        plain[name] = {"value": pb / (time.perf_counter() - t0) / 1e9, "unit": "GB/s",
                       "sample": "%d (batch, KV head) rows at full context %d" % (n_rows, ctx)}
    return {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": workers, "kind": "oracle",
            "llama_layer": plain["llama_layer"], "asym": plain["asym"],
            "sample": "%d (batch, KV head) rows of the workload at full context (%.2f GB of algorithmic bytes) on "
                      "%d worker processes with single-threaded BLAS: numpy float64 dequantize + softmax attention "
                      "for the 4 query heads of each row" % (len(tasks), nbytes / 1e9, workers),
            "quantize": {"value": token_heads / HKV / qwall / 1e6, "unit": "Mtokens/s",
                         "sample": "%d slices of 2048 tokens of one (batch, KV head) of the quantize workload, K 3-bit "
                                   "and V 4-bit (a token = one position with all 8 KV heads)" % len(qtasks),
                         "widths": widths}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    lens = synth.seq_lengths(SEED, B, LO, HI)
    q16 = synth.queries_fp16(SEED, B, HQ, D)
    pool, workers = oracle_pool()
    # size each step (one row per worker) so that the whole run stays within a few minutes
    dt_cal, nb_cal = oracle_sample_step(lens, q16, 0, 0, 4096)
    rate = nb_cal / dt_cal  # bytes/s of one core
    per_row_bytes = max(200_000.0, min(rate * 100.0 / max(1, args.steps + args.warmup), 5e8))
    bytes_per_token = (D * KB // 8 + 4) + (D * VB // 8 + 4)
    n_tok = int(max(512, min(HI, per_row_bytes / bytes_per_token)))

    def step_tasks(s):
        return [(lens, q16, (s * workers + i) % B, ((s * workers + i) // B) % HKV,
                 min(n_tok, int(lens[(s * workers + i) % B]))) for i in range(workers)]
    for s in range(args.warmup):
        pooled_rows(pool, step_tasks(s))
    tt, tb = 0.0, 0
    for s in range(args.steps):
        dt, nb = pooled_rows(pool, step_tasks(args.warmup + s))
        tt += dt
        tb += nb
    pool.shutdown()
    value = tb / tt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "host cores (oracle)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle", "cores": workers,
                         "sample": "per step one (batch, KV head) row per worker process (%d processes, "
                                   "single-threaded BLAS), first %d context positions of each row, float64 "
                                   "dequantize + attention for its 4 query heads" % (workers, n_tok)},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def build_decode_cache(torch, cap):
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    lens = synth.seq_lengths(SEED, B, LO, HI)
    tc = TurboQuantKVCache(B, HKV, HQ, cap, bits=(KB, VB), hot_window=W)
    for b in range(B):
        L = int(lens[b])
        for h in range(HKV):
            kw, kn = synth.packed_row(SEED, synth.STREAM_CODES_K, b, h, L, D * KB // 32, 12.0)
            vw, vn = synth.packed_row(SEED, synth.STREAM_CODES_V, b, h, L, D * VB // 32, 30.0)
            tc.k_cache[b, h, :L].copy_(torch.from_numpy(kw.view(np.int32)))
            tc.k_norms[b, h, :L].copy_(torch.from_numpy(kn))
            tc.v_cache[b, h, :L].copy_(torch.from_numpy(vw.view(np.int32)))
            tc.v_norms[b, h, :L].copy_(torch.from_numpy(vn))
    ring = synth.kv_fp16(SEED, synth.STREAM_V, B, HKV, W, D, synth.channel_scales(SEED, synth.STREAM_SCALE_V, HKV, D))
    tc.v_hot.copy_(torch.from_numpy(ring))
    torch.cuda.synchronize()
    return tc, lens


def build_plain_cache(torch, batch, ctx, k_fp16, seed):
    """Decode cache of `batch` sequences of length ctx, no hot window: packed V (and
    packed K) rows of random words with lognormal norms, or fp16 K drawn
    N(0,1) x lognormal channel scales."""
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    tc = TurboQuantKVCache(batch, HKV, HQ, ctx, bits=(KB, VB), k_fp16=k_fp16)
    if k_fp16:
        sk = synth.channel_scales(seed, synth.STREAM_SCALE_K, HKV, D)
        for b in range(batch):  # one sequence at a time to bound host memory
            k = synth.kv_fp16(seed + b, synth.STREAM_K, 1, HKV, ctx, D, sk)
            tc.k_cache[b].copy_(torch.from_numpy(k[0]))
    for b in range(batch):
        for h in range(HKV):
            if not k_fp16:
                kw, kn = synth.packed_row(seed, synth.STREAM_CODES_K, b, h, ctx, D * KB // 32, 12.0)
                tc.k_cache[b, h].copy_(torch.from_numpy(kw.view(np.int32)))
                tc.k_norms[b, h].copy_(torch.from_numpy(kn))
            vw, vn = synth.packed_row(seed, synth.STREAM_CODES_V, b, h, ctx, D * VB // 32, 30.0)
            tc.v_cache[b, h].copy_(torch.from_numpy(vw.view(np.int32)))
            tc.v_norms[b, h].copy_(torch.from_numpy(vn))
    torch.cuda.synchronize()
    return tc


def graph_call_ms(torch, fn, n):
    """Mean time (ms) of fn over n back-to-back calls captured as one CUDA graph
    and replayed once between two events (after 3 calls on the stream)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(n):
            fn()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    del graph
    return e0.elapsed_time(e1) / n


def time_plain_decode(torch, batch, ctx, k_fp16, reps=50, flush=False):
    """Mean decode-call time (ms) and algorithmic bytes of one call on a
    build_plain_cache cache, after 3 untimed calls.  With ``flush`` a 256 MB
    buffer (twice L2) is written before every call and only the call itself is
    between the events, so the cache is read from HBM; without it the calls run
    back to back, replayed as one CUDA graph."""
    tc = build_plain_cache(torch, batch, ctx, k_fp16, SEED + 3)
    q = torch.from_numpy(synth.queries_fp16(SEED + 3, batch, HQ, D)).cuda()
    lens = torch.full((batch,), ctx, dtype=torch.int32, device="cuda")
    out = torch.empty(batch, HQ, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(tc.workspace_bytes(ctx), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        tc.decode(q, lens, ctx, out=out, workspace=ws)
    st = torch.cuda.current_stream()
    if flush:
        scrub = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            scrub.fill_(1)
            e0.record(st)
            tc.decode(q, lens, ctx, out=out, workspace=ws)
            e1.record(st)
        torch.cuda.synchronize()
        ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in ev]))
        del scrub
    else:  # back-to-back calls, replayed as a CUDA graph
        ms = graph_call_ms(torch, lambda: tc.decode(q, lens, ctx, out=out, workspace=ws), reps)
    if tc.device_status() != 0:
        raise RuntimeError("device status set by the decode timing")
    k_tok = D * 2 if k_fp16 else D * KB // 8 + 4
    nbytes = batch * HKV * ctx * (k_tok + D * VB // 8 + 4) + batch * HQ * D * (2 + 4)
    del tc
    return ms, nbytes


# int8-mode scales giving K and V the magnitudes of the packed workload (|k| ~ 12,
# |v| ~ 30): a uniform random code has rms 73.3, a 128-vector of them norm ~ 829
INT8_K_SCALE, INT8_V_SCALE = 12.0 / 829.4, 30.0 / 829.4


def build_int8_cache(torch, lens, cap):
    """int8-mode cache (no hot window) with random codes and lognormal scales
    in rows [0, L_b) of every (b, h)."""
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    tc = TurboQuantKVCache(len(lens), HKV, HQ, cap, bits="int8")
    for b, L in enumerate(lens):
        L = int(L)
        for h in range(HKV):
            kw, ks = synth.packed_row(SEED + 7, synth.STREAM_CODES_K, b, h, L, D // 4, INT8_K_SCALE)
            vw, vs = synth.packed_row(SEED + 7, synth.STREAM_CODES_V, b, h, L, D // 4, INT8_V_SCALE)
            tc.k_cache[b, h, :L].copy_(torch.from_numpy(kw.view(np.int32)))
            tc.k_norms[b, h, :L].copy_(torch.from_numpy(ks))
            tc.v_cache[b, h, :L].copy_(torch.from_numpy(vw.view(np.int32)))
            tc.v_norms[b, h, :L].copy_(torch.from_numpy(vs))
    torch.cuda.synchronize()
    return tc


def time_int8(torch, lens, reps=20):
    """int8 mode on the long-context lengths: mean decode-call time (ms) and its
    algorithmic bytes (128 code bytes + a 4-byte scale for K and for V of every
    position, fp16 queries, float32 outputs); then the quantize-append time of
    the quantize workload (B16 x 8192 tokens x 8 heads)."""
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    cap = int(np.max(lens))
    tc = build_int8_cache(torch, lens, cap)
    q = torch.from_numpy(synth.queries_fp16(SEED + 7, len(lens), HQ, D)).cuda()
    sl = torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    out = torch.empty(len(lens), HQ, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(tc.workspace_bytes(cap), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()

    def timed(fn, n):
        for _ in range(3):
            fn()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        torch.cuda.synchronize()
        ev[0].record(st)
        for i in range(n):
            fn()
            ev[i + 1].record(st)
        torch.cuda.synchronize()
        return float(np.mean([ev[i].elapsed_time(ev[i + 1]) for i in range(n)]))

    dec_ms = graph_call_ms(torch, lambda: tc.decode(q, sl, cap, out=out, workspace=ws), reps)
    if tc.device_status() != 0:
        raise RuntimeError("device status set by the int8 decode timing")
    dec_bytes = int(np.sum(lens)) * HKV * 2 * (D + 4) + len(lens) * HQ * D * (2 + 4)
    del tc, ws
    kq, vq = quantize_inputs(torch)
    qc = TurboQuantKVCache(QB, HKV, HKV * 4, QT, bits="int8")
    zero = torch.zeros(QB, dtype=torch.int32, device="cuda")
    q_ms = timed(lambda: qc.append(kq, vq, zero), 10)
    if qc.device_status() != 0:
        raise RuntimeError("device status set by the int8 quantize timing")
    q_bytes = 2 * QB * HKV * QT * (D * 2 + D + 4)
    del kq, vq, qc
    return dec_ms, dec_bytes, q_ms, q_bytes


def paged_copy(torch, tc, bs=64, permute=True):
    """Block-table copy of the decode cache `tc`: blocks of `bs` tokens in a
    randomly permuted pool (or in order)."""
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    cap = (tc.capacity + bs - 1) // bs * bs
    mb = cap // bs
    nb = B * mb
    pg = TurboQuantKVCache(B, HKV, HQ, cap, bits=(KB, VB), hot_window=W, block_size=bs, num_blocks=nb)
    order = np.random.default_rng(SEED).permutation(nb) if permute else np.arange(nb)
    table = torch.from_numpy(order.astype(np.int32).reshape(B, mb)).cuda()
    pg.block_table.copy_(table)
    for name in ("k_cache", "k_norms", "v_cache", "v_norms"):
        src, dst = getattr(tc, name), getattr(pg, name)
        for b in range(B):
            full = torch.zeros((HKV, cap) + tuple(src.shape[3:]), dtype=src.dtype, device=src.device)
            full[:, :tc.capacity] = src[b]
            dst[table[b].long()] = full.view((HKV, mb, bs) + tuple(src.shape[3:])).transpose(0, 1)
    pg.v_hot.copy_(tc.v_hot)
    return pg


def paged_decode_ms(torch, tc, lens0, q, seqs, max_len, bs=64, reps=20, permute=True):
    """Mean decode-call time of a paged copy of `tc` (back-to-back calls replayed as
    one CUDA graph, after 3 calls on the stream)."""
    pg = paged_copy(torch, tc, bs, permute)
    out = torch.empty(B, HQ, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(pg.workspace_bytes(max_len), dtype=torch.uint8, device="cuda")
    ms = graph_call_ms(torch, lambda: pg.decode(q, seqs, max_len, out=out, workspace=ws), reps)
    if pg.device_status() != 0:
        raise RuntimeError("device status set by the paged decode")
    del pg
    return ms


def quantize_inputs(torch):
    """The quantize workload's new K and V tokens on the device: fp16 [16, 8, 8192,
    128], N(0,1) times lognormal(0,1) scales per (KV head, channel), drawn on the
    host one sequence at a time to bound host memory."""
    gq = synth.rng(SEED + 2, synth.STREAM_K)
    qsk = torch.from_numpy(synth.channel_scales(SEED + 2, synth.STREAM_SCALE_K, HKV, D).astype(np.float32)).cuda()
    qsv = torch.from_numpy(synth.channel_scales(SEED + 2, synth.STREAM_SCALE_V, HKV, D).astype(np.float32)).cuda()
    kq = torch.empty(QB, HKV, QT, D, dtype=torch.float16, device="cuda")
    vq = torch.empty_like(kq)
    for b in range(QB):
        kq[b].copy_((torch.from_numpy(gq.standard_normal((HKV, QT, D), dtype=np.float32)).cuda()
                     * qsk[:, None, :]).half())
        vq[b].copy_((torch.from_numpy(gq.standard_normal((HKV, QT, D), dtype=np.float32)).cuda()
                     * qsv[:, None, :]).half())
    return kq, vq


def time_quantize(torch, qc, kq, vq, zero, kb, vb, reps=10):
    """Quantize-append of the whole quantize workload into `qc` (K kb bits, V vb
    bits): mean time over `reps` calls after 3 untimed ones, Mtokens/s, HBM GB/s."""
    st = torch.cuda.current_stream()
    for _ in range(3):
        qc.append(kq, vq, zero)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record(st)
    for i in range(reps):
        qc.append(kq, vq, zero)
        ev[i + 1].record(st)
    torch.cuda.synchronize()
    if qc.device_status() != 0:
        raise RuntimeError("device status set by the quantize benchmark")
    ms = float(np.mean([ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]))
    tokens = kq.shape[0] * kq.shape[2]
    nbytes = 2 * kq.numel() * 2 + kq.shape[0] * HKV * kq.shape[2] * ((D * kb // 8 + 4) + (D * vb // 8 + 4))
    return {"k_bits": kb, "v_bits": vb, "ms": ms, "value": tokens / (ms * 1e-3) / 1e6, "unit": "Mtokens/s",
            "token_heads_per_s": tokens * HKV / (ms * 1e-3), "hbm_gbs": nbytes / (ms * 1e-3) / 1e9,
            "algorithmic_bytes_per_launch": nbytes}


def step_inputs(n_steps):
    """Per-step new K/V tokens [S, B, Hkv, 1, D] and queries [S, B, Hq, D], fp16."""
    g = synth.rng(SEED + 1, synth.STREAM_Q)
    q = g.standard_normal((n_steps, B, HQ, D), dtype=np.float32).astype(np.float16)
    sk = synth.channel_scales(SEED, synth.STREAM_SCALE_K, HKV, D).astype(np.float32)
    sv = synth.channel_scales(SEED, synth.STREAM_SCALE_V, HKV, D).astype(np.float32)
    gk = synth.rng(SEED + 1, synth.STREAM_K)
    gv = synth.rng(SEED + 1, synth.STREAM_V)
    k = (gk.standard_normal((n_steps, B, HKV, 1, D), dtype=np.float32) * sk[None, None, :, None, :]).astype(np.float16)
    v = (gv.standard_normal((n_steps, B, HKV, 1, D), dtype=np.float32) * sv[None, None, :, None, :]).astype(np.float16)
    return k, v, q


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from bit_kv_cache_10_gb300 import build as tq_build
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    pool, workers = oracle_pool() if want_cpu else (None, 0)  # spawned before any GPU work
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    if rank == 0:
        tq_build.build()
    if world > 1:
        dist.barrier()
    from bit_kv_cache_10_gb300 import native
    native.lib()

    e2e_steps, e2e_warm = max(3, min(args.steps, 500)), 3
    graph_steps = max(3, min(args.steps, 300))
    probe_steps = 10000
    total_steps = args.warmup + args.steps + e2e_warm + e2e_steps + 1 + graph_steps + probe_steps
    cap = HI + total_steps + 64
    tc, lens0 = build_decode_cache(torch, cap)
    kn, vn, qn = step_inputs(total_steps)
    k_dev = torch.from_numpy(kn).cuda()
    v_dev = torch.from_numpy(vn).cuda()
    q_dev = torch.from_numpy(qn).cuda()
    starts = torch.from_numpy((lens0[None, :] + np.arange(total_steps)[:, None]).astype(np.int32)).cuda()
    seqs = starts + 1
    max_len = HI + total_steps
    out = torch.empty(B, HQ, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(tc.workspace_bytes(max_len), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(s):
        tc.append(k_dev[s], v_dev[s], starts[s])
        tc.decode(q_dev[s], seqs[s], max_len, out=out, workspace=ws)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    # the timed steps, captured as one CUDA graph (the kernels of K steps in order,
    # without launch gaps between them) and replayed once; the decode call of every
    # DECODE_SAMPLE-th step is bracketed by two events that are nodes of the graph
    # (its duration, for the roofline).  Capturing runs nothing: the steps run in
    # the replay.
    sampled = list(range(0, args.steps, DECODE_SAMPLE))
    dev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * len(sampled))]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(args.steps):
            s = args.warmup + i
            tc.append(k_dev[s], v_dev[s], starts[s])
            if i % DECODE_SAMPLE == 0:
                dev[2 * (i // DECODE_SAMPLE)].record()
            tc.decode(q_dev[s], seqs[s], max_len, out=out, workspace=ws)
            if i % DECODE_SAMPLE == 0:
                dev[2 * (i // DECODE_SAMPLE) + 1].record()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.15)
    torch.cuda.synchronize()
    ev[0].record(stream)
    graph.replay()
    ev[1].record(stream)
    torch.cuda.synchronize()
    clock_rows = sampler.stop()
    total_ms = ev[0].elapsed_time(ev[1])
    decode_ms = [dev[2 * k].elapsed_time(dev[2 * k + 1]) for k in range(len(sampled))]
    del graph
    status = tc.device_status()
    if status != 0:
        raise RuntimeError("device status %#x during the benchmark" % status)
    step_bytes = [decode_bytes(lens0 + args.warmup + i + 1) for i in range(args.steps)]
    total_ms = max_over_ranks(total_ms, world, dist, "cuda")
    value = job_throughput(sum(step_bytes), total_ms, world)
    s0 = args.warmup + args.steps

    clocks = ClockSampler.summarize(clock_rows, "timed region")
    if clocks["samples"] < 3:  # timed region too short for nvidia-smi: sample a longer run of the same step
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        time.sleep(0.15)
        for i in range(probe_steps):
            step(total_steps - probe_steps + i)
        torch.cuda.synchronize()
        clocks = ClockSampler.summarize(sampler.stop(), "%d further steps right after the timed region "
                                                        "(the timed region was shorter than the sampling period)"
                                        % probe_steps)

    # sparse-V decode on the same cache (threshold 1e-3; the dense call above is the headline)
    tc.desc.sparse_v_threshold = 1e-3
    sv_s = args.warmup + args.steps
    sparse_ms = graph_call_ms(torch, lambda: tc.decode(q_dev[sv_s], seqs[sv_s], max_len, out=out, workspace=ws), 20)
    tc.desc.sparse_v_threshold = 0.0
    if tc.device_status() != 0:
        raise RuntimeError("device status set by the sparse-V decode")
    # speculative verification on the same cache: the 8 newest tokens of every
    # sequence attend causally (each query one more sequence of the split work list)
    mq_n = 8
    mq_q = torch.from_numpy(synth.queries_fp16(SEED + 9, B * mq_n, HQ, D).reshape(B, mq_n, HQ, D)).cuda()
    mq_out = torch.empty(B, mq_n, HQ, D, dtype=torch.float32, device="cuda")
    mq_ws = torch.empty(native.tq_multi_query_workspace_bytes(tc.desc, mq_n, max_len), dtype=torch.uint8,
                        device="cuda")
    mq_ms = graph_call_ms(torch, lambda: tc.multi_query(mq_q, seqs[sv_s], max_len, out=mq_out, workspace=mq_ws), 10)
    if tc.device_status() != 0:
        raise RuntimeError("device status set by the multi-query attention")
    mq_lens = lens0 + sv_s + 1
    mq_pairs = int(sum(max(0, int(L) - mq_n + i + 1) for L in mq_lens for i in range(mq_n)))  # (query, key) pairs
    mq_fma = mq_pairs * HQ * 2 * D  # score and V multiply-adds per (query, key, head)

    # paged layout: the same cache copied into 64-token blocks scattered over a pool
    paged_ms = paged_decode_ms(torch, tc, lens0, q_dev[sv_s], seqs[sv_s], max_len)
    paged_inorder_ms = paged_decode_ms(torch, tc, lens0, q_dev[sv_s], seqs[sv_s], max_len, permute=False)

    # end to end through the public API with host buffers: each step's new K and V
    # tokens, queries, start positions and lengths packed in one pinned host record
    # (one host-to-device copy per step; every part 16-byte aligned), the output
    # read back into pinned host memory.  Copies run on their own streams into
    # double buffers, ordered by events: the record of step s + 1 uploads while
    # step s computes, and the output of step s downloads while step s + 1 computes
    starts_h = (lens0[None, :] + np.arange(total_steps)[:, None]).astype(np.int32)
    parts = [kn.reshape(total_steps, -1).view(np.uint8), vn.reshape(total_steps, -1).view(np.uint8),
             qn.reshape(total_steps, -1).view(np.uint8), starts_h.view(np.uint8), (starts_h + 1).view(np.uint8)]
    offs = np.cumsum([0] + [pt.shape[1] for pt in parts])
    assert all(o % 16 == 0 for o in offs[:-1])
    h_rec = torch.from_numpy(np.ascontiguousarray(np.concatenate(parts, axis=1))).pin_memory()
    h_outs = [torch.empty(B, HQ, D, dtype=torch.float32).pin_memory() for _ in range(2)]
    d_recs = [torch.empty(h_rec.shape[1], dtype=torch.uint8, device="cuda") for _ in range(2)]
    d_outs = [torch.empty(B, HQ, D, dtype=torch.float32, device="cuda") for _ in range(2)]

    def rec_views(d_rec):  # (k, v, q, start positions, lengths) of a device record
        return (d_rec[offs[0]:offs[1]].view(torch.float16).view(k_dev[0].shape),
                d_rec[offs[1]:offs[2]].view(torch.float16).view(v_dev[0].shape),
                d_rec[offs[2]:offs[3]].view(torch.float16).view(q_dev[0].shape),
                d_rec[offs[3]:offs[4]].view(torch.int32), d_rec[offs[4]:offs[5]].view(torch.int32))

    views = [rec_views(d) for d in d_recs]
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]  # record i uploaded
    done = [torch.cuda.Event() for _ in range(2)]      # the step that used record / output i computed
    out_read = [torch.cuda.Event() for _ in range(2)]  # output i downloaded

    first_use = [True, True]  # no earlier step has used record / output i yet

    def e2e_step(s, cs):
        """Step s on compute stream cs: upload, append + decode, download."""
        i = s % 2
        d_k, d_v, d_q, d_start, d_seq = views[i]
        if not first_use[i]:
            h2d_stream.wait_event(done[i])  # the step two back has read this record
        with torch.cuda.stream(h2d_stream):
            d_recs[i].copy_(h_rec[s], non_blocking=True)
        in_ready[i].record(h2d_stream)
        cs.wait_event(in_ready[i])
        if not first_use[i]:
            cs.wait_event(out_read[i])  # the output two steps back has been read
        with torch.cuda.stream(cs):
            tc.append(d_k, d_v, d_start)
            tc.decode(d_q, d_seq, max_len, out=d_outs[i], workspace=ws)
        done[i].record(cs)
        d2h_stream.wait_event(done[i])
        with torch.cuda.stream(d2h_stream):
            h_outs[i].copy_(d_outs[i], non_blocking=True)
        out_read[i].record(d2h_stream)
        first_use[i] = False

    for i in range(e2e_warm):
        e2e_step(s0 + i, stream)
    torch.cuda.synchronize()
    # the timed steps (uploads, kernels, downloads and the events that order them)
    # captured as one CUDA graph, the copy streams forked from and joined to the
    # capture; the replay is the timed region
    graph = torch.cuda.CUDAGraph()
    first_use[:] = [True, True]
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream()
        h2d_stream.wait_stream(cap)
        d2h_stream.wait_stream(cap)
        for i in range(e2e_steps):
            e2e_step(s0 + e2e_warm + i, cap)
        cap.wait_stream(h2d_stream)
        cap.wait_stream(d2h_stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # three replays (each rewrites the same tokens at the same positions and reads
    # the same lengths), each between two events; the median is reported, so that
    # one replay slowed by the host's side of the copies does not set the number
    e2e_runs = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()  # ends after the last output is on the host
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_runs.append(e0.elapsed_time(e1))
    del graph
    e2e_ms = max_over_ranks(float(np.median(e2e_runs)), world, dist, "cuda")
    e2e_bytes = sum(decode_bytes(lens0 + s0 + e2e_warm + i + 1) for i in range(e2e_steps))
    h2d = int(h_rec.shape[1])  # K, V, q, start positions and lengths of one step
    d2h = B * HQ * D * 4
    if tc.device_status() != 0:
        raise RuntimeError("device status set by the end-to-end steps")

    # the same step launched on the stream, one call after the other (no graph)
    sg0 = s0 + e2e_warm + e2e_steps
    step(sg0)
    stream_runs = []
    for _ in range(3):  # the same steps three times (same tokens, positions and lengths); the median
        se0, se1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        se0.record(stream)
        for i in range(graph_steps):
            step(sg0 + 1 + i)
        se1.record(stream)
        torch.cuda.synchronize()
        stream_runs.append(se0.elapsed_time(se1))
    stream_ms = max_over_ranks(float(np.median(stream_runs)), world, dist, "cuda")
    stream_bytes = sum(decode_bytes(lens0 + sg0 + 1 + i + 1) for i in range(graph_steps))
    if tc.device_status() != 0:
        raise RuntimeError("device status set by the stream-launched steps")

    # quantize throughput: batch 16 x 8192 new tokens x 8 KV heads at 3.5 bits (K3 / V4)
    del k_dev, v_dev
    kq, vq = quantize_inputs(torch)
    zero = torch.zeros(QB, dtype=torch.int32, device="cuda")
    quant = {}
    for name, kb, vb in (("3.5", KB, VB), ("3", 3, 3), ("4", 4, 4)):
        qc = TurboQuantKVCache(QB, HKV, HKV * 4, QT, bits=(kb, vb))
        quant[name] = time_quantize(torch, qc, kq, vq, zero, kb, vb)
        del qc
    del kq, vq
    # the other decode workloads: asym (fp16 K + 4-bit V, B8, context 16384) and the
    # 3.5-bit Llama-3-8B-like layer (B1, context 4096; launch- and L2-bound)
    asym_ms, asym_bytes = time_plain_decode(torch, 8, 16384, True)
    small_ms, small_bytes = time_plain_decode(torch, 1, 4096, False, reps=200)
    small_cold_ms, _ = time_plain_decode(torch, 1, 4096, False, reps=100, flush=True)
    i8_ms, i8_bytes, i8q_ms, i8q_bytes = time_int8(torch, lens0)

    peak, peak_kind = measured_peak()
    dec_avg_ms = float(np.mean(decode_ms))
    dec_bytes = float(np.mean([step_bytes[i] for i in sampled]))  # the bracketed calls
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = profile_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "mean_context": float(np.mean(lens0) + args.warmup + args.steps / 2),
            "l2": "inputs larger than L2: %.0f MB of packed cache read per step" % (dec_bytes / 1e6),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {"bound": "hbm", "kernel": "decode attention (split-K kernel + merge kernel, one call)",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": dec_bytes, "avg_launch_ms": dec_avg_ms},
        "quantize": dict(quant["3.5"], frac=quant["3.5"]["hbm_gbs"] / peak,
                         token="one (batch, position) with all 8 KV heads, K and V",
                         workload="batch 16 x 8192 new tokens x 8 KV heads, N(0,1) x lognormal(0,1) channel "
                                  "scales; 3.5 bits = K 3-bit / V 4-bit",
                         widths={w: dict(quant[w], frac=quant[w]["hbm_gbs"] / peak) for w in ("3", "4", "3.5")}),
        "sparse_v": {"threshold": 1e-3, "ms": sparse_ms, "dense_ms": dec_avg_ms,
                     "value": decode_bytes(lens0 + sv_s + 1) / (sparse_ms * 1e-3) / 1e9, "unit": "GB/s",
                     "note": "same long-context decode call with V skipped for weights below 1e-3 of the running "
                             "maximum (random synthetic codes: diffuse attention, few skips); back-to-back calls "
                             "replayed as one CUDA graph"},
        "paged": {"block_size": 64, "ms": paged_ms, "ms_blocks_in_order": paged_inorder_ms,
                  "value": decode_bytes(lens0 + sv_s + 1) / (paged_ms * 1e-3) / 1e9, "unit": "GB/s",
                  "note": "same long-context decode call on a block-table copy of the cache (64-token blocks, "
                          "permuted pool); back-to-back calls replayed as one CUDA graph"},
        "multi_query": {"n_query": mq_n, "ms": mq_ms, "value": mq_fma / (mq_ms * 1e-3) / 1e12, "unit": "T FMA/s",
                        "frac": mq_fma / (mq_ms * 1e-3) / FP32_FMA_PEAK, "bound": "alu",
                        "peak": FP32_FMA_PEAK / 1e12, "cache_gbs": decode_bytes(mq_lens) / (mq_ms * 1e-3) / 1e9,
                        "workload": "speculative verification: the 8 newest tokens of each long-context sequence, "
                                    "causal, B4, 32q/8kv, K3/V4 + 256 fp16 hot V; back-to-back calls replayed as "
                                    "one CUDA graph"},
        "asym": {"value": asym_bytes / (asym_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": asym_ms,
                 "frac": asym_bytes / (asym_ms * 1e-3) / 1e9 / peak, "algorithmic_bytes_per_launch": asym_bytes,
                 "workload": "asym decode: fp16 K + 4-bit V, B8, 32q/8kv, d128, context 16384, no hot window; "
                             "back-to-back calls replayed as one CUDA graph"},
        "int8": {"value": i8_bytes / (i8_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": i8_ms,
                 "frac": i8_bytes / (i8_ms * 1e-3) / 1e9 / peak, "algorithmic_bytes_per_launch": i8_bytes,
                 "workload": "int8-mode decode (per-token INT8 absmax K and V, no hot window): B4, 32q/8kv, "
                             "d128, the long-context lengths; back-to-back calls replayed as one CUDA graph",
                 "quantize_mtokens_s": QB * QT / (i8q_ms * 1e-3) / 1e6, "quantize_ms": i8q_ms,
                 "quantize_hbm_gbs": i8q_bytes / (i8q_ms * 1e-3) / 1e9},
        "llama_layer": {"value": small_bytes / (small_cold_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": small_cold_ms,
                        "ms_l2_resident": small_ms, "algorithmic_bytes_per_launch": small_bytes,
                        "workload": "3.5-bit decode: B1, 32q/8kv, d128, context 4096, K3/V4; ms after a 256 MB "
                                    "write flushed L2 before each call (ms_l2_resident: back-to-back calls "
                                    "replayed as one CUDA graph, the 4 MB cache stays in L2)"},
        "e2e": {"value": job_throughput(e2e_bytes, e2e_ms, world), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "replay_ms": [round(x, 4) for x in e2e_runs], "of_replays": "median",
                "copies": "pinned host record uploaded and output downloaded every step on two copy streams "
                          "into double buffers, overlapping the previous and next step's kernels; the steps "
                          "captured as one CUDA graph with the copies and replayed"},
        "launch": "the timed steps captured as one CUDA graph (each step's kernels in order) and replayed once",
        "stream_launched": {"value": job_throughput(stream_bytes, stream_ms, world), "unit": "GB/s",
                            "ms_per_step": stream_ms / graph_steps, "steps": graph_steps,
                            "run_ms": [round(x, 4) for x in stream_runs], "of_runs": "median",
                            "note": "the same step launched call by call on the stream instead of replayed as a "
                                    "CUDA graph"},
        "clocks": clocks,
        # per timed step: the one-token append (evict fused), the split-K kernel and the merge
        "gpu_launches": args.steps * 3,
    }
    if want_cpu:
        line["cpu_baseline"] = cpu_baseline(lens0, synth.queries_fp16(SEED, B, HQ, D), pool, workers)
        pool.shutdown()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile(args):
    """Only the decode step or only the quantize append, at the bench shapes
    (quantize batch reduced to --profile-batch), for profiler captures."""
    import torch
    from bit_kv_cache_10_gb300 import build as tq_build
    from bit_kv_cache_10_gb300.cache import TurboQuantKVCache
    tq_build.build()
    total = args.warmup + args.steps
    if args.profile == "decode":
        tc, lens0 = build_decode_cache(torch, HI + total + 64)
        kn, vn, qn = step_inputs(total)
        k_dev, v_dev, q_dev = (torch.from_numpy(a).cuda() for a in (kn, vn, qn))
        starts = torch.from_numpy((lens0[None, :] + np.arange(total)[:, None]).astype(np.int32)).cuda()
        seqs = starts + 1
        max_len = HI + total
        out = torch.empty(B, HQ, D, dtype=torch.float32, device="cuda")
        ws = torch.empty(tc.workspace_bytes(max_len), dtype=torch.uint8, device="cuda")
        t0 = None
        for s in range(total):
            if s == args.warmup:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            tc.append(k_dev[s], v_dev[s], starts[s])
            tc.decode(q_dev[s], seqs[s], max_len, out=out, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "decode", "steps": args.steps, "wall_ms_per_step":
                          (time.perf_counter() - t0) * 1e3 / max(1, args.steps), "status": tc.device_status()}))
    elif args.profile == "paged":
        tc, lens0 = build_decode_cache(torch, HI + 64)
        pg = paged_copy(torch, tc)
        del tc
        q = torch.from_numpy(synth.queries_fp16(SEED, B, HQ, D)).cuda()
        sl = torch.from_numpy(np.asarray(lens0, np.int32)).cuda()
        out = torch.empty(B, HQ, D, dtype=torch.float32, device="cuda")
        ws = torch.empty(pg.workspace_bytes(HI), dtype=torch.uint8, device="cuda")
        for s in range(total):
            pg.decode(q, sl, HI, out=out, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "paged", "steps": total, "status": pg.device_status()}))
    elif args.profile == "int8":
        lens = synth.seq_lengths(SEED, B, LO, HI)
        cap = int(np.max(lens))
        tc = build_int8_cache(torch, lens, cap)
        q = torch.from_numpy(synth.queries_fp16(SEED + 7, B, HQ, D)).cuda()
        sl = torch.from_numpy(np.asarray(lens, np.int32)).cuda()
        out = torch.empty(B, HQ, D, dtype=torch.float32, device="cuda")
        ws = torch.empty(tc.workspace_bytes(cap), dtype=torch.uint8, device="cuda")
        for s in range(total):
            tc.decode(q, sl, cap, out=out, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "int8", "steps": total, "status": tc.device_status()}))
    elif args.profile == "llama":
        tc = build_plain_cache(torch, 1, 4096, False, SEED + 3)
        q = torch.from_numpy(synth.queries_fp16(SEED + 3, 1, HQ, D)).cuda()
        lens = torch.full((1,), 4096, dtype=torch.int32, device="cuda")
        out = torch.empty(1, HQ, D, dtype=torch.float32, device="cuda")
        ws = torch.empty(tc.workspace_bytes(4096), dtype=torch.uint8, device="cuda")
        for s in range(total):
            tc.decode(q, lens, 4096, out=out, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "llama", "steps": total, "status": tc.device_status()}))
    elif args.profile == "asym":
        tc = build_plain_cache(torch, 8, 16384, True, SEED + 3)
        q = torch.from_numpy(synth.queries_fp16(SEED + 3, 8, HQ, D)).cuda()
        lens = torch.full((8,), 16384, dtype=torch.int32, device="cuda")
        out = torch.empty(8, HQ, D, dtype=torch.float32, device="cuda")
        ws = torch.empty(tc.workspace_bytes(16384), dtype=torch.uint8, device="cuda")
        for s in range(total):
            tc.decode(q, lens, 16384, out=out, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "asym", "steps": total, "status": tc.device_status()}))
    else:
        qb = args.profile_batch
        g = synth.rng(SEED + 2, synth.STREAM_K)
        kq = torch.from_numpy(g.standard_normal((qb, HKV, QT, D), dtype=np.float32).astype(np.float16)).cuda()
        vq = torch.from_numpy(g.standard_normal((qb, HKV, QT, D), dtype=np.float32).astype(np.float16)).cuda()
        qc = TurboQuantKVCache(qb, HKV, HKV * 4, QT, bits=(KB, VB))
        zero = torch.zeros(qb, dtype=torch.int32, device="cuda")
        for s in range(total):
            qc.append(kq, vq, zero)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "quantize", "batch": qb, "steps": total, "status": qc.device_status()}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle timing")
    ap.add_argument("--profile", choices=["decode", "quantize", "asym", "int8", "paged", "llama"],
                    help="run only warm-up + timed steps of one part (for ncu captures); prints a short line")
    ap.add_argument("--profile-batch", type=int, default=4, help="batch of the quantize part in --profile mode")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
