#!/usr/bin/env python
"""Throughput bench of the quantized lightning indexer on one or more GB300s.

A step is one full indexer call (plan, score, select) over one batch of the
chosen workload, with every input resident in HBM. The metric is scored
(query, position) pairs per second. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Multi-GPU (torchrun, one process per GPU): independent replicas, no data
exchange; the per-rank times are reduced with a max and the pairs summed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_indexer_qli_gb300 import synth  # noqa: E402

METRIC = "QLI scored (query,position) pairs/s; % of HBM (decode) / INT8 (prefill) roof"
UNIT = "pairs/s"
L2_BYTES = 129 * 1024 * 1024
# input sets cycled so that a step never finds its index K in L2 (the
# prefill workload's K is 8.4 MB per set: 16 sets exceed the 129 MB L2)
ROTATE_SETS = {1: 1, 2: 3, 3: 16, 4: 8, 5: 1}
SCORE_SRC = os.path.join(ROOT, "sparse_attention_indexer_qli_gb300", "csrc", "qli_score.cu")
PREFILL_SRC = os.path.join(ROOT, "sparse_attention_indexer_qli_gb300", "csrc", "qli_prefill.cu")
ATTN_SRC = os.path.join(ROOT, "sparse_attention_indexer_qli_gb300", "csrc", "qli_attn.cu")
SMALL_SRC = os.path.join(ROOT, "sparse_attention_indexer_qli_gb300", "csrc", "qli_small.cu")
QUANT_SRC = os.path.join(ROOT, "sparse_attention_indexer_qli_gb300", "csrc", "qli_quant.cu")
# workload -> (committed ncu summary, the kernel source it was taken on)
PROFILES = {
    # one token: the single-launch path (its kernel also selects)
    1: ("small_kernel_decode_b1_ratio2.md", SMALL_SRC, "small_source_sha256"),
    2: ("stream_kernel_decode_b64_ratio1.md", SCORE_SRC, "stream_source_sha256"),
    3: ("prefill_kernel_prefill_t4096_2x2048.md", PREFILL_SRC, "prefill_source_sha256"),
    4: ("stream_kernel_consumer_b32_ratio2.md", SCORE_SRC, "stream_source_sha256"),
    # captured on 2 of the 8 1M-context requests and scaled by scored pairs
    5: ("stream_kernel_longctx_2of8x1M.md", SCORE_SRC, "stream_source_sha256"),
    "attn": ("attn_kernel_decode_b64_h64_topk2048.md", ATTN_SRC, "attn_source_sha256"),
    "quantize_q": ("quant_kernel_queries_t4096_n64.md", QUANT_SRC, "quant_source_sha256"),
    "write_index_k": ("quant_kernel_index_k_2x32768.md", QUANT_SRC, "quant_source_sha256"),
}


# ---------------------------------------------------------------- accounting

def visible(case, t, b):
    """Visible compressed positions of token t (bench accounting only)."""
    c0, c1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
    lk = int(case.k_lens[b])
    res = 0 if case.residual is None else int(case.residual[b])
    seen = lk * case.ratio + res - (c1 - c0) + (t - c0) + 1
    return 0 if seen <= 0 else min(lk, seen // case.ratio)


def pairs_of(case) -> int:
    """Scored pairs of one step: sum over tokens of the eligible positions."""
    total = 0
    for b in range(case.B):
        for t in range(int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])):
            V = visible(case, t, b)
            if case.cand_mode == "consumer":
                nb = (V + 7) // 8
                ids = np.unique(case.cand_in[t, 0])
                ids = ids[(ids >= 0) & (ids < nb)]
                total += int(np.minimum(8, V - 8 * ids).sum())
            else:
                total += V
    return total


def score_algorithmic_bytes(case, pairs: int) -> int:
    """Bytes the score kernel must move per launch: 130 B per pair (INT8 K row
    + FP16 K scale), each query's N*128 INT8 Q bytes and 4N bytes of FP16
    weights and scales, and one 4-byte block-table entry per page touched."""
    pages = sum(case.request_pages(b) for b in range(case.B))
    return 130 * pairs + case.T * case.N * (128 + 4) + 4 * pages


def step_bytes_in(case) -> int:
    n = case.q.nbytes + case.cu_seqlens_q.nbytes + case.k_lens.nbytes + case.block_table.nbytes
    n += case.head_weights.nbytes + case.q_scale.nbytes
    n += 0 if case.residual is None else case.residual.nbytes
    n += 0 if case.cand_in is None else case.cand_in.nbytes
    return int(n)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def roofline(idx, sets, args, score_ms_avg):
    """Roofline of the score stage, the step's dominant kernel: HBM-bound for
    the decode workloads (algorithmic bytes), tensor-bound for prefill
    (2*128*N flops per scored pair; FP16 operands, the measured BF16 dense
    peak being the same nominal rate)."""
    nsets = len(sets)
    chosen = [sets[(args.warmup + k) % nsets] for k in range(args.steps)]
    if idx == 3:
        flops = sum(2 * 128 * c.N * p for c, _, p in chosen) / len(chosen)
        achieved = flops / (score_ms_avg / 1e3) / 1e12
        peak, kind = tensor_peak()
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profiled_traffic(idx), "kernel": "prefill_kernel",
                "peak_source": kind, "kernel_ms": score_ms_avg, "algorithmic_flops": flops}
    alg = sum(score_algorithmic_bytes(c, p) for c, _, p in chosen) / len(chosen)
    achieved = alg / (score_ms_avg / 1e3) / 1e9
    peak, kind = peaks()
    # the workload-5 summary gives the whole workload's traffic; a cut has none
    traffic = profiled_traffic(idx) if idx != 5 or args.long_requests >= 8 else None
    # a small batch runs the single-launch kernel, whose score stage also selects
    small = sets[0][1].launches(3) == 0
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic,
            "kernel": "small_kernel" if small else "stream_kernel",
            "peak_source": kind, "kernel_ms": score_ms_avg, "algorithmic_bytes": alg}


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (bf16 burst; fp16 same nominal rate)"
    return 1900.0, "fallback"


def profiled_traffic(idx):
    """Per-launch DRAM traffic of the workload's score kernel from its
    committed ncu summary, if there is one for this workload and it was taken
    on the current kernel source; else None."""
    if idx not in PROFILES:
        return None
    name, src, key = PROFILES[idx]
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", txt)
    h = re.search(key + r":\s*([0-9a-f]{64})", txt)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return int(m.group(1)) if h.group(1) == cur else None


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return ws, rank, local


def _reduce(x: float, ws: int, op: str, device: str) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def reduce_max(x: float, ws: int, device: str = "cuda") -> float:
    """Slowest rank's time: replicas are timed together, the job ends with the last."""
    return _reduce(x, ws, "max", device)


def reduce_sum(x: float, ws: int, device: str = "cuda") -> float:
    """Pairs scored by all replicas."""
    return _reduce(x, ws, "sum", device)


def aggregate(ms: float, pairs: float, ws: int, device: str = "cuda"):
    """Whole-job throughput of N independent replicas: all ranks' pairs over
    the slowest rank's time (weak scaling, no data exchange)."""
    ms_max = reduce_max(ms, ws, device)
    total = reduce_sum(pairs, ws, device)
    return total / (ms_max / 1e3), ms_max, total


def repeats_for(first_ms: float, min_seconds: float, ws: int, cap: int = 500) -> int:
    """How many times to run the K-step timed region so that about
    `min_seconds` of GPU time pass in total (the same count on every rank)."""
    want = 1 if first_ms <= 0 else int(np.ceil(1e3 * min_seconds / first_ms))
    want = max(1, min(cap, want))
    return int(reduce_max(float(want), ws))


def barrier(ws: int):
    import torch
    torch.cuda.synchronize()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


# ---------------------------------------------------------------- CPU oracle

def oracle_rate(case, budget_s: float, rows_per_chunk: int):
    """Times the oracle, as it stands, on successive row chunks of the
    workload until `budget_s` of work is done; returns (pairs/s, rows, cores)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    prep = oracle.prepare(case)
    order = np.random.default_rng(12345).permutation(case.T)
    done_pairs, done_rows, spent = 0, 0, 0.0
    i = 0
    while spent < budget_s and i < case.T:
        rows = order[i:i + rows_per_chunk]
        i += rows.size
        t0 = time.perf_counter()
        out = oracle.run(prep, rows=rows, nthreads=cores)
        spent += time.perf_counter() - t0
        done_rows += rows.size
        if case.cand_mode == "consumer":
            sub = 0
            for r, t in enumerate(rows):
                V = int(out["visible"][r])
                nb = (V + 7) // 8
                ids = np.unique(case.cand_in[t, 0])
                ids = ids[(ids >= 0) & (ids < nb)]
                sub += int(np.minimum(8, V - 8 * ids).sum())
            done_pairs += sub
        else:
            done_pairs += int(out["visible"].sum())
    return done_pairs / spent, done_rows, cores, spent


# ---------------------------------------------------------------- arms

def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case = synth.config(args.config)
    import oracle
    cores = len(os.sched_getaffinity(0))
    prep = oracle.prepare(case)
    per_step = max(1, min(case.T, args.ref_rows))
    order = np.random.default_rng(777).permutation(case.T)

    def step(k):
        lo = (k * per_step) % case.T
        rows = np.take(order, np.arange(lo, lo + per_step), mode="wrap")
        out = oracle.run(prep, rows=rows, nthreads=cores)
        return int(out["visible"].sum()) if case.cand_mode != "consumer" else None

    for k in range(args.warmup):
        step(k)
    pairs = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        p = step(args.warmup + k)
        pairs += p if p is not None else 0
    dt = time.perf_counter() - t0
    if case.cand_mode == "consumer":
        pairs = int(round(pairs_of(case) * per_step / case.T)) * args.steps
    value = pairs / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic",
        "config": {"workload": synth.CONFIG_NAMES[args.config],
                   "reference": "CPU oracle (plain C, OpenMP over positions), no GPU"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d query rows per step of the workload, cycled" % per_step},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_ours(args):
    import torch

    from sparse_attention_indexer_qli_gb300 import qli

    world, rank, local = dist_setup()
    qli.lib()
    idx = args.config
    nsets = args.sets or ROTATE_SETS[idx]
    base_seed = idx - 1
    sets = []
    for s in range(nsets):
        case = synth.config(idx, seed=base_seed + 1000 * s + 100 * rank,
                            long_requests=args.long_requests)
        kw = synth.upload(case, "cuda")
        call = qli.Call(**kw)
        sets.append((case, call, pairs_of(case)))
    ws_bytes = max(c.workspace_bytes() for _, c, _ in sets)
    workspace = torch.empty(max(256, ws_bytes), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    launches_per_step = sets[0][1].launches(0)

    # One CUDA graph per input set holding the whole call (its kernels keep
    # their programmatic launch edges), so that the timed loop measures the
    # device work and not the host's argument marshalling. A second set of
    # graphs, one per stage, is replayed with events between the stages (on
    # the stream they run on) to time the score kernel alone for the roofline.
    for _, call, _ in sets:                  # first calls outside capture
        call.run(workspace, stream)
    torch.cuda.synchronize()
    whole, staged = [], []
    for _, call, _ in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            call.run(workspace)
        whole.append(g)
        gs = []
        for stage in (qli.STAGE_PLAN, qli.STAGE_SCORE, qli.STAGE_SELECT):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                call.run_stage(stage, workspace)
            gs.append(g)
        staged.append(gs)
    torch.cuda.synchronize()

    def staged_step(k, ev):
        gs = staged[k % nsets]
        ev[0].record(stream)
        gs[0].replay()
        ev[1].record(stream)
        gs[1].replay()
        ev[2].record(stream)
        gs[2].replay()
        ev[3].record(stream)

    for k in range(args.warmup):
        whole[k % nsets].replay()
    # timed region: K whole-call steps, bracketed by a barrier and a
    # synchronize; the region is repeated (K steps each time) until about
    # `--min-seconds` of GPU time has run, so that the clock sampler sees the
    # GPU under load, and the median repeat is reported
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kbytes = 130 * int(sets[0][0].k_lens.sum())
    flush = None
    if nsets * kbytes <= L2_BYTES:
        # the input sets fit in L2 together: every step is timed on its own
        # (events around it) after a 256 MB read that evicts the previous
        # steps' data, outside the events
        flush = torch.ones(256 << 20, dtype=torch.uint8, device="cuda")
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]

    def timed_region():
        barrier(world)
        if flush is not None:
            for k in range(args.steps):
                flush.max()              # a read: evicts L2 and leaves no dirty lines behind
                step_ev[k][0].record(stream)
                whole[(args.warmup + k) % nsets].replay()
                step_ev[k][1].record(stream)
            torch.cuda.synchronize()
            barrier(world)
            return sum(a.elapsed_time(b) for a, b in step_ev)
        start.record(stream)
        for k in range(args.steps):
            whole[(args.warmup + k) % nsets].replay()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(stop)

    with ClockSampler(torch.cuda.current_device()) as clk:
        region_ms = [timed_region()]
        repeats = repeats_for(region_ms[0], args.min_seconds, world)
        for _ in range(repeats - 1):
            region_ms.append(timed_region())
    ms = statistics.median(region_ms)
    my_pairs = sum(sets[(args.warmup + k) % nsets][2] for k in range(args.steps))
    value, ms_max, all_pairs = aggregate(ms, my_pairs, world)

    # the score kernel's own duration: K staged steps, events between stages
    for k in range(args.warmup):
        staged_step(k, [torch.cuda.Event(enable_timing=True) for _ in range(4)])
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for k in range(args.steps):
        staged_step(args.warmup + k, evs[k])
    torch.cuda.synchronize()
    score_ms = [e[1].elapsed_time(e[2]) for e in evs]
    score_ms_avg = sum(score_ms) / len(score_ms)
    roof = roofline(idx, sets, args, score_ms_avg)
    # an on-chip wait that gave up (200 ms) sets the device error word; any
    # other disturbance (a profiler serialising the kernels, a neighbour on
    # the GPU) shows as steps far slower than their stages timed one by one
    staged_ms = sum(e[0].elapsed_time(e[3]) for e in evs) / len(evs)
    stage_ms = {"plan": sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs),
                "score": score_ms_avg,
                "select": sum(e[2].elapsed_time(e[3]) for e in evs) / len(evs)}
    err = sets[0][1].device_error(workspace)
    if err != 0:
        sys.stderr.write("device error word %d after the timed region: not a valid run\n" % err)
        sys.exit(3)
    if ms / args.steps > 3 * staged_ms:
        sys.stderr.write("warning: %.3f ms per step against %.3f ms for the stages timed one by "
                         "one: the timed region was disturbed\n" % (ms / args.steps, staged_ms))

    # e2e: the public call from pinned host buffers, copies inside the timed region
    e2e = run_e2e(args, sets, workspace, stream, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows, cores, spent = oracle_rate(sets[0][0], args.cpu_seconds, args.cpu_rows)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d of %d query rows of the workload (%.1f s of oracle time)"
                         % (rows, sets[0][0].T, spent)}
    if rank != 0:
        return
    case0 = sets[0][0]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {
            "workload": synth.CONFIG_NAMES[idx] + (
                "" if idx != 5 or args.long_requests >= 8
                else " (cut: %d of the 8 1M-context requests)" % args.long_requests),
            "global_batch": case0.B * world,
            "query_tokens": case0.T, "heads": case0.N, "ratio": case0.ratio,
            "topk": case0.topk, "cand_mode": case0.cand_mode,
            "pairs_per_step": my_pairs / args.steps,
            "l2": ("inputs larger than L2: the steps rotate over %d independent input sets, "
                   "%.1f MB of index K (rows and scales) each, %.0f MB in all (L2 129 MB)"
                   % (nsets, kbytes / 1e6, nsets * kbytes / 1e6)) if flush is None else
                  ("L2 flushed between steps: a 256 MB read before each step, outside the "
                   "events that time the step (%.2f MB of index K per step)" % (kbytes / 1e6)),
            "parallelism": "replicas" if world > 1 else "single",
            "launch": "one CUDA graph per input set holding the whole call",
            "timing": "median of %d repeats of the %d-step timed region (%.0f ms of steps in all)"
                      % (len(region_ms), args.steps, sum(region_ms)),
        },
        "repeats": len(region_ms),
        "roofline": roof,
        "stage_ms": stage_ms,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line))


def _packed(tensors, device=None):
    """One buffer holding the given tensors at 256-byte aligned offsets:
    pinned host memory (device None) or device memory. Returns the buffer and
    the tensors as views into it."""
    import torch
    offs, off = [], 0
    for t in tensors:
        if t is None:
            offs.append(None)
            continue
        off = (off + 255) & ~255
        offs.append(off)
        off += t.numel() * t.element_size()
    buf = (torch.empty(max(off, 1), dtype=torch.uint8, pin_memory=True) if device is None
           else torch.empty(max(off, 1), dtype=torch.uint8, device=device))
    views = []
    for t, o in zip(tensors, offs):
        if t is None:
            views.append(None)
            continue
        n = t.numel() * t.element_size()
        views.append(buf[o:o + n].view(t.dtype).view(t.shape))
    return buf, views


def run_e2e(args, sets, workspace, stream, world):
    """The public call from host buffers: each step copies its inputs from
    one pinned host buffer to one device buffer (the call's inputs are views
    into it), runs the call, and copies its outputs (one device buffer) back
    to pinned host memory, all inside the timed region.

    Two loops are timed. In order: the copies and the call of each step one
    after another on one stream. Pipelined, as a serving loop would run:
    the inputs of step k+1 go up on one copy stream and the outputs of step
    k come down on another while the calls run in order on the compute
    stream; steps use the input sets in turn, each with its own host and
    device buffers, and events keep every buffer from being reused while a
    copy or call still needs it. `value` is the faster of the two (named in
    `mode`; short steps lose more to the streams' event waits than the
    overlap gains), and both are reported."""
    import torch

    from sparse_attention_indexer_qli_gb300 import qli
    nsets = len(sets)
    hbufs, dbufs, obufs, ohost, calls = [], [], [], [], []
    for case, call, _ in sets:
        ins = list(call.keep[:4]) + list(call.keep[5:9])   # everything but the page pool
        hb, hviews = _packed([None if t is None else t.cpu() for t in ins])
        for hv, t in zip(hviews, ins):
            if t is not None:
                hv.copy_(t.cpu())
        db, dv = _packed(ins, device="cuda")
        q, cu, kl, res, bt, hw, qs, cin = dv
        ob, (idx_o, cand_o) = _packed([call.indices, call.cand], device="cuda")
        c = qli.Call(q, cu, kl, res, call.keep[4], bt, hw, qs, ratio=case.ratio,
                     rows_per_page=case.rows_per_page, page_stride=case.page_stride,
                     k_offset=case.k_offset, scale_offset=case.scale_offset, topk=case.topk,
                     cand_mode=case.cand_mode, cand_blocks=case.cand_blocks, cand_in=cin,
                     indices_out=idx_o, cand_out=cand_o)
        hbufs.append(hb)
        dbufs.append(db)
        obufs.append(ob)
        ohost.append(torch.empty(ob.shape, dtype=torch.uint8, pin_memory=True))
        calls.append(c)

    def serial_step(k):
        i = k % nsets
        dbufs[i].copy_(hbufs[i], non_blocking=True)
        calls[i].run(workspace, stream)
        ohost[i].copy_(obufs[i], non_blocking=True)

    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nsets)]     # inputs of set i on the device
    ev_run = [torch.cuda.Event() for _ in range(nsets)]    # call on set i finished
    ev_out = [torch.cuda.Event() for _ in range(nsets)]    # outputs of set i on the host

    def piped_step(k):
        i = k % nsets
        up.wait_event(ev_run[i])               # the last call on set i has read its inputs
        with torch.cuda.stream(up):
            dbufs[i].copy_(hbufs[i], non_blocking=True)
        ev_in[i].record(up)
        stream.wait_event(ev_in[i])
        stream.wait_event(ev_out[i])           # the last copy of set i's outputs is done
        calls[i].run(workspace, stream)
        ev_run[i].record(stream)
        down.wait_event(ev_run[i])
        with torch.cuda.stream(down):
            ohost[i].copy_(obufs[i], non_blocking=True)
        ev_out[i].record(down)

    def timed(step):
        for e in ev_run + ev_out:
            e.record(stream)
        for k in range(args.warmup):
            step(k)
        torch.cuda.synchronize()
        barrier(world)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        up.wait_event(t0)
        down.wait_event(t0)
        for k in range(args.steps):
            step(args.warmup + k)
        stream.wait_stream(up)
        stream.wait_stream(down)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return reduce_max(t0.elapsed_time(t1), world)

    with torch.cuda.stream(stream):
        ms_serial = timed(serial_step)
        ms = timed(piped_step)
    pairs = reduce_sum(sum(sets[(args.warmup + k) % nsets][2] for k in range(args.steps)), world)
    h2d = sum(hbufs[(args.warmup + k) % nsets].numel() for k in range(args.steps))
    d2h = sum(ohost[(args.warmup + k) % nsets].numel() for k in range(args.steps))
    piped, serial = pairs / (ms / 1e3), pairs / (ms_serial / 1e3)
    return {"value": max(piped, serial), "unit": UNIT,
            "h2d_bytes_per_step": h2d // args.steps, "d2h_bytes_per_step": d2h // args.steps,
            "mode": "pipelined" if piped >= serial else "in-order",
            "pipelined_value": piped, "serial_value": serial}


# ------------------------------------------------ query quantiser / K writer

OP_ROWS = {"quantize_q": 4096 * 64, "write_index_k": 2 * 32768}


def op_inputs(op: str, seed: int, case=None):
    """Host inputs of one step of the quantiser / writer workloads: the
    prefill workload's 4096 query tokens x 64 heads, or the index-K rows of
    its two 65536-token requests (ratio 2, 32768 compressed rows each) with
    their slots under `case`'s block table."""
    if op == "quantize_q":
        return {"x": synth.bf16_rows(seed, (4096, 64, 128), sigma=1.0)}
    slots = np.concatenate([synth.slots_of(case, b, np.arange(int(case.k_lens[b])))
                            for b in range(case.B)])
    return {"x": synth.bf16_rows(seed, (slots.size, 128), sigma=2.0), "slots": slots,
            "case": case}


def op_bytes(op: str, rows: int) -> int:
    """Algorithmic bytes: 256 B of BF16 read and 128 + 2 B written per row,
    plus the 8-byte slot of each written index-K row."""
    return rows * (256 + 130 + (8 if op == "write_index_k" else 0))


def run_op(args):
    import torch

    from sparse_attention_indexer_qli_gb300 import qli
    world, rank, local = dist_setup()
    qli.lib()
    op = args.op
    nsets = 3
    pool_case = (synth.make_case(100 * rank + 7, [65536, 65536], [1, 1], N=64, ratio=2, topk=2048)
                 if op == "write_index_k" else None)
    host = [op_inputs(op, 1000 * s + 100 * rank + 7, pool_case) for s in range(nsets)]
    rows = OP_ROWS[op]
    dev_x = [torch.from_numpy(h["x"].view(np.int16)).cuda() for h in host]
    if op == "quantize_q":
        q = torch.empty((4096, 64, 128), dtype=torch.int8, device="cuda")
        sc = torch.empty((4096, 64), dtype=torch.int16, device="cuda")

        def launch(i):
            qli.quantize_q(dev_x[i], q, sc)
        outs = [q, sc]
        workload = "prefill-queries-t4096-n64-d128-bf16"
    else:
        case = host[0]["case"]
        pool = torch.zeros((case.num_pages, case.page_stride), dtype=torch.uint8, device="cuda")
        dev_slots = [torch.from_numpy(h["slots"]).cuda() for h in host]
        err = torch.zeros(1, dtype=torch.int32, device="cuda")

        def launch(i):
            qli.write_index_k(dev_x[i], dev_slots[i], pool, rows_per_page=case.rows_per_page,
                              page_stride=case.page_stride, k_offset=case.k_offset,
                              scale_offset=case.scale_offset, err_word=err)
        outs = []
        workload = "prefill-index-k-2x32768-rows-r2-pages64"
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda").fill_(1)
    for k in range(args.warmup):
        launch(k % nsets)
    torch.cuda.synchronize()
    # one graph per input set, so the timed launch does not wait on the host
    graphs = []
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        for i in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                launch(i)
            graphs.append(g)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    with ClockSampler(torch.cuda.current_device()) as clk:
        for k in range(args.steps):
            flush.max()                      # evict the previous step's data from L2 (reads only)
            evs[k][0].record(stream)
            graphs[(args.warmup + k) % nsets].replay()
            evs[k][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = sum(a.elapsed_time(b) for a, b in evs)
    ms_max = reduce_max(ms, world)
    value = reduce_sum(rows * args.steps, world) / (ms_max / 1e3)
    per_ms = ms / args.steps
    achieved = op_bytes(op, rows) / (per_ms / 1e3) / 1e9
    peak, kind = peaks()
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": profiled_traffic(op), "kernel": "quant_kernel",
            "peak_source": kind, "kernel_ms": per_ms, "algorithmic_bytes": op_bytes(op, rows)}

    # e2e: inputs from pinned host memory, outputs (codes and scales) back
    pin = [torch.from_numpy(h["x"].view(np.int16)).pin_memory() for h in host]
    pin_slots = ([torch.from_numpy(h["slots"]).pin_memory() for h in host]
                 if op == "write_index_k" else None)
    out_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    if op == "write_index_k":
        out_h = [torch.empty(1, dtype=torch.int32, pin_memory=True)]
        outs = [err]

    def e2e_step(k):
        i = k % nsets
        dev_x[i].copy_(pin[i], non_blocking=True)
        if pin_slots is not None:
            dev_slots[i].copy_(pin_slots[i], non_blocking=True)
        launch(i)
        for h, o in zip(out_h, outs):
            h.copy_(o, non_blocking=True)
    for k in range(args.warmup):
        e2e_step(k)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        e2e_step(args.warmup + k)
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(t0.elapsed_time(t1), world)
    h2d = pin[0].numel() * 2 + (pin_slots[0].numel() * 8 if pin_slots is not None else 0)
    d2h = sum(h.numel() * h.element_size() for h in out_h)
    e2e = {"value": reduce_sum(rows * args.steps, world) / (e2e_ms / 1e3), "unit": "rows/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = 16384
        xs = host[0]["x"].reshape(-1, 128)[:n]
        t_0 = time.perf_counter()
        if op == "quantize_q":
            oracle.quantize_rows(xs)
        else:
            c = host[0]["case"]
            pages = np.zeros((c.num_pages, c.page_stride), dtype=np.uint8)
            oracle.write_index_k(xs, host[0]["slots"][:n], pages, c.rows_per_page, c.k_offset,
                                 c.scale_offset)
        spent = time.perf_counter() - t_0
        cpu = {"value": n / spent, "unit": "rows/s", "cores": 1, "kind": "oracle",
               "sample": "%d of %d rows of the workload (%.3f s)" % (n, rows, spent)}
    if rank != 0:
        return
    line = {
        "metric": "%s rows/s (%% of HBM roof)" % op, "value": value, "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16->int8", "data": "synthetic",
        "config": {"workload": workload, "rows_per_step": rows,
                   "l2": "a 256 MB read between steps evicts the previous step (outside the events)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line))


# ------------------------------------------------- attention over the indices

ATTN_SCALE = 1.0 / np.sqrt(512.0)


def attn_algorithmic_bytes(case) -> int:
    """Bytes the attention kernel must move: each listed position's KV row
    (1024 B) once per token, the token's queries and outputs (H x 512 BF16
    each), its LSE (4 B per head), its index list (4 B per entry) and one
    4-byte block-table entry per listed position."""
    listed = int((case.attn_indices >= 0).sum())
    T, H = case.q_attn.shape[:2]
    return 1024 * listed + 2 * (T * H * 512 * 2) + 4 * T * H + 4 * case.attn_indices.size + 4 * listed


def run_attn(args):
    import torch

    from sparse_attention_indexer_qli_gb300 import qli
    world, rank, local = dist_setup()
    qli.lib()
    case = synth.attention_workload(seed=21 + 100 * rank)
    dev = "cuda"
    cache = case.pack_pages_torch(dev)
    q = torch.from_numpy(case.q_attn.view(np.int16)).to(dev).view(torch.bfloat16)
    cu = torch.from_numpy(case.cu_seqlens_q).to(dev)
    bt = torch.from_numpy(case.block_table).to(dev)
    idx = torch.from_numpy(case.attn_indices).to(dev)
    T, H = q.shape[:2]
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    pairs = int((case.attn_indices >= 0).sum())

    def launch():
        qli.sparse_attention(q, cu, cache, bt, idx, rows_per_page=case.rows_per_page,
                             page_stride=case.page_stride, scale=ATTN_SCALE, out=out, lse=lse,
                             err_word=err)
    # one step reads 134 MB of KV rows, about the size of L2: every step is
    # timed on its own after a 256 MB read that evicts the previous one (a
    # read leaves no dirty lines whose write-back the step would pay for)
    flush = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]

    def region():
        barrier(world)
        for k in range(args.steps):
            flush.max()
            evs[k][0].record(stream)
            g.replay()
            evs[k][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return sum(a.elapsed_time(b) for a, b in evs)

    with ClockSampler(torch.cuda.current_device()) as clk:
        times = [region()]
        for _ in range(repeats_for(times[0], args.min_seconds, world) - 1):
            times.append(region())
    ms = statistics.median(times)
    value, ms_max, _ = aggregate(ms, pairs * args.steps, world)
    if int(err.item()) != 0:
        sys.stderr.write("device error word %d: not a valid run\n" % int(err.item()))
        sys.exit(3)
    per_ms = ms / args.steps
    alg = attn_algorithmic_bytes(case)
    peak, kind = peaks()
    roof = {"bound": "hbm", "achieved": alg / (per_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
            "frac": alg / (per_ms / 1e3) / 1e9 / peak, "traffic": profiled_traffic("attn"),
            "kernel": "attn_kernel", "peak_source": kind, "kernel_ms": per_ms,
            "algorithmic_bytes": alg}
    # e2e: the public call from pinned host buffers, outputs back to the host
    h_q = torch.from_numpy(case.q_attn.view(np.int16)).pin_memory()
    h_idx = torch.from_numpy(case.attn_indices).pin_memory()
    h_out = torch.empty((T, H, 512), dtype=torch.bfloat16, pin_memory=True)
    h_lse = torch.empty((T, H), dtype=torch.float32, pin_memory=True)
    qv = q.view(torch.int16)

    def e2e_step():
        qv.copy_(h_q, non_blocking=True)
        idx.copy_(h_idx, non_blocking=True)
        launch()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)
    for _ in range(args.warmup):
        e2e_step()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    t0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(t0.elapsed_time(t1), world)
    e2e = {"value": reduce_sum(pairs * args.steps, world) / (e2e_ms / 1e3), "unit": "pairs/s",
           "h2d_bytes_per_step": h_q.numel() * 2 + h_idx.numel() * 4,
           "d2h_bytes_per_step": h_out.numel() * 2 + h_lse.numel() * 4}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import csa
        rows = csa.rows_from_logical(case)
        done, spent, tok = 0, 0.0, 0
        while spent < min(args.cpu_seconds, 10.0) and tok < T:
            t_0 = time.perf_counter()
            csa.attention(case, ATTN_SCALE, tokens=[tok], rows=rows)
            spent += time.perf_counter() - t_0
            done += int((case.attn_indices[tok] >= 0).sum())
            tok += 1
        cpu = {"value": done / spent, "unit": "pairs/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle", "sample": "%d of %d tokens (%.1f s, numpy float64)" % (tok, T, spent)}
    if rank != 0:
        return
    print(json.dumps({
        "metric": "sparse attention over the selected positions: (token, listed position) pairs/s "
                  "(% of HBM roof)",
        "value": value, "unit": "pairs/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": synth.ATTN_WORKLOAD, "query_tokens": T, "heads": H,
                   "listed_per_token": case.attn_indices.shape[-1],
                   "l2": "a 256 MB read before each step, outside the events that time it",
                   "timing": "median of %d repeats of the %d-step region" % (len(times), args.steps),
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
        "clocks": clk.summary()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5],
                    help="workload (default 3: the prefill chunk, the largest single-GPU one)")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the timed region until this much GPU time has run")
    ap.add_argument("--op", default="index",
                    choices=["index", "quantize_q", "write_index_k", "sparse_attention"],
                    help="index: the indexer (default); the others time the query quantiser, "
                         "the index-K cache writer or the attention over the indices alone")
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0 = default)")
    ap.add_argument("--long-requests", type=int, default=8,
                    help="workload 5 only: 1M-context requests kept (8 = the workload; fewer "
                         "for profiler captures that must stay small)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-rows", type=int, default=4)
    ap.add_argument("--ref-rows", type=int, default=4, help="oracle rows per reference step")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.op != "index":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "op": args.op,
                              "unavailable": "the reference arm times the indexer only"}))
            return
        run_attn(args) if args.op == "sparse_attention" else run_op(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
