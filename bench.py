#!/usr/bin/env python
"""Decode-step benchmark of the Locks hot path on GB300.

A step is one decode step of one attention layer over the whole batch:
locks_select (page scoring, shares, share-average, top-k) followed by
locks_sparse_decode (attention over the selected pages).  Summaries are built
once before timing (their build rate is reported separately), and the dense
full-cache decode kernel is timed on the same inputs as the comparison point.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl locks|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
replica batch (weak scaling, no collective on the data path); value is the
tokens of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step µs and tokens/s at 1 GB300 (sparse vs dense); achieved HBM GB/s vs peak"
DEFAULT_CONFIG = "llama32k"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("locks", "reference"), default="locks")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--summary", choices=("f32", "bf16", "i4"), default="f32",
                    help="summary record: fp32, bf16, or quantised (int4 basis, int8 "
                         "coefficients and centroid)")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-worker", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# peaks, clocks, profile summaries
# --------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(self.interval_ms / 1000.0 * 1.5)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = []
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((t, float(parts[2]), float(parts[3]), parts[5:]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or r[0])]
        use = inside or rows
        if not use:
            return None
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in use:
            for name, v in zip(names, r[3][1:5]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed region" if inside else "whole run (no sample inside the timed region)"}


def source_digest(files) -> str:
    """sha256 over the given repository files, concatenated in order."""
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic(kernel_key: str, config: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or None
    when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel_key}_{config}.md")
    if not os.path.exists(path):
        return None, None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    src = fields.get("source")
    want = fields.get("source_sha256")
    if not src or not want:
        return None, path
    if source_digest([x.strip() for x in src.split(",")]) != want:
        return None, path
    try:
        return float(fields["dram_bytes_per_launch"]), path
    except (KeyError, ValueError):
        return None, path


# --------------------------------------------------------------------------
# summary build diagnostics
# --------------------------------------------------------------------------
# FP32 ALU peak: 152 SMs x 128 FP32 lanes x 2 flops per fused multiply-add x
# 2.07 GHz (the maximum SM clock)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def build_flop_count(sweeps, B: int, d_head: int = 128, r: int = 8) -> float:
    """Floating-point operations the summary build executes, from the Jacobi
    sweeps each page-head used: centring (B d), the full Gram product
    (2 B^2 d), per sweep B-1 rounds that rotate the B x B matrix as (B/2)^2
    2 x 2 blocks (24 flops each) and the B x B eigenvector matrix (6 flops per
    row and pair), the convergence norms (2 B^2 per check), and the basis
    V = D^T U_r (2 d B r)."""
    import numpy as np
    sweeps = np.asarray(sweeps, dtype=np.float64)
    per_sweep = (B - 1) * (24 * (B // 2) ** 2 + 6 * B * (B // 2))
    fixed = B * d_head + 2 * B * B * d_head + 2 * d_head * B * r
    return float(sweeps.size * fixed + sweeps.sum() * per_sweep + (sweeps + 1).sum() * 2 * B * B)


def captured_energy(layer, ids_t, tail, w, sample: int = 4096):
    """Energy the rank-r summary captures per page-head, 1 - tau / ||D||_F^2
    (a diagnostic the paper reports for real pages, App. D): tau is the build's
    tail output; ||D||_F^2 of the centred keys is recomputed for a seeded
    sample of page-heads.  Outside the timed region."""
    import torch
    n = ids_t.numel()
    if n == 0:
        return None
    g = torch.Generator(device="cpu").manual_seed(12345)
    pick = torch.randperm(n, generator=g)[:max(1, sample // w.n_kv_heads)].to(ids_t.device)
    K = layer.k_cache[ids_t[pick].long()].float()               # [s, H_kv, B, d]
    D = K - K.mean(dim=2, keepdim=True)
    trace = (D * D).sum(dim=(2, 3))                              # [s, H_kv]
    frac = (1.0 - tail[pick] / trace.clamp_min(1e-30)).flatten().cpu()
    q = torch.quantile(frac, torch.tensor([0.1, 0.5, 0.9]))
    return {"page_heads_sampled": int(frac.numel()), "median": float(q[1]),
            "p10": float(q[0]), "p90": float(q[2]), "mean": float(frac.mean())}


# --------------------------------------------------------------------------
# replicas across ranks (weak scaling: every rank runs its own batch)
# --------------------------------------------------------------------------
def replica_workload(w, rank: int):
    """Rank r's replica of workload w: same shapes, its own seed."""
    return w.with_(seed=w.seed + 7919 * rank) if rank else w


def reduce_max(value: float, dist=None, device="cpu") -> float:
    """Maximum of a per-rank value over all ranks (the slowest rank's time)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(world: int, batch: int, step_ms_max: float) -> float:
    """Whole-job throughput: every rank's batch per step over the slowest rank's step."""
    return world * batch / (step_ms_max / 1e3)


# --------------------------------------------------------------------------
# CPU baseline: the oracle, in a fresh single-threaded process
# --------------------------------------------------------------------------
def cpu_worker(spec: str):
    """Run the oracle's decode step on a bounded sample; print JSON."""
    import numpy as np  # noqa: F401  (threads pinned by the parent's environment)
    import oracle as O
    import workloads as W
    d = json.loads(spec)
    w = W.get(d["config"])
    seqs = d["seqs"]
    w_s = w.with_(batch=seqs, seed=w.seed)      # the first `seqs` sequences' shapes and recipe
    x = W.generate(w_s)
    units = [(b, h) for b in range(seqs) for h in range(w.n_kv_heads)]
    summaries = {}
    t0 = time.time()
    for b, h in units:
        summaries[(b, h)] = O.build_unit(x.k_cache, x.block_table, int(x.seq_lens[b]), b, h, w.rank)
    t_build = time.time() - t0
    times = []
    for rep in range(d["steps"] + d["warmup"]):
        t0 = time.perf_counter()
        for b, h in units:
            O.run_unit(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, w.n_kv_heads,
                       w.rank, w.budget_tokens, b, h, summaries=summaries[(b, h)])
        dt = time.perf_counter() - t0
        if rep >= d["warmup"]:
            times.append(dt)
    per_step = statistics.median(times)
    print(json.dumps({"tokens_per_s": seqs / per_step, "step_s": per_step, "build_s": t_build,
                      "units": len(units), "seqs": seqs, "steps": len(times)}))


def run_cpu_baseline(config: str, seqs: int, steps: int, warmup: int):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    spec = json.dumps({"config": config, "seqs": seqs, "steps": steps, "warmup": warmup})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", spec],
                       capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle worker failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


# --------------------------------------------------------------------------
# reference arm: the oracle as the reference implementation
# --------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import workloads as W
    w = W.get(args.config)
    seqs = 1
    t0 = time.time()
    res = run_cpu_baseline(args.config, seqs, max(1, args.steps), max(0, args.warmup))
    wall = time.time() - t0
    value = res["tokens_per_s"]
    sample = (f"{seqs} of {w.batch} sequences ({res['units']} (sequence, KV head) units) of "
              f"{args.config}; oracle summaries built once ({res['build_s']:.1f} s) outside the "
              f"timed step; median of {res['steps']} steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["step_s"] * 1e3 * w.batch / seqs,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "batch": w.batch,
                                        "context": w.context, "description": w.description},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def algorithmic_bytes(layer, inputs, selected):
    """Bytes the method must move in one step (summary scan + selected K/V + q/o/ids)."""
    import numpy as np
    w = inputs.workload
    B = w.page_size
    rec = layer.rec_bytes
    n_cand_total = 0
    kv_tokens = 0
    for b in range(w.batch):
        t = int(inputs.seq_lens[b])
        n = -(-t // B)
        n_cand = max(0, min(n - 1, t // B) - 1)
        n_cand_total += n_cand * w.n_kv_heads
        for h in range(w.n_kv_heads):
            for j in selected[b, h]:
                if j >= 0:
                    kv_tokens += min(B, t - int(j) * B)
    q_bytes = w.batch * w.n_q_heads * w.head_dim * 2
    sel_bytes = selected.size * 4
    select_bytes = n_cand_total * rec + q_bytes + sel_bytes
    decode_bytes = kv_tokens * w.head_dim * 2 * 2 + q_bytes + sel_bytes + q_bytes
    dense_tokens = int(np.sum(inputs.seq_lens)) * w.n_kv_heads
    dense_bytes = dense_tokens * w.head_dim * 2 * 2 + 2 * q_bytes
    return select_bytes, decode_bytes, dense_bytes


def run_gpu(args):
    import numpy as np
    import torch
    import workloads as W
    from sparse_paged_kv_gb300 import binding as Bd
    from sparse_paged_kv_gb300 import build_lib, runtime

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # the oracle baseline runs first, in a fresh process, before this one does heavy GPU work
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_steps = 3
        cpu = run_cpu_baseline(args.config, 1, cpu_steps, 1)

    build_lib.build()
    Bd.load_library()
    w = replica_workload(W.get(args.config), rank)
    t0 = time.time()
    inputs = W.generate(w)
    gen_s = time.time() - t0
    sdt = {"f32": Bd.LOCKS_SUMMARY_F32, "bf16": Bd.LOCKS_SUMMARY_BF16,
           "i4": Bd.LOCKS_SUMMARY_I4}[args.summary]
    layer = runtime.LocksLayer.from_inputs(inputs, summary_dtype=sdt)
    stream = torch.cuda.current_stream()

    # ---- summary build (one-time, reported separately) ----
    ids = runtime.complete_page_blocks(inputs.block_table, inputs.seq_lens, w.page_size)
    ids_t = torch.from_numpy(ids).cuda()
    bstat = torch.zeros((len(ids), w.n_kv_heads), dtype=torch.int32, device="cuda")
    tail = torch.zeros((len(ids), w.n_kv_heads), dtype=torch.float32, device="cuda")
    layer.build(ids_t, status=bstat, tail_energy=tail)
    captured = captured_energy(layer, ids_t, tail, w)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    build_ms = []
    for _ in range(2):
        e0.record(stream)
        layer.build(ids_t, status=bstat)
        e1.record(stream)
        torch.cuda.synchronize()
        build_ms.append(e0.elapsed_time(e1))
    build_ms = min(build_ms)
    page_heads = len(ids) * w.n_kv_heads
    bstat_np = bstat.cpu().numpy()
    not_conv = int(((bstat_np >> 16) != 0).sum())
    build_flops = build_flop_count(bstat_np & 0xFFFF, w.page_size, r=w.rank)

    # In a decode loop each sequence completes a page every B steps and its
    # summary is built then (off the step's critical path, section 4): time the
    # build of one page per sequence (its last complete page, every KV head).
    last = torch.from_numpy(np.array(
        [inputs.block_table[b, max(0, int(inputs.seq_lens[b]) // w.page_size - 1)]
         for b in range(w.batch)], dtype=np.int32)).cuda()
    for _ in range(3):
        layer.build(last)
    torch.cuda.synchronize()
    crossing_us = []
    for _ in range(20):
        e0.record(stream)
        layer.build(last)
        e1.record(stream)
        torch.cuda.synchronize()
        crossing_us.append(e0.elapsed_time(e1) * 1e3)
    crossing_us = statistics.median(crossing_us)

    # L2 flush between steps: write 256 MiB (> the 129 MB L2), then read another
    # 256 MiB so the dirty lines are written back before the next timed step
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
    flush_rd = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
    flush_sink = torch.empty((), dtype=torch.float32, device="cuda")

    def flush_l2(i):
        flush.fill_(float(i & 7))
        torch.sum(flush_rd, dim=0, out=flush_sink)

    K, Wm = args.steps, args.warmup

    def timed(fn, n_steps, n_warm, marks=3):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(marks)] for _ in range(n_steps)]
        for i in range(n_warm):
            flush_l2(i)
            fn(None)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(n_steps):
            flush_l2(i)
            fn(evs[i])
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t_wall = time.perf_counter() - t_wall
        return evs, t_wall

    # ---- sparse step: select + sparse decode (events only at step bounds, so
    # the decode's programmatic launch overlaps the selection's tail) ----
    def step(ev):
        if ev:
            ev[0].record(stream)
        layer.select()
        layer.sparse_decode()
        if ev:
            ev[1].record(stream)

    sampler = ClockSampler(local)
    sampler.start()
    for i in range(max(Wm, 3)):          # clock ramp
        flush_l2(i)
        step(None)
    torch.cuda.synchronize()
    sampler.mark_begin()
    evs, wall = timed(step, K, Wm, marks=2)
    sampler.mark_end()
    clocks = sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    status = int(layer.status.cpu()[0])
    selected = layer.selected.cpu().numpy()
    select_bytes, decode_bytes, dense_bytes = algorithmic_bytes(layer, inputs, selected)
    mean_step = sum(step_ms) / K
    mean_step_max = reduce_max(mean_step, dist, "cuda")

    # ---- the same step replayed from a CUDA graph ----
    graph_ms, graph_err = None, None
    try:
        graph = layer.capture_step()

        def gstep(ev):
            if ev:
                ev[0].record(stream)
            graph.replay()
            if ev:
                ev[1].record(stream)

        gevs, _ = timed(gstep, max(1, min(K, 500)), min(Wm, 10), marks=2)
        graph_ms = [e[0].elapsed_time(e[1]) for e in gevs]
    except RuntimeError as exc:          # reported in the JSON line, never hidden
        graph_err = str(exc).splitlines()[0][:200]

    # ---- the two calls on their own (events between them), for the roofline ----
    K2 = max(1, min(K, 200))

    def sel_only(ev):
        if ev:
            ev[0].record(stream)
        layer.select()
        if ev:
            ev[1].record(stream)

    sevs, _ = timed(sel_only, K2, min(Wm, 10), marks=2)
    sel_ms = [e[0].elapsed_time(e[1]) for e in sevs]

    def dec_only(ev):
        layer.select()
        if ev:
            ev[0].record(stream)
        layer.sparse_decode()
        if ev:
            ev[1].record(stream)

    devs_, _ = timed(dec_only, K2, min(Wm, 10), marks=2)
    dec_ms = [e[0].elapsed_time(e[1]) for e in devs_]

    # ---- dense comparison ----
    dense = None
    if not args.no_dense:
        def dstep(ev):
            if ev:
                ev[0].record(stream)
            layer.dense_decode()
            if ev:
                ev[1].record(stream)
        devs, _ = timed(dstep, K, Wm, marks=2)
        dms = [e[0].elapsed_time(e[1]) for e in devs]
        dmean = sum(dms) / K
        dense = {"tokens_per_s": w.batch / (dmean / 1e3), "us_per_step": dmean * 1e3,
                 "us_median": statistics.median(dms) * 1e3,
                 "gbs": dense_bytes / (dmean / 1e3) / 1e9, "bytes_per_step": dense_bytes}

    # ---- end to end through the public API, host buffers ----
    e2e = None
    if not args.no_e2e:
        q_host = layer.q.cpu().pin_memory()
        out_host = torch.empty(layer.out.shape, dtype=layer.out.dtype).pin_memory()

        def estep(ev):
            if ev:
                ev[0].record(stream)
            layer.q.copy_(q_host, non_blocking=True)
            layer.step()
            out_host.copy_(layer.out, non_blocking=True)
            if ev:
                ev[1].record(stream)
        eevs, _ = timed(estep, K, Wm, marks=2)
        ems = reduce_max(sum(e[0].elapsed_time(e[1]) for e in eevs) / K, dist, "cuda")
        e2e = {"value": aggregate_tokens_per_s(world, w.batch, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
               "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
               "us_per_step": ems * 1e3}

    if dist:
        dist.barrier()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    sel_mean = sum(sel_ms) / len(sel_ms)
    achieved = select_bytes / (sel_mean / 1e3) / 1e9
    traffic, prof = profile_traffic("select", w.name if args.summary == "f32"
                                    else f"{w.name}_{args.summary}")
    step_gbs = (select_bytes + decode_bytes) / (mean_step / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": aggregate_tokens_per_s(world, w.batch, mean_step_max),
        "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": mean_step_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
                   "context": w.context, "rank": w.rank, "budget_tokens": w.budget_tokens,
                   "summary": args.summary, "kv": "bf16",
                   "l2": "flushed before every timed step (256 MiB write, then a 256 MiB read)",
                   "step": "locks_select + locks_sparse_decode, one layer",
                   "parallelism": f"replicas x{world}"},
        "step_us": {"mean": mean_step * 1e3, "median": statistics.median(step_ms) * 1e3,
                    "p10": sorted(step_ms)[K // 10] * 1e3, "p90": sorted(step_ms)[(9 * K) // 10] * 1e3,
                    "select_alone_mean": sel_mean * 1e3,
                    "sparse_decode_alone_mean": sum(dec_ms) / len(dec_ms) * 1e3,
                    "graph_replay_mean": (sum(graph_ms) / len(graph_ms) * 1e3) if graph_ms else None,
                    "graph_replay_median": statistics.median(graph_ms) * 1e3 if graph_ms else None},
        "graph_error": graph_err,
        "step_gbs": step_gbs,
        "step_frac": step_gbs / peak,
        "roofline": {"bound": "hbm", "kernel": "locks_select (score_kernel + finalize_kernel)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes": select_bytes},
        "sparse_decode": {"gbs": decode_bytes / (sum(dec_ms) / len(dec_ms) / 1e3) / 1e9,
                          "bytes_per_step": decode_bytes},
        "dense": dense,
        "speedup_vs_dense": (dense["us_per_step"] / (mean_step * 1e3)) if dense else None,
        "build": {"ms": build_ms, "page_heads": page_heads, "pages_per_s": len(ids) / (build_ms / 1e3),
                  "page_heads_per_s": page_heads / (build_ms / 1e3), "not_converged": not_conv,
                  "mean_sweeps": float((bstat_np & 0xFFFF).mean()),
                  "roofline": {"bound": "alu", "achieved": build_flops / (build_ms / 1e3) / 1e12,
                               "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s",
                               "frac": build_flops / (build_ms / 1e3) / 1e12 / FP32_ALU_TFLOPS,
                               "flops": build_flops},
                  "captured_energy": captured,
                  "page_crossing_us": crossing_us,
                  "page_crossing_per_step_us": crossing_us / w.page_size,
                  "page_crossing_fraction_of_step": crossing_us / w.page_size / (mean_step * 1e3),
                  "page_crossing_note": "one completed page per sequence (all KV heads) "
                                        "built every B decode steps; amortised per step"},
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clocks,
        "device_status": status,
        "input_gen_s": gen_s,
        "wall_timed_s": wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = {"value": cpu["tokens_per_s"], "unit": "tokens/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"1 of {w.batch} sequences ({cpu['units']} units) of "
                                          f"{w.name}, median of {cpu['steps']} oracle steps "
                                          f"(select + attend; summaries prebuilt)"}
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_worker:
        cpu_worker(args.cpu_worker)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
