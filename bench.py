#!/usr/bin/env python
"""Decode-step benchmark of the Locks hot path on GB300.

A step is one decode step of one attention layer over the whole batch:
locks_select (page scoring, shares, share-average, top-k) followed by
locks_sparse_decode (attention over the selected pages).  Summaries are built
once before timing (their build rate is reported separately), and the dense
full-cache decode kernel is timed on the same inputs as the comparison point.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config all|NAME]
                  [--summary f32|bf16|i4] [--extra-summary i4,...] [--impl locks|reference]

With the default ``--config all`` every workload is measured in one process
(tiny, llama32k, long128k, qwen16k, 1m); the headline numbers of the JSON line
are those of the largest, 1m (Llama-3.1-8B layer shape, batch 1, 1,048,576
tokens), and ``per_config`` holds every workload's step, select and decode
times, HBM fractions, the dense kernel and the CPU oracle beside them.

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
replica batch (weak scaling, no collective on the data path); value is the
tokens of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
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
HEADLINE_CONFIG = "1m"
ALL_CONFIGS = ("tiny", "llama32k", "long128k", "qwen16k", "1m")
FALLBACK_HBM_GBS = 6800.0
# kernels one sparse step launches: score, finalize (select) and decode
LAUNCHES_PER_STEP = 3


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("locks", "reference"), default="locks")
    ap.add_argument("--config", default="all",
                    help="'all' (every workload, 1m as the headline) or one workload name")
    ap.add_argument("--summary", choices=("f32", "bf16", "i4"), default="f32",
                    help="summary record of the headline step: fp32, bf16, or quantised "
                         "(int4 basis, int8 coefficients and centroid)")
    ap.add_argument("--extra-summary", default="i4",
                    help="comma-separated record types also measured per workload ('' for none)")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-loop", action="store_true", help="skip the decode-loop measurement")
    ap.add_argument("--cpu-worker", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def config_list(arg: str):
    if arg == "all":
        return list(ALL_CONFIGS), HEADLINE_CONFIG
    return [arg], arg


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
    """SM clock and clock-event (throttle) reasons of one GPU, read through
    NVML by a background thread every half millisecond while a region runs,
    plus one reading at each end of the region.  Reading only: nothing is
    set.  Without NVML the sampler reports nothing."""

    NVML_CLOCK_SM = 1
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, interval_s: float = 0.0005):
        self.interval_s = interval_s
        self.lib = None
        self.handle = ctypes.c_void_p()
        self.samples = {}            # region name -> [(sm_mhz, reasons mask)]
        self.max_mhz = None
        self.error = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            if not self._handle(lib, cuda_index):
                raise OSError("no NVML handle for the CUDA device")
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(self.handle, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.lib = lib
        except (OSError, AttributeError) as exc:
            self.error = str(exc)[:200]

    def _handle(self, lib, cuda_index: int) -> bool:
        try:
            import torch
            p = torch.cuda.get_device_properties(cuda_index)
            bus = "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle)) == 0:
                return True
        except (AttributeError, RuntimeError):
            pass
        return lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.handle)) == 0

    def read(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ctypes.byref(clk)) != 0:
            return None
        if self.reason_fn(self.handle, ctypes.byref(rs)) != 0:
            return None
        return float(clk.value), int(rs.value)

    class _Region:
        def __init__(self, sampler, name):
            self.s, self.name, self.stop = sampler, name, threading.Event()

        def _loop(self):
            out = self.s.samples.setdefault(self.name, [])
            while not self.stop.is_set():
                r = self.s.read()
                if r:
                    out.append(r)
                time.sleep(self.s.interval_s)

        def __enter__(self):
            if self.s.lib is None:
                return self
            r = self.s.read()
            if r:
                self.s.samples.setdefault(self.name, []).append(r)
            self.t = threading.Thread(target=self._loop, daemon=True)
            self.t.start()
            return self

        def __exit__(self, *exc):
            if self.s.lib is None:
                return False
            self.stop.set()
            self.t.join(timeout=2)
            r = self.s.read()
            if r:
                self.s.samples.setdefault(self.name, []).append(r)
            return False

    def region(self, name: str):
        return self._Region(self, name)

    def summary(self, names=None):
        if self.lib is None:
            return {"error": self.error or "NVML unavailable"}
        rows = [r for n, v in self.samples.items() if names is None or n in names for r in v]
        if not rows:
            return {"error": "no sample"}
        reasons = sorted({name for _, m in rows for bit, name in self.REASON_BITS.items() if m & bit})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_min_mhz": min(r[0] for r in rows),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(rows),
                "window": "timed region (NVML, in process)"}


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


def trd_flop_count(n_page_heads: int, B: int, d_head: int = 128, r: int = 8, rounds: int = 6,
                   iters: int = 2) -> float:
    """Floating-point operations of the tridiagonal top-r build per page-heads:
    centring (B d), the Gram (2 B^2 d), the Householder reduction (a
    matrix-vector product and a rank-2 update of the trailing m x m block per
    step, 6 m^2, about 2 B^3 in all), the bisection (r eigenvalues x rounds x
    16 Sturm counts of B steps, 4 flops each), inverse iteration (r x iters x
    B x 12), the Rayleigh quotients (6 r B), the back-transformation (4 m per
    vector and step, about 2 r B^2) and the basis V = D^T U_r (2 d B r)."""
    tri = sum(6 * m * m for m in range(2, B))
    per = (B * d_head + 2 * B * B * d_head + tri + r * rounds * 16 * B * 4 + r * iters * B * 12 +
           6 * r * B + 2 * r * B * B + 2 * d_head * B * r)
    return float(n_page_heads) * per


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
# CPU baseline: the oracle, in fresh single-threaded processes
# --------------------------------------------------------------------------
def baseline_units(w):
    """(sequence, KV head) units the CPU sample covers: the whole first
    sequence of the small workload, one unit of the others."""
    if w.context * w.n_kv_heads <= 16384:
        return [(0, h) for h in range(w.n_kv_heads)]
    return [(0, 0)]


def cpu_worker(spec: str):
    """Run the oracle's decode step on a bounded sample; print JSON.

    The sample is a list of (sequence, KV head) units of the workload; only
    their keys and values are generated (the same bytes as in the full
    workload).  Their summaries are built once, outside the timed steps; a
    timed step is select + attend for every listed unit."""
    import oracle as O
    import workloads as W
    d = json.loads(spec)
    w = W.get(d["config"])
    units = [tuple(u) for u in d["units"]]
    seqs = 1 + max(b for b, _ in units)
    w_s = w.with_(batch=seqs)                  # the first sequences' shapes and recipe
    t0 = time.time()
    x = W.generate(w_s, units=units)
    t_gen = time.time() - t0
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
    tokens = len(units) / w.n_kv_heads         # a token of one sequence needs every KV head
    print(json.dumps({"tokens_per_s": tokens / per_step, "step_s": per_step, "steps_s": times,
                      "build_s": t_build, "gen_s": t_gen, "units": len(units),
                      "tokens_per_step": tokens, "steps": len(times)}))


def start_cpu_baseline(config: str, units, steps: int, warmup: int):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    spec = json.dumps({"config": config, "units": [list(u) for u in units], "steps": steps,
                       "warmup": warmup})
    return subprocess.Popen([sys.executable, os.path.abspath(__file__), "--cpu-worker", spec],
                            stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env)


def finish_cpu_baseline(proc, timeout=1800):
    out, err = proc.communicate(timeout=timeout)
    if proc.returncode != 0:
        raise RuntimeError("oracle worker failed: " + err[-2000:])
    return json.loads(out.strip().splitlines()[-1])


def cpu_baseline_entry(w, res):
    return {"value": res["tokens_per_s"], "unit": "tokens/s", "cores": 1,
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{res['units']} of {w.batch * w.n_kv_heads} (sequence, KV head) units of "
                      f"{w.name} per step ({res['tokens_per_step']:g} token of one sequence's "
                      f"layer step); fp64 NumPy oracle, one thread, median of {res['steps']} "
                      f"steps of select + attend (summaries built once outside, "
                      f"{res['build_s']:.1f} s)"}


# --------------------------------------------------------------------------
# reference arm: the oracle as the reference implementation
# --------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import workloads as W
    _, head = config_list(args.config)
    w = W.get(head)
    units = baseline_units(w)
    t0 = time.time()
    res = finish_cpu_baseline(start_cpu_baseline(head, units, max(1, args.steps),
                                                 max(0, args.warmup)))
    wall = time.time() - t0
    value = res["tokens_per_s"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(res["steps_s"]) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "batch": w.batch,
                                        "context": w.context, "description": w.description},
        "cpu_baseline": cpu_baseline_entry(w, res),
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


FLUSH_NOTE = "flushed before every timed step (256 MiB write, then a 256 MiB read)"


def record_stream_bytes(w, rec_bytes: int) -> int:
    """Summary-record bytes one step scans (every candidate page of every unit)."""
    B = w.page_size
    n = 0
    for t in w.lengths():
        pages = -(-t // B)
        n += max(0, min(pages - 1, t // B) - 1)
    return n * w.n_kv_heads * rec_bytes


def l2_policy(torch, w, rec_bytes: int):
    """(flush?, note): no flush when the records a step streams are at least
    twice the L2, so that no step finds the previous one's data there; else an
    L2 flush before every timed step."""
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0)) or 132 * 2 ** 20
    rb = record_stream_bytes(w, rec_bytes)
    if rb >= 2 * l2:
        return False, (f"inputs larger than L2: every step streams {rb / 1e6:.0f} MB of summary "
                       f"records (>= 2x the {l2 / 1e6:.0f} MB L2) before its decode; no flush")
    return True, FLUSH_NOTE


def gpu_spin(torch, stream, ms: float = 5.0):
    """Keep the device busy for about ms milliseconds (torch's spin kernel,
    at the 2.07 GHz SM clock) on `stream`."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 2.07e6))


class Timer:
    """Event-timed loops on one stream, with (flush=True) an L2 flush before
    every iteration: write 256 MiB (> the 129 MB L2), then read another
    256 MiB so the dirty lines are written back before the timed work."""

    def __init__(self, torch, stream, dist):
        self.torch, self.stream, self.dist = torch, stream, dist
        self.flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
        self.flush_rd = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
        self.flush_sink = torch.empty((), dtype=torch.float32, device="cuda")
        self.enabled = True

    def flush_l2(self, i):
        if not self.enabled:
            return
        self.flush.fill_(float(i & 7))
        self.torch.sum(self.flush_rd, dim=0, out=self.flush_sink)

    def run(self, fn, n_steps, n_warm, region=None):
        """fn(ev) with ev = (start, end) events to record around the timed
        work, or None during warm-up; returns per-iteration milliseconds."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_steps)]
        for i in range(n_warm):
            self.flush_l2(i)
            fn(None)
        torch.cuda.synchronize()
        if self.dist:
            self.dist.barrier()
        torch.cuda.synchronize()
        ctx = region if region is not None else _Null()
        with ctx:
            for i in range(n_steps):
                self.flush_l2(i)
                fn(evs[i])
            torch.cuda.synchronize()
        if self.dist:
            self.dist.barrier()
        return [a.elapsed_time(b) for a, b in evs]

    def run_region(self, fn, n_steps, n_warm, region=None):
        """fn(None) n_steps times back to back, timed as one region: events
        at its two ends only, a synchronize and a barrier on both sides.
        Returns milliseconds per iteration.  For workloads timed without an
        L2 flush (the flush kernels would otherwise fall inside the region)."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(n_warm):
            fn(None)
        torch.cuda.synchronize()
        if self.dist:
            self.dist.barrier()
        torch.cuda.synchronize()
        ctx = region if region is not None else _Null()
        with ctx:
            # a spin on the device before the region, so that the host has
            # queued the region's launches by the time it starts: the region
            # then holds device time only, not the host's first launches
            gpu_spin(torch, self.stream)
            e0.record(self.stream)
            for _ in range(n_steps):
                fn(None)
            e1.record(self.stream)
            torch.cuda.synchronize()
        if self.dist:
            self.dist.barrier()
        return e0.elapsed_time(e1) / n_steps


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def stats_us(ms):
    s = sorted(ms)
    n = len(s)
    return {"mean": sum(s) / n * 1e3, "median": statistics.median(s) * 1e3,
            "p10": s[n // 10] * 1e3, "p90": s[(9 * n) // 10] * 1e3}


def measure_record(layer, inputs, timer, K, Wm, sampler, tag, full, args, world, dist):
    """Build, then time the sparse step and its parts on one layer."""
    import numpy as np
    import torch
    from sparse_paged_kv_gb300 import runtime
    w = inputs.workload
    stream = torch.cuda.current_stream()
    res = {}
    timer.enabled, res["l2"] = l2_policy(torch, w, layer.rec_bytes)

    # ---- summary build (one-time, reported separately) ----
    ids = runtime.complete_page_blocks(inputs.block_table, inputs.seq_lens, w.page_size)
    ids_t = torch.from_numpy(ids).cuda()
    bstat = torch.zeros((len(ids), w.n_kv_heads), dtype=torch.int32, device="cuda")
    tail = torch.zeros((len(ids), w.n_kv_heads), dtype=torch.float32, device="cuda")
    layer.build(ids_t, status=bstat, tail_energy=tail)
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
    trd = w.page_size == 64            # the default solver at B = 64 (no sweep cap passed)
    build_flops = (trd_flop_count(bstat_np.size, w.page_size, r=w.rank) if trd
                   else build_flop_count(bstat_np & 0xFFFF, w.page_size, r=w.rank))
    res["build"] = {"solver": "tridiagonal (Householder, bisection, inverse iteration)" if trd
                    else "cyclic Jacobi", "ms": build_ms, "page_heads": page_heads,
                    "pages_per_s": len(ids) / (build_ms / 1e3),
                    "page_heads_per_s": page_heads / (build_ms / 1e3),
                    "not_converged": int(((bstat_np >> 16) != 0).sum()),
                    "mean_sweeps": float((bstat_np & 0xFFFF).mean()) if bstat_np.size else 0.0,
                    "roofline": {"bound": "alu",
                                 "achieved": build_flops / (build_ms / 1e3) / 1e12,
                                 "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s",
                                 "peak_kind": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz",
                                 "frac": build_flops / (build_ms / 1e3) / 1e12 / FP32_ALU_TFLOPS,
                                 "flops": build_flops}}
    if full:
        res["build"]["captured_energy"] = captured_energy(layer, ids_t, tail, w)
        # In a decode loop each sequence completes a page every B decode steps
        # and its summary is built then (off the step's critical path, section
        # 4): time the build of one page per sequence (its last complete page,
        # every KV head).
        last = torch.from_numpy(np.array(
            [inputs.block_table[b, max(0, int(inputs.seq_lens[b]) // w.page_size - 1)]
             for b in range(w.batch)], dtype=np.int32)).cuda()
        for _ in range(3):
            layer.build(last)
        torch.cuda.synchronize()
        cr = []
        for _ in range(20):
            e0.record(stream)
            layer.build(last)
            e1.record(stream)
            torch.cuda.synchronize()
            cr.append(e0.elapsed_time(e1) * 1e3)
        cr = statistics.median(cr)
        res["build"].update({"page_crossing_us": cr, "page_crossing_per_step_us": cr / w.page_size,
                             "page_crossing_note": "one completed page per sequence (all KV heads) "
                                                   "built every B decode steps; amortised per step"})

    # ---- sparse step: select + sparse decode (events only at step bounds, so
    # the decode's programmatic launch overlaps the selection's tail) ----
    def step(ev):
        if ev:
            ev[0].record(stream)
        layer.select()
        layer.sparse_decode()
        if ev:
            ev[1].record(stream)

    for i in range(max(Wm, 3)):          # clock ramp
        timer.flush_l2(i)
        step(None)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    step_ms = timer.run(step, K, Wm, sampler.region(f"{tag}:step"))
    res["wall_timed_s"] = time.perf_counter() - t_wall
    res["step_ms"] = step_ms
    res["status"] = int(layer.status.cpu()[0])
    selected = layer.selected.cpu().numpy()
    res["bytes"] = algorithmic_bytes(layer, inputs, selected)
    # Without a flush between steps the K steps also run back to back as one
    # timed region (as a decode loop runs them: each step's first kernel
    # launches while the previous step's last one finishes), and that time
    # per step is the headline; with a flush, the per-step events are.
    if not timer.enabled:
        t_wall = time.perf_counter()
        res["step_region_ms"] = timer.run_region(step, K, Wm, sampler.region(f"{tag}:step"))
        res["wall_timed_s"] += time.perf_counter() - t_wall
        res["step_timing"] = "K steps back to back, timed as one region (no L2 flush)"
        res["step_mean_max_ms"] = reduce_max(res["step_region_ms"], dist, "cuda")
    else:
        res["step_timing"] = "CUDA events around each step (L2 flushed between steps)"
        res["step_mean_max_ms"] = reduce_max(sum(step_ms) / K, dist, "cuda")

    # ---- the same step replayed from a CUDA graph ----
    res["graph_ms"], res["graph_error"] = None, None
    if full:
        try:
            graph = layer.capture_step()

            def gstep(ev):
                if ev:
                    ev[0].record(stream)
                graph.replay()
                if ev:
                    ev[1].record(stream)

            res["graph_ms"] = timer.run(gstep, K, Wm)
        except RuntimeError as exc:          # reported in the JSON line, never hidden
            res["graph_error"] = str(exc).splitlines()[0][:200]

    # ---- the two calls on their own, for the roofline ----
    def sel_only(ev):
        if ev:
            ev[0].record(stream)
        layer.select()
        if ev:
            ev[1].record(stream)

    res["sel_ms"] = timer.run(sel_only, K, Wm, sampler.region(f"{tag}:select"))

    def dec_only(ev):
        layer.select()
        if ev:
            ev[0].record(stream)
        layer.sparse_decode()
        if ev:
            ev[1].record(stream)

    res["dec_ms"] = timer.run(dec_only, K, Wm)

    # ---- end to end through the public API, host buffers ----
    # Every step copies its queries from pinned host memory and reads its
    # output back.  Without an L2 flush the steps run back to back as one
    # timed region, pipelined the way a serving loop runs them: the queries
    # of step i go up on one copy stream while step i - 1 computes, its output
    # comes down on another while step i + 1 computes (two device buffers of
    # each); the region ends when the last output is in host memory.  With a
    # flush each step is timed alone, copies in line.
    res["e2e"] = None
    if full and not args.no_e2e:
        q0, out0 = layer.q, layer.out
        q_host = q0.cpu().pin_memory()
        out_host = [torch.empty(out0.shape, dtype=out0.dtype).pin_memory() for _ in range(2)]
        if timer.enabled:
            def estep(ev):
                if ev:
                    ev[0].record(stream)
                layer.q.copy_(q_host, non_blocking=True)
                layer.step()
                out_host[0].copy_(layer.out, non_blocking=True)
                if ev:
                    ev[1].record(stream)
            ems = reduce_max(sum(timer.run(estep, K, Wm)) / K, dist, "cuda")
            how = "each step timed alone: H2D of q, select + sparse decode, D2H of out, in line"
        else:
            qd, od = [q0, torch.empty_like(q0)], [out0, torch.empty_like(out0)]
            up, down = torch.cuda.Stream(), torch.cuda.Stream()
            ev_step = [torch.cuda.Event(), torch.cuda.Event()]
            ev_in = [torch.cuda.Event(), torch.cuda.Event()]
            ev_out = [torch.cuda.Event(), torch.cuda.Event()]

            def pipelined(n):
                for i in range(n):
                    b = i & 1
                    if i >= 2:
                        up.wait_event(ev_step[b])         # step i - 2 has read qd[b]
                        stream.wait_event(ev_out[b])      # and its output has left od[b]
                    with torch.cuda.stream(up):
                        qd[b].copy_(q_host, non_blocking=True)
                    ev_in[b].record(up)
                    stream.wait_event(ev_in[b])
                    layer.q, layer.out = qd[b], od[b]
                    layer.step()
                    ev_step[b].record(stream)
                    down.wait_event(ev_step[b])
                    with torch.cuda.stream(down):
                        out_host[b].copy_(od[b], non_blocking=True)
                    ev_out[b].record(down)
                stream.wait_event(ev_out[(n - 1) & 1])

            def erun(ev):
                if ev:
                    gpu_spin(torch, stream)               # host launches queue up first
                    ev[0].record(stream)
                    up.wait_event(ev[0])                  # the first copy is inside the region
                pipelined(K)
                if ev:
                    ev[1].record(stream)
            try:
                ems = reduce_max(sum(timer.run(erun, 1, 1)) / K, dist, "cuda")
            finally:
                torch.cuda.synchronize()
                layer.q, layer.out = q0, out0
            how = ("K steps back to back as one region: H2D of each step's q on one copy "
                   "stream, D2H of its out on another, overlapping the neighbouring steps")
        res["e2e"] = {"value": aggregate_tokens_per_s(world, w.batch, ems), "unit": "tokens/s",
                      "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
                      "d2h_bytes_per_step": out0.numel() * out0.element_size(),
                      "us_per_step": ems * 1e3, "timing": how}
    return res


def measure_decode_loop(layer, w, sampler, tag, reps=5):
    """B consecutive decode-loop steps (locks_append_kv, locks_build_completed
    on a side stream, select, sparse decode) starting from length T - B, so
    the last step completes one page per sequence and its build runs as it
    would in an engine; against B consecutive plain steps (select + sparse
    decode) on the same inputs.  No L2 flush inside either run.  The
    difference per step is the amortised cost of appending and of the
    page-crossing refresh.  The appended rows overwrite the last page's keys
    and values with new random ones; lengths end where they started."""
    import numpy as np
    import torch
    from sparse_paged_kv_gb300 import runtime
    B = w.page_size
    stream = torch.cuda.current_stream()
    g = torch.Generator(device="cuda").manual_seed(99)
    rows = torch.randn((B, 2, w.batch, w.n_kv_heads, w.head_dim), generator=g, device="cuda")
    rows = rows.to(torch.bfloat16)
    lens0 = layer.seq_lens.clone()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def plain():
        gpu_spin(torch, stream)
        e0.record(stream)
        for _ in range(B):
            layer.select()
            layer.sparse_decode()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    host_lens = np.asarray(layer.host_seq_lens, dtype=np.int64)

    def looped():
        layer.seq_lens.copy_(lens0 - B)
        loop = runtime.DecodeLoop(layer, host_lengths=host_lens - B)
        torch.cuda.synchronize()
        gpu_spin(torch, stream)
        e0.record(stream)
        for s in range(B):
            loop.step(rows[s, 0], rows[s, 1])
        loop.finish()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), loop

    plain()
    looped()
    with sampler.region(f"{tag}:loop"):
        p_ms = [plain() for _ in range(reps)]
        l_out = [looped() for _ in range(reps)]
    l_ms = [x[0] for x in l_out]
    done = l_out[-1][1].completed[(B - 1) & 1].cpu().numpy()
    ok = bool((done >= 0).all()) and torch.equal(layer.seq_lens, lens0)
    p_us = statistics.median(p_ms) * 1e3 / B
    l_us = statistics.median(l_ms) * 1e3 / B
    return {"steps": B, "runs": reps, "plain_us_per_step": p_us, "loop_us_per_step": l_us,
            "refresh_us_per_step": l_us - p_us, "refresh_fraction_of_step": (l_us - p_us) / p_us,
            "pages_completed_per_run": int((done >= 0).sum()), "completions_as_expected": ok,
            "note": "B consecutive steps, no L2 flush: append + (on the step that completes a "
                    "page) its build on a side stream + select + sparse decode, against select + "
                    "sparse decode"}


def measure_dense(layer, inputs, timer, K, Wm, sampler, tag):
    """The dense decode on the same inputs; it reads the whole K/V cache, so
    it is flushed like a step only when the cache is under twice the L2."""
    import torch
    stream = torch.cuda.current_stream()
    w = inputs.workload
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0)) or 132 * 2 ** 20
    timer.enabled = sum(w.lengths()) * w.n_kv_heads * w.head_dim * 4 < 2 * l2

    def dstep(ev):
        if ev:
            ev[0].record(stream)
        layer.dense_decode()
        if ev:
            ev[1].record(stream)
    return timer.run(dstep, K, Wm, sampler.region(f"{tag}:dense"))


def summarise(w, res, peak, world, dense_ms=None):
    """Per-workload numbers of one record type."""
    select_bytes, decode_bytes, dense_bytes = res["bytes"]
    step = stats_us(res["step_ms"])
    step_t = res["step_mean_max_ms"] * 1e3          # the headline time per step, us
    sel_us = stats_us(res["sel_ms"])["mean"]
    dec_us = stats_us(res["dec_ms"])["mean"]
    step_gbs = (select_bytes + decode_bytes) / (step_t / 1e6) / 1e9
    sel_gbs = select_bytes / (sel_us / 1e6) / 1e9
    out = {"l2": res["l2"], "step_timing": res["step_timing"], "step_time_us": step_t,
           "step_us": step,
           "tokens_per_s": aggregate_tokens_per_s(world, w.batch, res["step_mean_max_ms"]),
           "select_alone_us": sel_us, "sparse_decode_alone_us": dec_us,
           "select_gbs": sel_gbs, "select_frac": sel_gbs / peak,
           "sparse_decode_gbs": decode_bytes / (dec_us / 1e6) / 1e9,
           "sparse_decode_frac": decode_bytes / (dec_us / 1e6) / 1e9 / peak,
           "step_gbs": step_gbs, "step_frac": step_gbs / peak,
           "select_bytes": select_bytes, "sparse_decode_bytes": decode_bytes,
           "build_page_heads_per_s": res["build"]["page_heads_per_s"],
           "device_status": res["status"]}
    if res.get("graph_ms"):
        out["graph_replay_us"] = stats_us(res["graph_ms"])
    if res.get("graph_error"):
        out["graph_error"] = res["graph_error"]
    if dense_ms is not None:
        d = stats_us(dense_ms)
        out["dense"] = {"us": d["mean"], "us_median": d["median"],
                        "tokens_per_s": w.batch / (d["mean"] / 1e6),
                        "gbs": dense_bytes / (d["mean"] / 1e6) / 1e9,
                        "frac": dense_bytes / (d["mean"] / 1e6) / 1e9 / peak,
                        "bytes_per_step": dense_bytes}
        out["speedup_vs_dense"] = d["mean"] / step_t
    return out


def run_gpu(args):
    import torch
    import workloads as W
    from sparse_paged_kv_gb300 import binding as Bd
    from sparse_paged_kv_gb300 import build_lib, runtime

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    names, head = config_list(args.config)
    extras = [s for s in args.extra_summary.split(",") if s and s != args.summary]
    SDT = {"f32": Bd.LOCKS_SUMMARY_F32, "bf16": Bd.LOCKS_SUMMARY_BF16, "i4": Bd.LOCKS_SUMMARY_I4}

    # the oracle baselines run first, in fresh single-threaded processes (one
    # per workload, side by side), before this one does any GPU work
    cpu = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        procs = {n: start_cpu_baseline(n, baseline_units(W.get(n)), 3, 1) for n in names}
        for n, p in procs.items():
            cpu[n] = finish_cpu_baseline(p)

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build_lib.build()
    Bd.load_library()
    sampler = ClockSampler(local)
    timer = Timer(torch, torch.cuda.current_stream(), dist)
    peak, peak_kind = measured_peaks()
    K, Wm = args.steps, args.warmup

    per_config, headline = {}, None
    for name in names:
        w = replica_workload(W.get(name), rank)
        t0 = time.time()
        inputs = W.generate(w)
        gen_s = time.time() - t0
        layer = runtime.LocksLayer.from_inputs(inputs, summary_dtype=SDT[args.summary])
        is_head = name == head
        res = measure_record(layer, inputs, timer, K, Wm, sampler, f"{name}:{args.summary}",
                             is_head, args, world, dist)
        dense_ms = None if args.no_dense else measure_dense(layer, inputs, timer, K, Wm, sampler,
                                                            name)
        entry = {"workload": name, "batch": w.batch, "context": w.context,
                 "k_pages": layer.k, "input_gen_s": gen_s}
        entry[args.summary] = summarise(w, res, peak, world, dense_ms)
        for ex in extras:
            other = layer.sharing_inputs(SDT[ex])
            r2 = measure_record(other, inputs, timer, K, Wm, sampler, f"{name}:{ex}", False,
                                args, world, dist)
            s2 = summarise(w, r2, peak, world, None)
            if dense_ms is not None:
                s2["speedup_vs_dense"] = stats_us(dense_ms)["mean"] / s2["step_time_us"]
            entry[ex] = s2
            del other
        if not args.no_loop:
            entry[args.summary]["decode_loop"] = measure_decode_loop(layer, w, sampler, name)
        if name in cpu:
            entry["cpu_baseline"] = cpu_baseline_entry(w, cpu[name])
        per_config[name] = entry
        if is_head:
            headline = (w, res, entry)
        del layer, inputs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    if dist:
        dist.barrier()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    w, res, entry = headline
    main = entry[args.summary]
    select_bytes, decode_bytes, _ = res["bytes"]
    traffic, _ = profile_traffic("select", w.name if args.summary == "f32"
                                 else f"{w.name}_{args.summary}")
    line = {
        "metric": METRIC,
        "value": main["tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": res["step_mean_max_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
                   "context": w.context, "rank": w.rank, "budget_tokens": w.budget_tokens,
                   "summary": args.summary, "kv": "bf16",
                   "l2": res["l2"],
                   "step": "locks_select + locks_sparse_decode, one layer",
                   "parallelism": f"replicas x{world}"},
        "step_timing": main["step_timing"],
        "step_us": main["step_us"],
        "select_alone_us": main["select_alone_us"],
        "sparse_decode_alone_us": main["sparse_decode_alone_us"],
        "graph_replay_us": main.get("graph_replay_us"),
        "step_gbs": main["step_gbs"],
        "step_frac": main["step_frac"],
        "roofline": {"bound": "hbm", "kernel": "locks_select (score_kernel + finalize_kernel)",
                     "achieved": main["select_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": main["select_frac"], "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes": select_bytes},
        "sparse_decode": {"gbs": main["sparse_decode_gbs"], "frac": main["sparse_decode_frac"],
                          "bytes_per_step": decode_bytes},
        "dense": main.get("dense"),
        "speedup_vs_dense": main.get("speedup_vs_dense"),
        "build": res["build"],
        "decode_loop": main.get("decode_loop"),
        "e2e": res["e2e"],
        "gpu_launches": LAUNCHES_PER_STEP * K,
        "clocks": sampler.summary([f"{w.name}:{args.summary}:step"]),
        "clocks_all_regions": sampler.summary(),
        "device_status": res["status"],
        "wall_timed_s": res["wall_timed_s"],
        "per_config": per_config,
    }
    if w.name in cpu:
        line["cpu_baseline"] = entry["cpu_baseline"]
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
