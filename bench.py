"""Benchmark of the attention forward pass (TFLOP/s, one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llm_prefill|long_sequence|max_shift|ragged_causal|tiny]

A step is one attention forward over the whole workload (all heads, all
query tiles). ``value`` is whole-job TFLOP/s (4·B·H·N²·d per step, halved
under the causal mask, summed over ranks) with inputs already in HBM, timed
with CUDA events over exactly K steps between barriers (max over ranks).
``e2e`` is the same metric with the inputs copied from pinned host memory
and O/LSE copied back inside the timed region, through the same C ABI call.
``roofline`` relates the kernel's median launch time to the measured dense
bf16 tensor peak; ``cpu_baseline`` is the fp64 oracle on the host cores over a
bounded sample of query rows.

``--impl reference`` times the oracle instead (rank 0 only), on the same
workload, over a bounded sample of rows per step.

Multi-GPU (torchrun): by default each rank runs its own independent batch
(seeded by rank: "scaling": "weak"); with ``--scaling strong`` the ranks
share one problem, each computing a contiguous range of its B·H heads
(``head_shards``). Either way no collective touches the data path: heads are
independent.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_attention_91_gb300 import inputs as fin  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "attention fwd TFLOP/s and % of GB300 dense-bf16 peak at 1 GPU"

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the forward
# kernel, from the ncu capture summarised under profiles/ (the file named in
# "source"), valid only while the kernel sources hash to "kernel_sha".
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# the sources that build the forward kernel and its launch
KERNEL_FILES = ("fa_api.cu", "fa_common.cuh", "fa_fwd_kernel.cuh", "ptx.cuh")


def kernel_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_91_gb300", "csrc")
    for name in KERNEL_FILES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def load_traffic(workload: str):
    try:
        with open(TRAFFIC_FILE, encoding="utf-8") as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    ent = t.get(workload)
    if not ent or ent.get("kernel_sha") != kernel_sha():
        return None
    return ent.get("bytes_per_launch")


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json"), encoding="utf-8") as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; samples carry the
    host time they were read at so the timed region can be picked out."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,pci.bus_id")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.bus_id and self.bus_id not in parts[8].lower() and parts[8].lower() not in self.bus_id:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "during timed region"
        if not inside:
            after = [p for (t, p) in self.samples if t > t1][:2]
            before = [p for (t, p) in self.samples if t < t0][-2:]
            inside = before + after
            note = "timed region shorter than the sampling period: nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[4 + i].lower().startswith("active")})
        power = [num(p[2]) for p in inside if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "power_w_max": max(power) if power else None,
                "note": note}


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_workload(w: fin.Workload, rank: int, world: int) -> fin.Workload:
    """Each rank's own batch: the same shape, independently seeded (weak
    scaling: heads are independent, so ranks share nothing)."""
    if world == 1:
        return w
    return fin.Workload(w.name, w.B, w.H, w.N, w.d, w.causal, w.values, w.seed + 1000 * rank)


def local_problem(w: fin.Workload, rank: int, world: int, scaling: str):
    """This rank's inputs (bf16 bits [B_l, H_l, N, d]) and the job's flops per
    step. Weak: the rank's own independently seeded batch of the workload's
    shape; the job does world x the workload's flops. Strong: the rank's
    contiguous range of the one workload's B·H heads (as [1, count, N, d]);
    the job does the workload's flops once."""
    from exact_attention_91_gb300 import head_shards
    if scaling == "weak" or world == 1:
        x = fin.make_inputs(rank_workload(w, rank, world))
        return x, (x.q, x.k, x.v), w.B, w.H, w.flops * world
    x = fin.make_inputs(w)
    BH = w.B * w.H
    start, n = head_shards(BH, world)[rank]
    part = tuple(np.ascontiguousarray(a.reshape(BH, w.N, w.d)[start:start + n][None]) for a in (x.q, x.k, x.v))
    return x, part, 1, n, w.flops


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (every rank must call it)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, flops_step: float, ms_total: float) -> float:
    """Whole-job TFLOP/s: every rank's steps over the slowest rank's time."""
    return world * steps * flops_step / (ms_total * 1e-3) / 1e12


def exp_roofline(w: fin.Workload, launch_s: float, clocks: dict, sm_count: int, heads: int | None = None,
                 ex2_per_clk: float | None = None) -> dict:
    """One ex2 per (query, visible key) of the `heads` heads a launch covers
    (all of the workload's by default) against the MUFU rate: the measured
    ex2 per SM clock (`measure_ex2_rate`) when given, else the nominal 32."""
    heads = w.B * w.H if heads is None else heads
    pairs = heads * (w.N * (w.N + 1) // 2 if w.causal else w.N * w.N)
    mhz = (clocks or {}).get("sm_mhz") or 2070.0
    rate = ex2_per_clk if ex2_per_clk else 32.0
    peak = rate * sm_count * mhz * 1e6
    achieved = pairs / launch_s
    basis = (f"measured {rate:.1f} ex2/clk/SM (fa_selftest_ex2_rate, median over the SMs)" if ex2_per_clk
             else "nominal 32 ex2/clk/SM")
    return {"achieved_per_s": achieved, "peak_per_s": peak, "frac": achieved / peak,
            "exps_per_launch": pairs, "peak_basis": f"{basis} x {sm_count} SMs x {mhz:.0f} MHz"}


def measure_ex2_rate(fa, torch, dev, sm_count: int, iters: int = 2048):
    """Exponentials per SM clock that the exponential unit sustains: one
    block of back-to-back independent ex2.approx chains per SM, each block
    timed in SM clocks by the library's probe; the median over the blocks.
    None if the probe fails."""
    cycles = torch.zeros(sm_count, dtype=torch.int64, device=dev)
    sink = torch.empty(sm_count * fa.EX2_RATE_THREADS, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    for n in (64, iters):  # the first launch warms the code and the clocks
        if fa.fa_selftest_ex2_rate(cycles.data_ptr(), sink.data_ptr(), sm_count, n, s) != 0:
            return None
    torch.cuda.synchronize(dev)
    c = cycles.cpu().numpy().astype(np.float64)
    if not (c > 0).all():
        return None
    return float(np.median(fa.EX2_RATE_THREADS * fa.EX2_RATE_CHAINS * iters / c))


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo", encoding="utf-8") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def row_flops(w: fin.Workload, rows: np.ndarray) -> float:
    """Algorithmic flops of the given flat query rows: 4·d per visible key."""
    if w.causal:
        keys = (rows % w.N) + 1
        return float(4.0 * w.d * keys.sum())
    return float(4.0 * w.d * w.N * len(rows))


class OracleSampler:
    """Times the fp64 oracle on random query rows of a few heads of the
    workload (the heads are widened to fp64 once)."""

    def __init__(self, w: fin.Workload, x: fin.Inputs, seed: int):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.w = w
        self.g = np.random.Generator(np.random.PCG64(seed))
        BH = w.B * w.H
        self.heads = np.unique(self.g.integers(0, BH, size=min(BH, 4)))
        self.q = fin.bf16_to_f64(x.q.reshape(BH, w.N, w.d)[self.heads])[None]
        self.k = fin.bf16_to_f64(x.k.reshape(BH, w.N, w.d)[self.heads])[None]
        self.v = fin.bf16_to_f64(x.v.reshape(BH, w.N, w.d)[self.heads])[None]
        self.n_local = len(self.heads) * w.N
        self.sec_per_flop = None

    def run(self, target_s: float):
        """Random rows timed in batches until about target_s seconds of
        oracle work have been done. Returns (flops, seconds, rows)."""
        w = self.w
        flops = secs = 0.0
        rows_done = 0
        batch = 16
        while secs < target_s and rows_done < 50 * self.n_local:
            rows = self.g.integers(0, self.n_local, size=batch)
            t = time.perf_counter()
            self.oracle.attn_rows(self.q, self.k, self.v, rows, w.scale, w.causal)
            dt = time.perf_counter() - t
            flops += row_flops(w, rows)
            secs += dt
            rows_done += batch
            # next batch sized to about a quarter of what is left
            per_row = dt / batch
            batch = int(max(16, min(self.n_local, 0.25 * (target_s - secs) / max(per_row, 1e-9))))
        return flops, secs, rows_done

    def describe(self, n_rows: int, seconds: float) -> str:
        return (f"{n_rows} random query rows from {len(self.heads)} heads of the {self.w.name} workload "
                f"({seconds:.2f} s of fp64 CPU work); host CPU {cpu_model()}")


# ------------------------------------------------------------------ reference arm

# seconds of oracle work that one `--impl reference` run spends in all
REFERENCE_BUDGET_S = 120.0


def run_reference(args, w: fin.Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    x = fin.make_inputs(w)
    # the whole run (warm-up + timed steps) stays near two minutes of CPU work
    per_step_s = max(0.005, min(20.0, REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)))
    sampler = OracleSampler(w, x, seed=w.seed + 17)
    flops_total = 0.0
    secs_total = 0.0
    rows_total = 0
    for i in range(args.warmup + args.steps):
        f, s_, n = sampler.run(per_step_s)
        if i >= args.warmup:
            flops_total += f
            secs_total += s_
            rows_total += n
    value = flops_total / secs_total / 1e12
    threads = sampler.oracle.host_threads()
    sample = (f"per step about {rows_total / args.steps:.0f} random query rows from "
              f"{len(sampler.heads)} heads of the {w.name} workload (~{per_step_s:.3f} s of fp64 CPU work "
              f"per step); host CPU {cpu_model()}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs_total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w: fin.Workload, world: int, scaling: str = "weak") -> dict:
    ws = 4 * w.B * w.H * w.N * w.d * 2
    if world == 1:
        par = "single GPU"
    elif scaling == "strong":
        par = f"one problem, B*H heads sharded x{world}"
    else:
        par = f"independent batches x{world}"
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "values": w.values, "scale": w.scale, "seed": w.seed, "parallelism": par,
            "l2": ("inputs larger than L2" if ws > 2 * L2_BYTES else "L2 flushed between timed launches")}


# ------------------------------------------------------------------ our arm

def run_ours(args, w: fin.Workload):
    import torch
    import exact_attention_91_gb300 as fa

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", rank=rank, world_size=world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.load_library()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    ex2_rate = measure_ex2_rate(fa, torch, dev, sm_count)

    x, (xq, xk, xv), B, H, job_flops = local_problem(w, rank, world, args.scaling)
    N, d = w.N, w.d

    def up(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v = up(xq), up(xk), up(xv)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    def launch():
        rc = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, H, N, d, w.scale, w.causal, sp)
        if rc != 0:
            raise fa.FaError(rc)

    working_set = 4 * B * H * N * d * 2
    flush = None if working_set > 2 * L2_BYTES else torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}"
    except AttributeError:
        pass
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.3)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 0)):
            launch()
            if flush is not None:
                flush.zero_()
    stream.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t_begin.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
            if flush is not None:
                flush.zero_()
        t_end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier()
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = sum(launch_ms)
    region_ms = t_begin.elapsed_time(t_end)
    # with an L2 flush between launches the flush is not part of the work
    step_total_ms = max_over_ranks(kernel_ms if flush is not None else region_ms, world, dev)
    clocks = sampler.summary(wall0, wall1)
    # small problems: the same launches back to back without the flush (warm L2)
    warm_ms = None
    if flush is not None:
        w0 = torch.cuda.Event(enable_timing=True)
        w1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            w0.record(stream)
            for _ in range(args.steps):
                launch()
            w1.record(stream)
        stream.synchronize()
        warm_ms = w0.elapsed_time(w1) / args.steps

    # ---- end to end: pinned host buffers, copies inside the timed region.
    # Every step copies its inputs host->device and reads its result back.
    # Two device buffer sets let the host->device copy of step i+1 (one
    # stream) and the device->host read of step i (another) overlap the
    # kernel of step i (a third), as a serving loop over this API would.
    hq = torch.from_numpy(xq.view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = torch.from_numpy(xk.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(xv.view(np.int16)).view(torch.bfloat16).pin_memory()
    ho = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(1, min(args.steps, 20))
    sets = [(q, k, v, o, lse),
            tuple(torch.empty_like(t) for t in (q, k, v, o, lse))]
    s_h2d = torch.cuda.Stream(device=dev)
    s_d2h = torch.cuda.Stream(device=dev)

    def e2e_run(n):
        k_done = [torch.cuda.Event() for _ in range(n)]
        d_done = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            bq, bk, bv, bo, bl = sets[i % 2]
            h_done = torch.cuda.Event()
            if i >= 2:
                s_h2d.wait_event(k_done[i - 2])  # kernel i-2 has read this set's inputs
            with torch.cuda.stream(s_h2d):
                bq.copy_(hq, non_blocking=True)
                bk.copy_(hk, non_blocking=True)
                bv.copy_(hv, non_blocking=True)
                h_done.record(s_h2d)
            stream.wait_event(h_done)
            if i >= 2:
                stream.wait_event(d_done[i - 2])  # this set's outputs have been read back
            rc = fa.fa_fwd(bq.data_ptr(), bk.data_ptr(), bv.data_ptr(), bo.data_ptr(), bl.data_ptr(),
                           B, H, N, d, w.scale, w.causal, sp)
            if rc != 0:
                raise fa.FaError(rc)
            k_done[i].record(stream)
            s_d2h.wait_event(k_done[i])
            with torch.cuda.stream(s_d2h):
                ho.copy_(bo, non_blocking=True)
                hl.copy_(bl, non_blocking=True)
                d_done[i].record(s_d2h)
        return d_done[-1]

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_h2d.wait_event(e0)
    last = e2e_run(e2e_steps)
    stream.wait_event(last)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    sampler.stop()

    flops_step = w.flops * B * H / (w.B * w.H)   # this rank's launch
    hbm_local = w.hbm_bytes * B * H // (w.B * w.H)
    value = job_throughput(1, args.steps, job_flops, step_total_ms)
    e2e_value = job_throughput(1, e2e_steps, job_flops, e2e_ms)
    avg_launch_s = kernel_ms / args.steps * 1e-3
    # the roofline uses the median launch (robust to a launch that met a clock
    # change or another process's work); the mean is reported beside it
    median_launch_s = statistics.median(launch_ms) * 1e-3
    achieved = flops_step / median_launch_s / 1e12
    peaks = load_peaks()
    if peaks and peaks.get("bf16_tflops"):
        peak, peak_src = float(peaks["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    else:
        peak, peak_src = FALLBACK_BF16_TFLOPS, "fallback"
    traffic = load_traffic(w.name)

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sampler = OracleSampler(w, x, seed=w.seed + 5)
        f, sec, n_rows = sampler.run(args.cpu_seconds)
        cpu = {"value": f / sec / 1e12, "unit": "TFLOP/s", "cores": sampler.oracle.host_threads(),
               "kind": "oracle", "sample": sampler.describe(n_rows, sec)}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_total_ms / args.steps, "higher_is_better": True,
        "scaling": args.scaling, "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, world, args.scaling),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "kernel": "fa_fwd", "flops_per_launch": flops_step,
                     "median_launch_ms": median_launch_s * 1e3, "avg_launch_ms": avg_launch_s * 1e3,
                     "launches_timed": len(launch_ms)},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                "h2d_bytes_per_step": 3 * B * H * N * d * 2,
                "d2h_bytes_per_step": B * H * N * d * 2 + B * H * N * 4, "steps": e2e_steps,
                "overlap": "two buffer sets: the H2D copy of step i+1 and the D2H read of step i "
                           "overlap the kernel of step i (three streams); host->device runs at "
                           "~211 GB/s (a 1 GB pinned copy on GB300), which bounds this number"},
        "gpu_launches": args.steps,
        "hbm": {"achieved_gbs": hbm_local / median_launch_s / 1e9,
                "peak_gbs": float((peaks or {}).get("hbm_gbs", 6800.0)),
                "frac": hbm_local / median_launch_s / 1e9 / float((peaks or {}).get("hbm_gbs", 6800.0)),
                "bytes_per_launch": hbm_local,
                "note": "compulsory bytes (Q, K, V read, O and LSE written) over the kernel time"},
        "warm_l2_ms_per_step": warm_ms,
        # the second ceiling: one ex2 per (query, visible key) against the
        # measured ex2 rate per SM clock, at the median SM clock of the timed
        # region
        "exp_roofline": exp_roofline(w, median_launch_s, clocks, sm_count, heads=B * H, ex2_per_clk=ex2_rate),
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# Variable-length batches (fa_fwd_varlen), measured apart from the headline:
#   prefill_mix  16 sequences with lengths drawn from U{256..8192} (Nq = Nk),
#                H = 32, d = 128, causal: tensor-bound, TFLOP/s counted like
#                the dense metric (4·H·d·N²/2 per causal sequence)
#   decode       64 sequences of one query against 8192 keys, H = 32,
#                d = 128, causal (the last query sees every key): bound by
#                reading K and V, reported as GB/s of compulsory bytes
#   decode_long  2 sequences of one query against 65536 keys, H = 32,
#                d = 128, causal: 64 (sequence, head) pairs for 152 SMs, so
#                each pair's key range is split and merged; GB/s as decode
VARLEN_MIXES = ("prefill_mix", "decode", "decode_long")


def varlen_batch(name: str):
    g = np.random.Generator(np.random.PCG64(fin.SEED_BASE + 70))
    if name == "prefill_mix":
        n = [int(x) for x in g.integers(256, 8193, size=16)]
        return n, n, 32, 128, True
    if name == "decode_long":
        return [1] * 2, [65536] * 2, 32, 128, True
    return [1] * 64, [8192] * 64, 32, 128, True


def run_varlen(args) -> int:
    import torch
    import exact_attention_91_gb300 as fa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load_library()
    sq, sk, H, d, causal = varlen_batch(args.varlen)
    x = fin.make_varlen_inputs(sq, sk, H, d, seed=fin.SEED_BASE + 71)
    up = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    q, k, v = up(x.q), up(x.k), up(x.v)
    cu_q, cu_k = torch.from_numpy(x.cu_q).to(dev), torch.from_numpy(x.cu_k).to(dev)
    total_q, total_k = q.shape[0], k.shape[0]
    o = torch.empty_like(q)
    lse = torch.empty((H, total_q), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    def launch():
        rc = fa.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              cu_q.data_ptr(), cu_k.data_ptr(), len(sq), H, total_q, total_k, max(sq), d,
                              scale, causal, sp)
        if rc != 0:
            raise fa.FaError(rc, "fa_fwd_varlen")

    bytes_step = (2 * total_q + 2 * total_k) * H * d * 2 + total_q * H * 4
    flops_step = sum(4.0 * H * d * (nq * nk / 2 if causal and nq == nk else
                                    (nq * nk if not causal else sum(min(nk, i + nk - nq + 1) for i in range(nq))))
                     for nq, nk in zip(sq, sk))
    flush = None if bytes_step > 2 * L2_BYTES else torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(None)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 0)):
            launch()
            if flush is not None:
                flush.zero_()
    stream.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    wall0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
            if flush is not None:
                flush.zero_()
    stream.synchronize()
    wall1 = time.time()
    sampler.stop()
    ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)) / args.steps
    peaks = load_peaks() or {}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nsplit = fa.fa_varlen_num_splits(len(sq), H, total_k, max(sq), sms)
    if args.varlen.startswith("decode"):
        value, unit = bytes_step / (ms * 1e-3) / 1e9, "GB/s"
        peak = float(peaks.get("hbm_gbs", 6800.0))
        roof = {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                "traffic": None, "bytes_per_launch": bytes_step}
        metric = "variable-length attention fwd (decode) GB/s of compulsory bytes at 1 GPU"
    else:
        value, unit = flops_step / (ms * 1e-3) / 1e12, "TFLOP/s"
        peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
        roof = {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s", "frac": value / peak,
                "traffic": None, "flops_per_launch": flops_step}
        metric = "variable-length attention fwd TFLOP/s at 1 GPU"
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"varlen_{args.varlen}", "B": len(sq), "H": H, "d": d, "causal": causal,
                   "seqlens_q": sq if len(set(sq)) > 1 else f"{len(sq)} x {sq[0]}",
                   "seqlens_k": sk if len(set(sk)) > 1 else f"{len(sk)} x {sk[0]}",
                   "l2": "inputs larger than L2" if flush is None else "L2 flushed between timed launches",
                   "key_range_splits": nsplit},
        "roofline": roof, "gpu_launches": args.steps, "clocks": sampler.summary(wall0, wall1),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(fin.WORKLOADS), default="llm_prefill")
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d,causal: a custom shape with N(0,1) values instead of a named workload "
                         "(for profiling small cases)")
    ap.add_argument("--varlen", choices=VARLEN_MIXES, default=None,
                    help="measure fa_fwd_varlen on a synthetic variable-length batch instead")
    ap.add_argument("--scaling", choices=["weak", "strong"], default="weak",
                    help="N > 1: weak = every rank its own batch; strong = the ranks share one problem's heads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    w = fin.WORKLOADS[args.workload]
    if args.shape:
        B, H, N, d, causal = (int(x) for x in args.shape.split(","))
        w = fin.custom(B, H, N, d, bool(causal), seed=fin.SEED_BASE + 99)
    if args.varlen:
        return run_varlen(args)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
