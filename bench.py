"""Throughput of the linear-recurrence scan on the pages' shape, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one linrec_scan_f32 call over a (B=32, L=4096, D=256) fp32 batch
(a ~ U[0,1), b ~ N(0,1), seed 1 + 1000*rank).  Inputs (268 MB) and output
(134 MB) together exceed the 129 MB L2, so no flush is needed between steps.
The metric is GB/s of algorithmic traffic, 12 bytes per element (read a and
b, write h once).  Under torchrun each rank scans its own batch (weak scaling,
no collective on the data path); rank 0 prints max-over-ranks timing.

--impl reference times the CPU oracle (plain sequential loop, all host cores)
on the same workload: the reference arm of this comparison.

--dtype bf16 | f16 stores a, b and h in 16 bits (fp32 arithmetic and carry):
6 bytes per element instead of 12, the same GB/s metric over those bytes.

--layout bdl holds the same values time-innermost, (B, D, L), and times the
(B, D, L) entry points on them.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "scan GB/s (a,b,h bytes) & % of GB300 HBM peak at B=32,L=4096,D=256 fp32"
UNIT = "GB/s"
WORKLOAD = "pages"          # the headline workload; --workload picks another for reports


STORAGE_BYTES = {"f32": 4, "bf16": 2, "f16": 2}


def metric_for(w, op: str = "forward", dtype: str = "f32", layout: str = "bld") -> str:
    if op == "backward":
        return (f"scan backward GB/s (a,h,g read, da,db written) & % of GB300 HBM peak at "
                f"B={w.B},L={w.L},D={w.D} fp32 ({w.name})")
    if w.name == WORKLOAD and dtype == "f32" and layout == "bld":
        return METRIC
    store = "fp32" if dtype == "f32" else f"{dtype} storage, fp32 arithmetic"
    lay = "" if layout == "bld" else ", (B,D,L) layout"
    return (f"scan GB/s (a,b,h bytes) & % of GB300 HBM peak at B={w.B},L={w.L},D={w.D} {store}{lay} "
            f"({w.name})")


def bytes_per_step(w, op: str, dtype: str = "f32") -> int:
    # forward: read a, b, write h; backward: read a, h, g, write da, db (each once)
    if op == "backward":
        return 20 * w.numel
    return 3 * STORAGE_BYTES[dtype] * w.numel


def launches_per_step(plan: dict, op: str, inner_plan=None) -> int:
    """Kernel launches of one call.  Speculative mode: two.  Two-pass mode: the reduce launch,
    the scan of the tile aggregates and the apply launch.  That scan is a call of its own on a (1, chunks,
    slices * tile_d) problem (inner_plan: its plan, None for one launch), which may itself
    take two-pass mode (three launches); the scan of its maps never does."""
    if plan["path_name"] == "chunked" and plan["twopass"]:
        return 2 + (launches_per_step(inner_plan, "forward") if inner_plan is not None else 1)
    if plan["path_name"] == "chunked" and plan.get("speculative"):
        return 2                              # speculative launch and repair launch
    if plan["path_name"] == "rows" and plan["twopass"]:
        return 3
    if plan["path_name"] == "regcarry" and plan["twopass"]:
        return 2                              # segmented register path: reduce and apply
    return 1
FALLBACK_HBM_GBS = 6800.0
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ---------------------------------------------------------------------------
# rank bookkeeping (host only; tested on CPU with gloo)
# ---------------------------------------------------------------------------

def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment, (0, 1, 0) without it."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank scans its own batch; rank 0's batch is the named workload itself."""
    return base_seed + 1000 * rank


def max_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank_step: int, world: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: the bytes every rank moved over the slowest rank's time."""
    return bytes_per_rank_step * world * steps / seconds / 1e9


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of one GPU's clocks, power and throttle reasons every period_ms.
    start() before the warm-up and wait_first() until the first sample is written, so that
    the warm-up runs straight into the timed region with no idle gap; stop() after it."""

    def __init__(self, index: int, period_ms: int = 20):
        self.index, self.period_ms = index, period_ms
        self.proc = None
        self.path = None
        self.fh = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period_ms)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def wait_first(self, timeout_s: float = 2.0):
        """Block until nvidia-smi has written its first sample (or timeout_s has passed)."""
        if self.proc is None:
            return
        t_end = time.perf_counter() + timeout_s
        while time.perf_counter() < t_end and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.01)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        window = (f"nvidia-smi every {self.period_ms} ms from before the warm-up to the end of the timed "
                  "region (the warm-up runs straight into the timed region)")
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(float(r[1]) for r in rows),
                "sm_max_mhz": max(float(r[2]) for r in rows),
                "power_w_max": max(power) if power else None,
                "reasons": reasons, "samples": len(rows), "window": window}


# ---------------------------------------------------------------------------
# measured peaks and committed counters
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest(names) -> str:
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "linear_recurrence_scan_fp32_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_capture(kernel: str, workload: str):
    """The committed ncu summary of the kernel on the workload: (dram read+write bytes per launch,
    whether the digest of its kernel sources still matches the tree, the file), or None."""
    rel = os.path.join("profiles", f"traffic_{kernel}_{workload}.txt")
    try:
        kv = {}
        with open(os.path.join(ROOT, rel)) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        src = kv["kernel_sources"].split(",")
        same = kernel_source_digest([s.strip() for s in src]) == kv["kernel_source_sha256_16"]
        return int(kv["dram_bytes_per_launch"]), same, rel
    except (OSError, KeyError, ValueError):
        return None


def committed_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    cap = committed_capture(kernel, workload)
    return cap[0] if cap and cap[1] else None


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

class OracleTimer:
    """Repeated calls of one form of the oracle over fixed inputs, writing into one output array
    allocated up front, so that repetitions time the scan rather than the page faults of a fresh
    output.  The bench line's cpu_baseline leg and the reference arm both time the oracle
    through this class.  form: "f64" (the definition in double precision) or "f32seq" (the
    fp32 twin); 16-bit storage: the oracle's decode of the words, then its fp64 scan."""

    def __init__(self, a, b, dtype: str = "f32", form: str = "f64", nthreads: int = 0):
        import oracle
        oracle.build()
        self.oracle, self.dtype, self.form, self.nthreads = oracle, dtype, form, nthreads
        self.a, self.b = a, b
        self.used = nthreads
        self.out = None
        if dtype == "f32":
            self.out = np.empty(np.shape(a), dtype=np.float64 if form == "f64" else np.float32)

    def __call__(self):
        o = self.oracle
        if self.dtype != "f32":
            h, _ = o.f64_16(self.dtype, self.a, self.b, nthreads=self.nthreads)
            return h
        fn = o.f64 if self.form == "f64" else o.f32seq
        h, self.used = fn(self.a, self.b, nthreads=self.nthreads, out=self.out)
        return h

    def repeat(self, budget_s: float, min_reps: int = 1):
        """Call until budget_s seconds of calls (at least min_reps); returns (reps, seconds, last h)."""
        reps, t_total, h = 0, 0.0, None
        while (t_total < budget_s or reps < min_reps) and reps < 100000:
            t0 = time.perf_counter()
            h = self()
            t_total += time.perf_counter() - t0
            reps += 1
        return reps, t_total, h


def _rate(nbytes: int, numel: int, reps: int, seconds: float, cores: int) -> dict:
    return {"value": round(nbytes * reps / seconds / 1e9, 3), "unit": UNIT, "cores": cores,
            "elements_per_s": round(numel * reps / seconds, 1), "ms_per_workload": round(1e3 * seconds / reps, 3),
            "repetitions": reps}


def cpu_baseline(a, b, w, budget_s: float = 10.0, dtype: str = "f32", h_gpu=None, layout: str = "bld"):
    """The oracle as it stands on the host cores: the reference arm itself (--impl reference, the
    fp64 definition on all cores, plus --extra-forms: one core, and the fp32 twin on all cores), run
    as a child process that does not use the GPU, on a budget of about budget_s seconds.  So the
    bench line and the reference arm report one measurement method.  Returns (baseline, parity):
    parity compares h_gpu, the output of the timed GPU run, with the fp64 oracle's result (computed
    here, untimed), element by element."""
    import oracle
    oracle.build()
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "LOCAL_WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", w.name,
           "--dtype", dtype, "--layout", layout, "--steps", "5", "--warmup", "3", "--ref-seconds", str(budget_s),
           "--extra-forms"]
    base = None
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=30 + 10 * budget_s)
        for line in out.stdout.splitlines():
            if line.startswith("{"):
                base = json.loads(line)["cpu_baseline"]
                base["method"] = ("the reference arm (bench.py --impl reference --extra-forms --steps 5 --warmup 3 "
                                  f"--ref-seconds {budget_s:g}) in a child process that does not use the GPU")
    except (OSError, subprocess.TimeoutExpired, ValueError, KeyError):
        base = None
    parity = None
    if h_gpu is not None:
        h64 = OracleTimer(a, b, dtype, "f64", oracle.hardware_threads())()
        # 16-bit storage: the output words, decoded by the oracle's own definition of the format
        got = np.asarray(h_gpu, dtype=np.float64) if dtype == "f32" else oracle.decode16(dtype, h_gpu)
        err = np.abs(got - h64)
        u = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}[dtype]
        bound = u * np.abs(h64) + (1 + u) * 1e-4 * (1 + np.abs(h64))
        parity = {"vs": "fp64 oracle, every element of the timed run's output",
                  "max_abs_err": float(err.max()), "max_rel_err": float((err / (1 + np.abs(h64))).max()),
                  "bound": "u*|h64| + (1+u)*1e-4*(1+|h64|), u = 0 (fp32), 2^-8 (bf16), 2^-11 (f16)",
                  "within_bound": bool((err <= bound).all())}
    return base, parity


def cpu_baseline_backward(a, h, g, w, nbytes, budget_s: float = 10.0):
    """The oracle's reverse loop (single thread: it has no threaded form), for ~budget_s."""
    import oracle
    oracle.build()
    reps, t_total = 0, 0.0
    while t_total < budget_s and reps < 100000:
        t0 = time.perf_counter()
        oracle.f64_backward(a, h, g)
        t_total += time.perf_counter() - t0
        reps += 1
    return {"value": nbytes * reps / t_total / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"full {w.name} workload {w.shape}, fp64 reverse loop, {reps} repetitions, {t_total:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from linear_recurrence_scan_fp32_gb300 import inputs
    import oracle
    oracle.build()
    w = inputs.WORKLOADS[args.workload]
    a, b = inputs.generate_workload(w)
    if args.dtype != "f32":
        a, b = inputs.to_storage16(a, args.dtype), inputs.to_storage16(b, args.dtype)
        a = a.view(__import__("torch").int16).numpy().view(np.uint16)
        b = b.view(__import__("torch").int16).numpy().view(np.uint16)
    else:
        a, b = a.numpy(), b.numpy()
    threads = oracle.hardware_threads()
    # size each step's sample so that warm-up + timed steps take about --ref-seconds
    t0 = time.perf_counter()
    OracleTimer(a, b, args.dtype, "f64", threads)()
    t_full = time.perf_counter() - t0
    per_step = args.ref_seconds / (args.steps + args.warmup)
    nb = max(1, min(w.B, int(w.B * per_step / t_full)))
    nl = w.L if nb > 1 else max(64, min(w.L, int(w.L * w.B * per_step / t_full)))
    a_s = np.ascontiguousarray(a[:nb, :nl])
    b_s = np.ascontiguousarray(b[:nb, :nl])
    timer = OracleTimer(a_s, b_s, args.dtype, "f64", threads)   # the cpu_baseline leg's timer
    # a sample shorter than a step's share of the budget is scanned several times per step, so that
    # the arm times sustained host throughput, as the bench line's cpu_baseline leg does
    t0 = time.perf_counter()
    timer()
    t_sample = time.perf_counter() - t0
    reps = max(1, int(per_step / max(t_sample, 1e-6)))
    sample_bytes = 3 * STORAGE_BYTES[args.dtype] * a_s.size * reps
    for _ in range(args.warmup):
        for _ in range(reps):
            timer()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for _ in range(reps):
            timer()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    used = timer.used
    value = sample_bytes * args.steps / total / 1e9
    elems = a_s.size * reps * args.steps
    extra = {}
    if args.extra_forms and args.dtype == "f32":
        # the other forms of the oracle on the same sample: the fp64 definition on one core and the
        # fp32 twin on all cores, each for a third of the budget
        for key, form, nthreads in (("fp64_1core", "f64", 1), ("f32seq_all_cores", "f32seq", threads)):
            t = OracleTimer(a_s, b_s, args.dtype, form, nthreads)
            r, secs, _ = t.repeat(args.ref_seconds / 3)
            extra[key] = _rate(3 * STORAGE_BYTES[args.dtype] * a_s.size, a_s.size, r, secs, t.used)
    line = {
        "impl": "reference", "metric": metric_for(w, "forward", args.dtype, args.layout), "value": round(value, 3), "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "gpu_launches": 0,
        "config": {"workload": w.about, "B": w.B, "L": w.L, "D": w.D, "seed": w.seed, "storage": args.dtype,
                   "l2": "host run: no device cache involved"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": used, "kind": "oracle",
                         "elements_per_s": round(elems / total, 1),
                         "ms_per_workload": round(1e3 * total / (reps * args.steps) * (w.numel / a_s.size), 3),
                         "sample": f"per step: {reps} scan(s) of batches 0..{nb - 1}, steps 0..{nl - 1}, all "
                                   f"{w.D} channels of the {w.name} workload {w.shape} ({a_s.size} elements), "
                                   "output allocated once, in a process that does not use the GPU",
                         **extra},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def side_measurements(args, lr, inputs, dev, stream, step, peak, a_pages, b_pages):
    """Secondary figures from the same run, outside the timed region (rank 0 on one GPU, the
    default workload only): the headline call with L2 flushed before every call; the other four
    fp32 workloads through linrec_scan_f32 (the dispatcher's choice); the headline shape in
    bfloat16 and binary16 storage.  Each: 3 warm-up calls, then K = min(steps, 20) calls between
    two events (the flushed figure: one event pair around each call, the flush outside it)."""
    import torch
    k = max(3, min(args.steps, 20))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def region(fn):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if lr.linrec_stream_status(stream) != lr.LINREC_OK:
            raise SystemExit("device-side failure in a side measurement")
        return e0.elapsed_time(e1) / 1e3 / k

    def entry(sec, nbytes, **extra):
        gbs = nbytes / sec / 1e9
        return {"value": round(gbs, 1), "unit": UNIT, "ms_per_step": round(sec * 1e3, 5),
                "frac_of_peak": round(gbs / peak, 4), "steps": k, **extra}

    out = {}
    w = inputs.WORKLOADS[WORKLOAD]
    # 1. the headline call with a cold L2: 256 MB (twice the L2) written before each call
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    evs = []
    with torch.cuda.stream(stream):
        for i in range(3 + k):
            flush.fill_(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            evs.append((e0, e1))
    torch.cuda.synchronize()
    sec = sum(e0.elapsed_time(e1) for e0, e1 in evs[3:]) / 1e3 / k
    out["pages_l2_flushed"] = entry(sec, bytes_per_step(w, "forward"),
                                    flush="256 MB written before every call; one event pair around each call")
    del flush, evs
    # 2. the other fp32 workloads
    for name in ("tiny", "long", "gated", "short"):
        v = inputs.WORKLOADS[name]
        a_c, b_c = inputs.generate(v.B, v.L, v.D, v.seed, v.a_dist, v.b_dist)
        a, b = a_c.to(dev), b_c.to(dev)
        h = torch.empty_like(a)
        plan = lr.linrec_plan_f32(v.B, v.L, v.D, sm_count=sms)
        how = plan["path_name"] + (" two-pass" if plan["twopass"] else " chain" if plan.get("chain") else
                                   " speculative" if plan.get("speculative") else "")
        sec = region(lambda: lr.linrec_scan_f32(a, b, h, stream=stream))
        out[name] = entry(sec, bytes_per_step(v, "forward"), shape=[v.B, v.L, v.D], path=how)
        del a, b, h, a_c, b_c
    # 3. the headline shape in 16-bit storage
    for dt, fn in (("bf16", lr.linrec_scan_bf16), ("f16", lr.linrec_scan_f16)):
        a16 = inputs.to_storage16(a_pages, dt).to(dev)
        b16 = inputs.to_storage16(b_pages, dt).to(dev)
        h16 = torch.empty_like(a16)
        sec = region(lambda: fn(a16, b16, h16, stream=stream))
        out["pages_" + dt] = entry(sec, bytes_per_step(w, "forward", dt), shape=[w.B, w.L, w.D], storage=dt)
        del a16, b16, h16
    out["note"] = ("outside the timed region; clocks not sampled; K = min(steps, 20) calls after 3 warm-up "
                   "calls, L2 not flushed except in pages_l2_flushed")
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import linear_recurrence_scan_fp32_gb300 as lr
    from linear_recurrence_scan_fp32_gb300 import _build, inputs

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev) if "device_id" in dist.init_process_group.__code__.co_varnames \
            else dist.init_process_group("nccl")
    _build.build()
    lr.lib()

    w = inputs.WORKLOADS[args.workload]
    a_cpu, b_cpu = inputs.generate(w.B, w.L, w.D, rank_seed(w.seed, rank), w.a_dist, w.b_dist)
    if args.dtype != "f32":
        if args.op != "forward":
            raise SystemExit("16-bit storage is forward only")
        a_cpu, b_cpu = inputs.to_storage16(a_cpu, args.dtype), inputs.to_storage16(b_cpu, args.dtype)
    bdl = args.layout == "bdl"
    if bdl:
        if args.op != "forward":
            raise SystemExit("the (B, D, L) layout is timed forward only")
        a_cpu = a_cpu.transpose(1, 2).contiguous()
        b_cpu = b_cpu.transpose(1, 2).contiguous()
    a = a_cpu.to(dev)
    b = b_cpu.to(dev)
    h = torch.empty_like(a)
    stream = torch.cuda.current_stream(dev)
    opt = {} if args.path == "auto" else {"path": args.path}
    if args.chunk_mode != "auto":
        opt.update(path="chunked", chunk_mode=args.chunk_mode)
    if args.tile:
        td, tt, st = (int(x) for x in args.tile.split(","))
        opt.update(path="chunked", tile_d=td, tile_t=tt, stages=st)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    store = "" if args.dtype == "f32" else "_" + args.dtype
    if bdl:
        if args.tile or args.path not in ("auto", "rows"):
            raise SystemExit("the (B, D, L) layout takes --chunk-mode own | twopass only")
        opt = {} if args.chunk_mode == "auto" else {"chunk_mode": args.chunk_mode}
        plan = lr.linrec_plan_bdl(w.B, w.D, w.L, elem_bytes=STORAGE_BYTES[args.dtype], sm_count=sms, **opt)
        kernel_tag = "rows" + store + ("_twopass" if plan["twopass"] else "")
        scan16 = {"f32": lr.linrec_scan_f32_bdl_ex, "bf16": lr.linrec_scan_bf16_bdl_ex,
                  "f16": lr.linrec_scan_f16_bdl_ex}[args.dtype]
    else:
        plan_fn = lr.linrec_plan_f32 if args.dtype == "f32" else lr.linrec_plan_16
        plan = plan_fn(w.B, w.L, w.D, sm_count=sms, **opt)
        if plan["path_name"] == "chunked":
            mode = ("_twopass" if plan["twopass"] else "_blocks" if plan.get("blocks") else
                    "_chain" if plan.get("chain") else "_speculative" if plan.get("speculative") else
                    "_lookback" if plan["lookback"] else "")
            kernel_tag = "chunked" + store + mode
        else:
            kernel_tag = "regcarry" + store + ("_segmented" if plan["twopass"] else "")
        scan16 = {"bf16": lr.linrec_scan_bf16_ex, "f16": lr.linrec_scan_f16_ex}.get(args.dtype)

    if args.op == "backward":
        lr.linrec_scan_f32(a, b, h, stream=stream)          # the forward output the gradient needs
        g_cpu = inputs.generate(w.B, w.L, w.D, rank_seed(w.seed, rank) + 7, "u[0,1)", "n(0,1)")[1]
        gd = g_cpu.to(dev)
        da = torch.empty_like(a)
        db = torch.empty_like(a)
        plan = lr.linrec_plan_f32_backward(w.B, w.L, w.D,
                                           sm_count=torch.cuda.get_device_properties(dev).multi_processor_count,
                                           **opt)
        kernel_tag = ("backward_twopass" if plan["twopass"] else "backward_lookback" if plan["lookback"]
                      else "backward") if plan["path_name"] == "chunked" else "regcarry_backward"

    def step():
        if args.op == "backward":
            lr.linrec_scan_f32_backward(a, h, gd, da=da, db=db, stream=stream, **opt)
        elif bdl and not opt and args.dtype == "f32":
            lr.linrec_scan_f32_bdl(a, b, h, stream=stream)
        elif scan16 is not None:
            scan16(a, b, h, stream=stream, **opt)
        elif opt:
            lr.linrec_scan_f32_ex(a, b, h, stream=stream, **opt)
        else:
            lr.linrec_scan_f32(a, b, h, stream=stream)

    # The clock sampler starts first; once it has written a sample the W warm-up calls run
    # straight into the timed region (a pause between them measured 2-3 us per call slower
    # at K = 20 on the pages shape), with only the synchronisation and barrier between.
    clocks = ClockSampler(local).start()
    clocks.wait_first()
    for _ in range(args.warmup):
        step()
    # Two events around the K steps, nothing between them: the chunked kernels are
    # launched as programmatic dependents, so a call may be scheduled while the one
    # before it drains (it waits for it before touching memory); an event recorded
    # between two launches would cut that overlap.
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
        torch.cuda.synchronize()
    t0 = time.perf_counter()
    e_start.record(stream)
    for i in range(args.steps):
        step()
    e_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    clocks.stop()
    elapsed_ms = e_start.elapsed_time(e_end)
    status = lr.linrec_stream_status(stream)          # covers the warm-up and the timed calls
    if status != lr.LINREC_OK:
        raise SystemExit(f"device-side failure: {lr.linrec_status_string(status)}")
    seconds = max_over_ranks(elapsed_ms / 1e3, dev)
    nbytes = bytes_per_step(w, args.op, args.dtype)
    value = aggregate_gbs(nbytes, world, args.steps, seconds)
    inner_plan = None
    if plan["path_name"] == "chunked" and plan["twopass"]:
        width = w.B * -(-w.D // plan["tile_d"]) * plan["tile_d"]
        inner_plan = lr.linrec_plan_f32(1, plan["chunks"], width, sm_count=sms)
    launches = launches_per_step(plan, args.op, inner_plan)

    # roofline of the scan: the kernel is the only work in the timed region, so its mean
    # duration per call (one launch, or the two-pass and speculative modes' several) is the
    # region over K
    mean_launch_s = elapsed_ms / 1e3 / args.steps
    achieved = nbytes / mean_launch_s / 1e9
    peak, peak_kind = hbm_peak()
    kernel = kernel_tag
    traffic = committed_traffic(kernel, w.name)
    capture = committed_capture(kernel, w.name)

    # in-run copy ceiling over the same byte count: 1.5*N floats read and written
    n_copy = nbytes // 8
    src = torch.empty(n_copy, device=dev).uniform_()
    dst = torch.empty_like(src)
    copy_gbs = {}
    for name, fn in (("copy_kernel", lambda: lr.linrec_copy_f32(src, dst, stream=stream)),
                     ("cudaMemcpy_d2d", lambda: dst.copy_(src))):
        for _ in range(5):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 50
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        copy_gbs[name] = round(8 * n_copy * reps / (e0.elapsed_time(e1) / 1e3) / 1e9, 1)
    del src, dst
    ceiling = max(copy_gbs.values())

    side = None
    if (rank == 0 and world == 1 and not args.no_side and args.workload == WORKLOAD and args.dtype == "f32"
            and args.op == "forward" and not bdl and not opt):
        side = side_measurements(args, lr, inputs, dev, stream, step, peak, a_cpu, b_cpu)

    # the CPU oracle first, before the e2e leg pins host memory
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if args.op == "backward":
            cpu = cpu_baseline_backward(a_cpu.numpy(), h.cpu().numpy(), g_cpu.numpy(), w, nbytes,
                                        budget_s=args.cpu_seconds)
        else:
            # the oracle scans (B, L, D); the (B, D, L) values are the same numbers transposed
            ca, cb = (a_cpu.transpose(1, 2).contiguous(), b_cpu.transpose(1, 2).contiguous()) if bdl \
                else (a_cpu, b_cpu)
            hc = h.cpu()
            if bdl:
                hc = hc.transpose(1, 2).contiguous()
            if args.dtype == "f32":
                cpu, parity = cpu_baseline(ca.numpy(), cb.numpy(), w, budget_s=args.cpu_seconds, h_gpu=hc.numpy(),
                                           layout=args.layout)
            else:
                words = hc.view(torch.int16).numpy().view(np.uint16)
                cpu, parity = cpu_baseline(ca, cb, w, budget_s=args.cpu_seconds, dtype=args.dtype, h_gpu=words,
                                           layout=args.layout)

    # end to end through the public API: pinned host inputs in, result out, every step
    e2e = None
    if not args.no_e2e and args.op == "forward":
        a_h = a_cpu.pin_memory()
        b_h = b_cpu.pin_memory()
        h_h = torch.empty_like(a_cpu).pin_memory()
        e_steps = max(3, min(args.steps, 20))

        if scan16 is None and not bdl:
            def e2e_step():
                lr.linrec_scan_f32_host(a_h, b_h, h_h, stream=stream)
            e2e_path = ("linrec_scan_f32_host on pinned host a, b, h: the kernel reads and writes host "
                        "memory in place over the host link")
        else:
            def e2e_step():
                a.copy_(a_h, non_blocking=True)
                b.copy_(b_h, non_blocking=True)
                scan16(a, b, h, stream=stream)
                h_h.copy_(h, non_blocking=True)
            e2e_path = (f"pinned host a, b copied in, linrec_scan_{args.dtype}{'_bdl' if bdl else ''}_ex, "
                        "h copied out, one stream")

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
        eb = STORAGE_BYTES[args.dtype]
        e2e = {"value": round(aggregate_gbs(nbytes, world, e_steps, e_sec), 3), "unit": UNIT,
               "h2d_bytes_per_step": 2 * eb * w.numel, "d2h_bytes_per_step": eb * w.numel, "steps": e_steps,
               "path": e2e_path}

    if rank == 0:
        clk = clocks.summary()
        line = {
            "metric": metric_for(w, args.op, args.dtype, args.layout), "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(seconds * 1e3 / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.about, "B": w.B, "L": w.L, "D": w.D, "seed": w.seed,
                       "global_batch": w.B * world,
                       "op": args.op, "storage": args.dtype, "layout": "(B,D,L)" if bdl else "(B,L,D)",
                       "l2": (f"inputs larger than L2: {nbytes / 1e6:.0f} MB per step vs 129 MB L2, "
                              "no flush") if nbytes > 129e6 else "working set fits L2: small case",
                       "path": plan["path_name"],
                       "plan": {k: plan.get(k, 0) for k in ("vec", "prefetch", "tile_t", "tile_d", "segments",
                                                            "stages", "lookback", "twopass", "blocks", "chain",
                                                            "speculative",
                                                            "threads", "grid")}},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "traffic_earlier_sources": ({"bytes": capture[0], "file": capture[2],
                                                      "note": "captured on an earlier digest of the kernel "
                                                              "sources; not the current kernel's"}
                                                     if capture and not capture[1] else None),
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s", "kernel": kernel,
                         "algorithmic_bytes_per_step": nbytes, "launches_per_step": launches,
                         "timed": "two events around the K back-to-back calls (every launch of each "
                                  "call); mean per call = region / K"},
            "copy_ceiling_gbs": copy_gbs,
            "frac_of_copy_ceiling": round(value / ceiling, 4),
            "cpu_baseline": cpu,
            "parity": parity,
            "e2e": e2e,
            "side": side,
            "gpu_launches": args.steps * launches,
            "clocks": clk,
            "wall_s": round(wall, 3),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=100)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--path", choices=("auto", "regcarry", "chunked"), default="auto")
    p.add_argument("--workload", default=WORKLOAD,
                   help="named workload (tiny, pages, long, gated, short, ...); pages is the headline")
    p.add_argument("--chunk-mode", choices=("auto", "own", "lookback", "twopass", "blocks", "chain", "speculative"),
                   default="auto")
    p.add_argument("--dtype", choices=("f32", "bf16", "f16"), default="f32",
                   help="storage of a, b and h (arithmetic is fp32 for all three)")
    p.add_argument("--layout", choices=("bld", "bdl"), default="bld",
                   help="bld: (B, L, D), channels innermost (the pages'); bdl: (B, D, L), time innermost")
    p.add_argument("--tile", default="", help="chunked tile as tile_d,tile_t,stages")
    p.add_argument("--op", choices=("forward", "backward"), default="forward",
                   help="forward scan (the headline) or its gradient")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-side", action="store_true",
                   help="skip the side figures (cold L2, the other workloads, 16-bit storage)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--ref-seconds", type=float, default=30.0,
                   help="reference arm: CPU time budget for warm-up + timed steps")
    p.add_argument("--extra-forms", action="store_true",
                   help="reference arm: also time the fp64 oracle on one core and the fp32 twin on all cores")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
