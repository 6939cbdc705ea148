#!/usr/bin/env python3
"""Benchmark of the quantized-weight matmul on GB300.

Default workload (one JSON line on stdout): int4 decode GEMV on the
attention-projection shape O=12288, I=6144, S=1.  One step = one token through
R resident copies of that [12288, 6144] int4 tensor (R * 37.9 MB > 3x the L2,
so every step streams its weights from HBM).  value = algorithmic bytes
(codes + scales + x + y) of all R calls / device time.  The line also carries
the W4A16 prefill throughput (O=12288, I=6144, S=1571, TFLOP/s), the roofline
of the dominant kernel, an end-to-end number through the host-buffer C-ABI
call, the clocks seen during the timed region, and the CPU oracle timed on
the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --workload sweep        # every config, one JSON line each

--impl reference times the CPU oracle (the only reference implementation of
this method that exists here) on the same workload and metric.
Multi-GPU: one process per GPU (torchrun); each rank runs its own replica of
the workload (the path does not shard across GPUs here: replicas only);
value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quant-matmul weight GB/s (% HBM peak) at S=1; W4A16 TFLOP/s at S=1571"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
L2_BYTES = 129 * 2 ** 20

I4 = 2


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def algorithmic_bytes(fmt_bits, O, I, S):
    """Codes + scales + x + y of one matmul call (row padding excluded)."""
    return O * ((I * fmt_bits + 7) // 8) + 4 * O + 4 * S * I + 4 * S * O


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch recorded from an ncu capture for this kernel,
    valid only while the kernel's sources hash to the recorded digest."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    for ln in lines:
        if not ln.strip() or ln.startswith("#"):
            continue
        kv = dict(p.split("=", 1) for p in ln.split() if "=" in p)
        if kv.get("key") != kernel_key:
            continue
        files = kv.get("sources", "").split(",")
        try:
            if source_digest(files) != kv.get("digest"):
                return None
        except OSError:
            return None
        return float(kv["bytes_per_launch"])
    return None


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for ln in open(self.path).read().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hwt": parts[6], "swt": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows),
                "power_w_max": max(r["power"] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- distributed

def dist_init(n_gpus):
    """One process per GPU (torchrun env); NCCL when GPUs are present, gloo
    otherwise.  The workload is replicated: no data crosses ranks, only the
    barrier and the max of the timings."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """Max of a host float over all ranks (NCCL on GPUs, gloo on the CPU)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step, steps, world, ms_max):
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return bytes_per_rank_step * steps * world / (ms_max * 1e-3) / 1e9


# ----------------------------------------------------------------------------- workloads

class Decode:
    """R distinct resident [O, I] tensors, S tokens: one step = R matmul calls."""

    def __init__(self, q, fmt, O, I, S, R, seed=0, gs=0, path=None):
        import torch
        import synth
        self.q, self.fmt, self.O, self.I, self.S, self.R = q, fmt, O, I, S, R
        self.path = path                # None: b200q_matmul (AUTO); else b200q_matmul_ex with this path
        self.tensors = []
        lo, hi = {0: (1e-3, 2e-2), 1: (1e-3, 1e-2), 2: (5e-3, 2e-2), 3: (1e-3, 2e-2)}[fmt]
        for r in range(R):
            codes, scales = synth.quant_tensor(fmt, O, I, seed, 1 + r, lo, hi)
            if gs:                      # group-wise scales, [O, ceil(I / gs)]
                scales = synth.uniform_f32((O, -(-I // gs)), lo, hi, seed, 500 + r)
            self.tensors.append(q.tensor_upload(fmt, O, I, codes, scales, gs=gs))
        x = synth.activations(S, I, seed, 9999)
        self.x = torch.from_numpy(x).cuda()
        self.y = torch.empty((R, S, O), dtype=torch.float32, device="cuda")
        bits = {0: 32, 1: 8, 2: 4, 3: 2}[fmt]
        self.bytes_per_call = algorithmic_bytes(bits, O, I, S) + (4 * O * (-(-I // gs) - 1) if gs else 0)
        self.bytes_per_step = self.bytes_per_call * R
        self.flops_per_step = 2.0 * O * I * S * R
        self.launches_per_step = None

    def step(self, stream):
        for r in range(self.R):
            if self.path is None:
                self.q.matmul(self.tensors[r], self.x, self.y[r], self.S, stream)
            else:
                self.q.matmul_ex(self.tensors[r], self.x, self.y[r], self.S, self.path, stream)

    def close(self):
        for t in self.tensors:
            t.free()


def time_steps(wl, steps, warmup, stream, world=1, graph=True):
    """Device time of `steps` steps on `stream` (CUDA events on that stream).
    With graph=True one step (all its library calls) is captured once into a
    CUDA graph and replayed, which is how a decode loop runs: the host's
    per-call launch cost stays out of the timed region.  Returns (ms, our
    kernel launches inside the timed region)."""
    import torch
    q = wl.q
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            wl.step(stream)
    torch.cuda.synchronize()
    g = None
    per_step = None
    if graph:
        g = torch.cuda.CUDAGraph()
        n0 = q.kernel_launches()
        with torch.cuda.graph(g, stream=stream):
            wl.step(stream)
        per_step = q.kernel_launches() - n0
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    n0 = q.kernel_launches()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            if g is not None:
                g.replay()
            else:
                wl.step(stream)
        e1.record(stream)
    launches = q.kernel_launches() - n0 if g is None else per_step * steps
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return ms, launches


def time_e2e_step(wl, steps, warmup):
    """The decode step end to end through the public API: every step copies
    the token's x from pinned host memory to the device, runs the R
    b200q_matmul calls on device buffers, copies all R outputs back to pinned
    host memory and synchronizes the stream.  Host wall clock."""
    import torch
    q = wl.q
    xh = torch.from_numpy(wl.x.cpu().numpy()).pin_memory()
    yh = torch.empty((wl.R, wl.S, wl.O), dtype=torch.float32).pin_memory()
    xd = torch.empty_like(wl.x)
    st = torch.cuda.current_stream()

    def step():
        xd.copy_(xh, non_blocking=True)
        for r in range(wl.R):
            q.matmul(wl.tensors[r], xd, wl.y[r], wl.S, st)
        yh.copy_(wl.y, non_blocking=True)
        st.synchronize()

    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    t1 = time.perf_counter()
    return (t1 - t0) * 1e3, wl.S * wl.I * 4, wl.R * wl.S * wl.O * 4


def time_e2e(wl, steps, warmup):
    """Same decode step through b200q_matmul_host: pinned host x in, host y out,
    copies and a stream sync inside every call."""
    import torch
    q = wl.q
    xh = torch.from_numpy(wl.x.cpu().numpy()).pin_memory()
    yh = torch.empty((wl.R, wl.S, wl.O), dtype=torch.float32).pin_memory()
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        for r in range(wl.R):
            q.matmul_host(wl.tensors[r], xh, yh[r], wl.S, st)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        for r in range(wl.R):
            q.matmul_host(wl.tensors[r], xh, yh[r], wl.S, st)
    t1 = time.perf_counter()
    h2d = wl.R * wl.S * wl.I * 4
    d2h = wl.R * wl.S * wl.O * 4
    return (t1 - t0) * 1e3, h2d, d2h


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def time_oracle(fn, seconds, min_calls=1):
    """Calls fn() until `seconds` of wall time (and at least min_calls calls)
    have passed, after one untimed warm call; returns (calls, seconds)."""
    fn()
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds and n >= min_calls:
            return n, dt


def cpu_baseline_decode(O, I, S, fmt=I4, seconds=3.0, seconds_1=2.0):
    """The oracle as it stands on the host cores, on the full decode workload
    repeated until `seconds` have passed: on all cores, then on one core."""
    import oracle
    import synth
    lo, hi = (5e-3, 2e-2)
    codes, scales = synth.quant_tensor(fmt, O, I, 0, 1, lo, hi)
    x = synth.activations(S, I, 0, 9999)
    bits = {0: 32, 1: 8, 2: 4, 3: 2}[fmt]
    per = algorithmic_bytes(bits, O, I, S)
    oracle.set_threads(0)
    cores = oracle.max_threads()
    n, dt = time_oracle(lambda: oracle.matmul(fmt, O, I, codes, scales, x), seconds)
    oracle.set_threads(1)
    n1, dt1 = time_oracle(lambda: oracle.matmul(fmt, O, I, codes, scales, x), seconds_1)
    oracle.set_threads(0)
    return {"value": round(per * n / dt / 1e9, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": "full O=%d I=%d S=%d int4 matmul, %d calls in %.1f s" % (O, I, S, n, dt),
            "cores_1": {"value": round(per * n1 / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                        "sample": "the same call on one core, %d calls in %.1f s" % (n1, dt1)}}


def run_cpu_plan(args):
    """The oracle timed on every workload on the host cores (one JSON line
    each): configs 1, 2 and 4 at S=1 on all cores and on one core, config 2
    at S=4, the MoE expert layer and the W4A16 prefill call on all cores."""
    import oracle
    import synth
    model = cpu_model()
    oracle.set_threads(0)
    cores = oracle.max_threads()

    def emit(name, per_call_bytes, flops, fn, threads, seconds):
        oracle.set_threads(threads)
        n, dt = time_oracle(fn, seconds)
        oracle.set_threads(0)
        ms = dt * 1e3 / n
        line = {"workload": name, "impl": "oracle", "cores": cores if threads == 0 else threads,
                "cpu_model": model, "ms_per_call": round(ms, 3), "calls": n,
                "GB/s": round(per_call_bytes / (ms * 1e-3) / 1e9, 4),
                "GFLOP/s": round(flops / (ms * 1e-3) / 1e9, 3)}
        print(json.dumps(line), flush=True)

    cases = [("int8 256x512 S=1", 1, 256, 512, 1, (1e-3, 1e-2)),
             ("int4 12288x6144 S=1", I4, 12288, 6144, 1, (5e-3, 2e-2)),
             ("int4 12288x6144 S=4", I4, 12288, 6144, 4, (5e-3, 2e-2))]
    cases += [("%s 8192x8192 S=1" % nm, f, 8192, 8192, 1, (1e-3, 2e-2))
              for nm, f in (("f32", 0), ("int8", 1), ("int4", 2), ("int2", 3))]
    for name, fmt, O, I, S, (lo, hi) in cases:
        codes, scales = synth.quant_tensor(fmt, O, I, 0, 1, lo, hi)
        x = synth.activations(S, I, 0, 9999)
        bits = {0: 32, 1: 8, 2: 4, 3: 2}[fmt]
        fn = (lambda c=codes, sc=scales, xx=x, f=fmt, o=O, i=I: oracle.matmul(f, o, i, c, sc, xx))
        for threads in ((0, 1) if S == 1 else (0,)):
            emit(name, algorithmic_bytes(bits, O, I, S), 2.0 * O * I * S, fn, threads, 1.0)
    # MoE expert layer, S=1: 8 experts' gate/up, silu(g)*u, down
    D, F = 6144, 2048
    ex = []
    for e in range(8):
        cg, sg = synth.quant_tensor(I4, F, D, 0, 10 + 3 * e, 5e-3, 2e-2)
        cu, su = synth.quant_tensor(I4, F, D, 0, 11 + 3 * e, 5e-3, 2e-2)
        cd, sd = synth.quant_tensor(I4, D, F, 0, 12 + 3 * e, 5e-3, 2e-2)
        ex.append((cg, sg, cu, su, cd, sd))
    xm = synth.activations(1, D, 0, 9999)

    def moe():
        for cg, sg, cu, su, cd, sd in ex:
            g, _, u, _ = oracle.matmul_gate_up(I4, F, D, cg, sg, cu, su, xm)
            _, h = oracle.silu_mul(g, u)
            oracle.matmul(I4, D, F, cd, sd, h)
    moe_bytes = 8 * (2 * algorithmic_bytes(4, F, D, 1) + algorithmic_bytes(4, D, F, 1))
    emit("MoE layer S=1, 8 experts (gate/up, silu*up, down)", moe_bytes, 8 * 3 * 2.0 * F * D, moe, 0, 1.0)
    # W4A16 prefill call, all cores (one call is about ten seconds)
    O, I, S = 12288, 6144, 1571
    codes, scales = synth.quant_tensor(I4, O, I, 0, 1, 5e-3, 2e-2)
    x = synth.activations(S, I, 0, 9999)
    oracle.set_threads(0)
    t0 = time.perf_counter()
    oracle.matmul(I4, O, I, codes, scales, x)
    dt = time.perf_counter() - t0
    print(json.dumps({"workload": "prefill W4A16 12288x6144 S=1571", "impl": "oracle", "cores": cores,
                      "cpu_model": model, "ms_per_call": round(dt * 1e3, 1), "calls": 1,
                      "GFLOP/s": round(2.0 * O * I * S / dt / 1e9, 3)}), flush=True)


def prefill_measure(q, steps, warmup, stream, gs=0):
    """W4A16 prefill O=12288, I=6144, S=1571 through b200q_matmul (tensor-core
    path; gs > 0: group-wise scales, one per row and gs columns); returns None
    while that path is not available."""
    import torch
    import synth
    O, I, S = 12288, 6144, 1571
    if gs:
        codes = synth.codes(I4, O, I, 0, 1)
        scales = synth.uniform_f32((O, -(-I // gs)), 5e-3, 2e-2, 0, 2)
        t = q.tensor_upload(I4, O, I, codes, scales, gs=gs)
    else:
        codes, scales = synth.quant_tensor(I4, O, I, 0, 1, 5e-3, 2e-2)
        t = q.tensor_upload(I4, O, I, codes, scales)
    try:
        if q.matmul_path(t, S) != q.PATH_TC:
            return None
        x = torch.from_numpy(synth.activations(S, I, 0, 9999)).cuda()
        y = torch.empty((S, O), dtype=torch.float32, device="cuda")
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        try:
            q.matmul(t, x, y, S, stream)
        except q.B200QError:
            return None
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                q.matmul(t, x, y, S, stream)
        torch.cuda.synchronize()
        times = []
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush.zero_()                               # L2 flush, ordered before the timed call
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            q.matmul(t, x, y, S, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        flops = 2.0 * O * I * S
        return {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "tokens_per_s": S / (ms * 1e-3)}
    finally:
        t.free()


# ----------------------------------------------------------------------------- main arms

def run_ours(args):
    import torch
    rank, world, local = dist_init(args.gpus)
    import quantized_weight_quant_gb300 as q
    torch.cuda.set_device(local)
    pk = peaks()
    O, I, S = 12288, 6144, 1
    per_copy = algorithmic_bytes(4, O, I, S)
    R = max(16, -(-3 * L2_BYTES // per_copy))
    wl = Decode(q, I4, O, I, S, R)
    stream = torch.cuda.Stream()
    with ClockSampler(local) as clk:
        ms, launches = time_steps(wl, args.steps, args.warmup, stream, world, graph=True)
        ms_eager, _ = time_steps(wl, args.steps, args.warmup, stream, world, graph=False)
    clocks = clk.summary()
    ms_max = max_over_ranks(ms, world)
    value = job_throughput(wl.bytes_per_step, args.steps, world, ms_max)
    per_launch_ms = ms / max(1, launches)
    achieved = per_copy / (per_launch_ms * 1e-3) / 1e9
    traffic = recorded_traffic("decode_i4_12288x6144_s1")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded: int4 codes uniform 0..15, scales U[5e-3,2e-2], x ~ N(0,1))",
        "config": {"workload": "int4 decode GEMV O=12288 I=6144 S=1, one step = one token through "
                               "%d resident copies" % R,
                   "O": O, "I": I, "S": S, "weights": "int4 codes, f32 row scales", "x_y": "f32",
                   "copies": R, "global_batch": S * world,
                   "l2": "inputs larger than L2: %d distinct weight copies, %.0f MB per step > 3x L2"
                         % (R, wl.bytes_per_step / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_hbm_peak": round(100.0 * value / world / pk["hbm_gbs"], 2),
        "timing": "one step captured once as a CUDA graph and replayed; eager (a host call per matmul) "
                  "gives %.1f GB/s" % (wl.bytes_per_step * args.steps * world / (max_over_ranks(ms_eager, world) * 1e-3) / 1e9),
        "gpu_launches": int(launches),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": traffic,
                     "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                     "per_launch_us": round(per_launch_ms * 1e3, 3),
                     "algorithmic_bytes_per_launch": per_copy},
        "clocks": clocks,
    }
    # W4A16 prefill TFLOP/s (second half of the metric)
    if not args.no_prefill:
        pf = prefill_measure(q, max(5, min(args.steps, 20)), max(3, args.warmup), stream)
        if pf is None:
            line["prefill_w4a16"] = {"unavailable": "tensor-core path not built"}
        else:
            peak_tc = pk["bf16_tflops"]
            line["prefill_w4a16"] = {
                "workload": "W4A16 prefill O=12288 I=6144 S=1571 (x f32 -> bf16 in the call)",
                "value": round(pf["tflops"], 2), "unit": "TFLOP/s", "ms": round(pf["ms"], 4),
                "tokens_per_s": round(pf["tokens_per_s"], 1),
                "roofline": {"bound": "tensor", "achieved": round(pf["tflops"], 2), "peak": peak_tc,
                             "unit": "TFLOP/s", "frac": round(pf["tflops"] / peak_tc, 4),
                             "traffic": recorded_traffic("prefill_i4_12288x6144_s1571"),
                             "peak_source": pk["source"] + " (MEASURED_PEAKS.json bf16_tflops, burst)"}}
    # MoE expert layer at S=1 (8 of 256 resident experts), grouped and per expert
    if not args.no_moe:
        line["moe_layer"] = moe_measure(q, max(5, min(args.steps, 20)), max(3, args.warmup), stream)
    line["layer_glue"] = glue_measure(q, max(5, min(args.steps, 20)), max(3, args.warmup), stream)
    if not args.no_mla:
        line["mla_decode"] = mla_measure(q, max(5, min(args.steps, 20)), max(3, args.warmup), stream)
    # end to end through the host-buffer C-ABI call
    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, h2d, d2h = time_e2e_step(wl, e2e_steps, 2)
    e2e_ms_max = max_over_ranks(e2e_ms, world)
    line["e2e"] = {"value": round(wl.bytes_per_step * e2e_steps * world / (e2e_ms_max * 1e-3) / 1e9, 2),
                   "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "call": "per step: pinned H2D of x, %d b200q_matmul calls on device buffers, D2H of all "
                           "outputs to pinned memory, stream sync (host wall clock)" % wl.R}
    hc_ms, hc_h2d, hc_d2h = time_e2e(wl, e2e_steps, 2)
    hc_ms_max = max_over_ranks(hc_ms, world)
    line["e2e_host_call"] = {"value": round(wl.bytes_per_step * e2e_steps * world / (hc_ms_max * 1e-3) / 1e9, 2),
                             "unit": "GB/s", "h2d_bytes_per_step": hc_h2d, "d2h_bytes_per_step": hc_d2h,
                             "call": "b200q_matmul_host per matmul (the pages' convention: pinned host x in, host "
                                     "y out, synchronous per call)"}
    wl.close()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(O, I, S)
    if rank == 0:
        # the headline's own figures close the line (a reader that keeps only
        # the end of stdout still has them): decode roofline, prefill last
        for k in ("e2e_host_call", "cpu_baseline", "e2e", "roofline", "prefill_w4a16"):
            if k in line:
                line[k] = line.pop(k)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_sweep(args):
    """Every decode config as one JSON line each (device time, weight rotation
    larger than L2), then the MoE layer and the prefill."""
    import torch
    import quantized_weight_quant_gb300 as q
    torch.cuda.set_device(0)
    pk = peaks()
    stream = torch.cuda.Stream()
    cases = [("int8 256x512", 1, 256, 512, 1)]
    cases += [("int4 12288x6144", I4, 12288, 6144, s) for s in (1, 4)]
    cases += [("%s 8192x8192" % n, f, 8192, 8192, s) for n, f in (("f32", 0), ("int8", 1), ("int4", 2), ("int2", 3))
              for s in (1, 2, 8)]
    cases = [c + (0,) for c in cases] + [("int4 12288x6144 gs=128", I4, 12288, 6144, 1, 128),
                                         ("int4 12288x6144 gs=128", I4, 12288, 6144, 4, 128)]
    for name, fmt, O, I, S, gs in cases:
        bits = {0: 32, 1: 8, 2: 4, 3: 2}[fmt]
        per = algorithmic_bytes(bits, O, I, S)
        R = max(2, min(64, -(-3 * L2_BYTES // per)))
        wl = Decode(q, fmt, O, I, S, R, gs=gs)
        ms, launches = time_steps(wl, args.steps, args.warmup, stream)
        gbs = wl.bytes_per_step * args.steps / (ms * 1e-3) / 1e9
        print(json.dumps({"workload": "%s S=%d" % (name, S), "GB/s": round(gbs, 1),
                          "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                          "us_per_call": round(ms * 1e3 / (args.steps * R), 3),
                          "launches_per_call": launches / (args.steps * R), "copies": R}), flush=True)
        wl.close()
    moe = moe_measure(q, args.steps, args.warmup, stream)
    print(json.dumps(moe), flush=True)
    print(json.dumps(glue_measure(q, max(5, min(args.steps, 20)), max(3, args.warmup), stream)), flush=True)
    pf = prefill_measure(q, max(5, min(args.steps, 20)), max(3, args.warmup), stream)
    print(json.dumps({"workload": "prefill W4A16 12288x6144 S=1571", "result": pf}), flush=True)
    pf = prefill_measure(q, max(5, min(args.steps, 20)), max(3, args.warmup), stream, gs=128)
    print(json.dumps({"workload": "prefill W4A16 12288x6144 S=1571 gs=128", "result": pf}), flush=True)


def run_single(args):
    """One configuration (for profiling runs): --workload decode|prefill with
    --fmt/--O/--I/--S/--copies (--gs: group-wise scales); one JSON line."""
    import torch
    import quantized_weight_quant_gb300 as q
    torch.cuda.set_device(0)
    pk = peaks()
    stream = torch.cuda.Stream()
    fmt = {"f32": 0, "i8": 1, "i4": 2, "i2": 3}[args.fmt]
    bits = {0: 32, 1: 8, 2: 4, 3: 2}[fmt]
    per = algorithmic_bytes(bits, args.O, args.I, args.S)
    R = args.copies or max(2, min(64, -(-3 * L2_BYTES // per)))
    path = {"auto": None, "f32": q.PATH_F32, "tc": q.PATH_TC, "tcx": q.PATH_TCX, "tcs": q.PATH_TCS}[args.path]
    wl = Decode(q, fmt, args.O, args.I, args.S, R, gs=args.gs, path=path)
    ms, launches = time_steps(wl, args.steps, args.warmup, stream)
    sec = ms * 1e-3
    print(json.dumps({"workload": "%s %s O=%d I=%d S=%d gs=%d" % (args.workload, args.fmt, args.O, args.I, args.S,
                                                                  args.gs),
                      "path": q.matmul_path(wl.tensors[0], args.S) if path is None else path,
                      "GB/s": round(wl.bytes_per_step * args.steps / sec / 1e9, 1),
                      "frac_hbm": round(wl.bytes_per_step * args.steps / sec / 1e9 / pk["hbm_gbs"], 4),
                      "TFLOP/s": round(wl.flops_per_step * args.steps / sec / 1e12, 2),
                      "us_per_call": round(ms * 1e3 / (args.steps * R), 3), "copies": R,
                      "launches": launches}), flush=True)
    wl.close()


def moe_measure(q, steps, warmup, stream):
    """MoE expert layer at S=1: 256 resident experts (int4 gate/up [2048,6144],
    down [6144,2048]); each step routes one token to 8 distinct experts
    (pre-drawn seeded ids).  Two forms of the same layer: per expert (fused
    gate/up -> silu*up -> down, 24 launches) and grouped (the 16 gate/up
    tensors in one call, the 8 down tensors on silu(g)*u in a second)."""
    import torch
    import synth
    D, F, E, K = 6144, 2048, 256, 8
    gates, ups, downs = [], [], []
    for e in range(E):
        cg, sg = synth.quant_tensor(I4, F, D, 0, 10 * e + 1, 5e-3, 2e-2)
        cu, su = synth.quant_tensor(I4, F, D, 0, 10 * e + 2, 5e-3, 2e-2)
        cd, sd = synth.quant_tensor(I4, D, F, 0, 10 * e + 3, 5e-3, 2e-2)
        gates.append(q.tensor_upload(I4, F, D, cg, sg))
        ups.append(q.tensor_upload(I4, F, D, cu, su))
        downs.append(q.tensor_upload(I4, D, F, cd, sd))
    ids = synth.expert_draws(E, K, steps + warmup, 0, 77)
    x = torch.from_numpy(synth.activations(1, D, 0, 78)).cuda()
    yg = torch.empty((K, F), device="cuda")
    yu = torch.empty((K, F), device="cuda")
    h = torch.empty((K, F), device="cuda")
    y = torch.empty((K, D), device="cuda")

    def step(r):
        for k in range(K):
            e = int(ids[r, k])
            q.matmul_gate_up(gates[e], ups[e], x, yg[k], yu[k], 1, stream)
            q.silu_mul(yg[k], yu[k], h[k], F, stream)
            q.matmul(downs[e], h[k], y[k], 1, stream)

    def step_grouped(r):
        sel = [int(e) for e in ids[r]]
        q.matmul_grouped([t for e in sel for t in (gates[e], ups[e])], [x] * (2 * K),
                         [v for k in range(K) for v in (yg[k], yu[k])], 1, stream)
        q.matmul_grouped_silu([downs[e] for e in sel], [yg[k] for k in range(K)], [yu[k] for k in range(K)],
                              [y[k] for k in range(K)], 1, stream)

    with torch.cuda.stream(stream):
        for r in range(warmup):
            step(r)
            step_grouped(r)
    torch.cuda.synchronize()

    def timed(fn):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms = timed(lambda: [step(warmup + r) for r in range(steps)])
    # the same routed sequence captured once as a CUDA graph
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(steps):
            step(warmup + r)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    ms_graph = timed(g.replay)
    ms_grp = timed(lambda: [step_grouped(warmup + r) for r in range(steps)])
    gg = torch.cuda.CUDAGraph()
    n0 = q.kernel_launches()
    with torch.cuda.graph(gg, stream=stream):
        for r in range(steps):
            step_grouped(warmup + r)
    grp_launches = (q.kernel_launches() - n0) / steps
    with torch.cuda.stream(stream):
        gg.replay()
    torch.cuda.synchronize()
    ms_grp_graph = timed(gg.replay)
    layer_bytes = K * (2 * algorithmic_bytes(4, F, D, 1) - 4 * D + algorithmic_bytes(4, D, F, 1) + 4 * 2 * F)
    for lst in (gates, ups, downs):
        for t in lst:
            t.free()
    hbm = peaks()["hbm_gbs"]
    def rate(ms_):
        return {"us_per_layer": round(ms_ * 1e3, 2), "layer_tokens_per_s": round(1e3 / ms_, 1),
                "GB/s": round(layer_bytes / (ms_ * 1e-3) / 1e9, 1),
                "frac_hbm": round(layer_bytes / (ms_ * 1e-3) / 1e9 / hbm, 4)}

    return {"workload": "MoE expert layer S=1, 8 of 256 experts",
            "grouped_graph": dict(rate(ms_grp_graph), launches_per_layer=grp_launches,
                                  form="matmul_grouped (16 gate/up tensors, one x) + matmul_grouped_silu "
                                       "(8 down tensors on silu(g)*u)"),
            "grouped_plain": rate(ms_grp),
            "per_expert_graph": rate(ms_graph),
            "per_expert_plain": rate(ms),
            "bytes_per_layer": layer_bytes}


MLA_SHAPE = {"H": 64, "Dn": 128, "Dv": 128, "K": 512, "R": 64}


def mla_fma(H, Dn, Dv, K, R, S, T, st0=0):
    """Multiply-adds of one absorbed-attention call: absorb, scores, latent
    context, value rows (each token's causal window)."""
    win = sum(T - S + s - st0 + 1 for s in range(S))
    return H * (S * Dn * K + win * (K + R) + win * K + S * Dv * K)


def mla_bytes(H, Dn, Dv, K, R, S, T, st0=0):
    """Cache rows of the window, int4 codes + row scales of Wkv_b, q and ctx."""
    rows = H * (Dn + Dv)
    return (T - st0) * (K + R) * 4 + rows * ((K + 1) // 2 + 4) + S * H * (Dn + R + Dv) * 4


def mla_measure(q, steps, warmup, stream, cases=((1, 4096), (4, 4096), (1, 32768))):
    """MLA decode attention with weight absorption (b200q_mla_absorb), int4
    Wkv_b [64 * 256, 512], latent 512 + rope 64, paged caches, per call:
    a CUDA graph of calls cycling over enough copies of the weights and
    caches to exceed L2 twice.  The dominant kernel does f32 FMAs on the
    SIMT pipe, so the roofline is the FP32 FMA peak at the sampled SM clock
    (152 SMs x 128 lanes x 2 FLOP x MHz); the HBM fraction is given beside it."""
    import torch
    import synth
    sh = MLA_SHAPE
    H, Dn, Dv, K, R = sh["H"], sh["Dn"], sh["Dv"], sh["K"], sh["R"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = {"workload": "MLA absorb decode, int4 Wkv_b, H=64 Dn=Dv=128 K=512 R=64, 64-position pages", "cases": []}
    for S, T in cases:
        per_copy = T * (K + R) * 4 + H * (Dn + Dv) * (K // 2 + 4)
        copies = max(2, min(16, -(-2 * L2_BYTES // per_copy)))
        ws, kvs = [], []
        for c in range(copies):
            codes, sc = synth.quant_tensor(I4, H * (Dn + Dv), K, 0, 900 + c, 5e-3, 2e-2)
            ws.append(q.tensor_upload(I4, H * (Dn + Dv), K, codes, sc))
            kv = q.PagedKV(K, R, T)
            kv.lat_pool.normal_()
            kv.rope_pool.normal_()
            kvs.append(kv)
        qn = torch.from_numpy(synth.normal_f32((S, H, Dn), 0, 901)).cuda()
        qr = torch.from_numpy(synth.normal_f32((S, H, R), 0, 902)).cuda()
        ctx = torch.empty((S, H, Dv), device="cuda")
        scale = (Dn + R) ** -0.5

        def call(c):
            kvs[c].attend(ws[c], H, Dn, Dv, qn, qr, T, 0, scale, ctx, S, stream)

        with torch.cuda.stream(stream):
            for r in range(max(warmup, copies)):
                call(r % copies)
        torch.cuda.synchronize()
        n = 2 * copies
        g = torch.cuda.CUDAGraph()
        n0 = q.kernel_launches()
        with torch.cuda.graph(g, stream=stream):
            for r in range(n):
                call(r % copies)
        launches = (q.kernel_launches() - n0) / n
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        reps = max(3, steps // 4)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
        ck = clk.summary()
        us = e0.elapsed_time(e1) * 1e3 / (reps * n)
        fma = mla_fma(H, Dn, Dv, K, R, S, T)
        nbytes = mla_bytes(H, Dn, Dv, K, R, S, T)
        mhz = ck.get("sm_mhz") or 2032.0
        peak = sms * 128 * 2 * mhz * 1e6 / 1e12
        tflops = 2 * fma / (us * 1e-6) / 1e12
        gbs = nbytes / (us * 1e-6) / 1e9
        out["cases"].append({
            "S": S, "T": T, "us_per_call": round(us, 2), "tokens_per_s": round(S / (us * 1e-6), 1),
            "launches_per_call": launches, "copies": copies,
            "roofline": {"bound": "alu", "achieved": round(tflops, 2), "peak": round(peak, 2), "unit": "TFLOP/s",
                         "frac": round(tflops / peak, 4),
                         "peak_source": "FP32 FMA: %d SMs x 128 lanes x 2 FLOP x %.0f MHz (sampled)" % (sms, mhz)},
            "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks()["hbm_gbs"], 4),
            "fma_per_call": fma, "bytes_per_call": nbytes, "clocks": ck})
        for t in ws:
            t.free()
        del kvs
        torch.cuda.empty_cache()
    return out


def glue_measure(q, steps, warmup, stream):
    """Layer glue: RMSNorm with a residual (h = x + r written back, y = norm(h) * w),
    D = 6144, at S = 1 (a chain of dependent calls as one CUDA graph) and
    S = 1571 (L2 flushed before each call, on the timed stream)."""
    import torch
    import synth
    D = 6144
    out = {"workload": "RMSNorm + residual, D=6144"}
    w = torch.from_numpy(synth.uniform_f32((D,), 0.5, 1.5, 0, 3)).cuda()
    for S in (1, 1571):
        x = torch.from_numpy(synth.normal_f32((S, D), 0, 1)).cuda()
        r = torch.from_numpy(synth.normal_f32((S, D), 0, 2)).cuda()
        h = torch.empty_like(x)
        y = torch.empty_like(x)
        nbytes = 4 * S * D * 4 + 4 * D
        if S == 1:
            n = 64
            with torch.cuda.stream(stream):
                for _ in range(warmup):
                    q.rmsnorm(x, w, y, S, D, 1e-6, r=r, h=h, stream=stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n):
                    q.rmsnorm(x, w, y, S, D, 1e-6, r=r, h=h, stream=stream)
            with torch.cuda.stream(stream):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(steps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (steps * n)
            out["S1_us_per_call"] = round(us, 3)
        else:
            flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
            with torch.cuda.stream(stream):
                for _ in range(warmup):
                    q.rmsnorm(x, w, y, S, D, 1e-6, r=r, h=h, stream=stream)
            torch.cuda.synchronize()
            times = []
            for _ in range(steps):
                with torch.cuda.stream(stream):
                    flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                q.rmsnorm(x, w, y, S, D, 1e-6, r=r, h=h, stream=stream)
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.median(times)
            gbs = nbytes / (ms * 1e-3) / 1e9
            out["S1571"] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                            "frac_hbm": round(gbs / peaks()["hbm_gbs"], 4), "bytes": nbytes}
    return out


def run_reference(args):
    """The CPU oracle on the same workload and metric, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import synth
    O, I, S = 12288, 6144, 1
    codes, scales = synth.quant_tensor(I4, O, I, 0, 1, 5e-3, 2e-2)
    x = synth.activations(S, I, 0, 9999)
    oracle.set_threads(0)
    for _ in range(args.warmup):
        oracle.matmul(I4, O, I, codes, scales, x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul(I4, O, I, codes, scales, x)
    dt = time.perf_counter() - t0
    per_step = algorithmic_bytes(4, O, I, S)
    value = per_step * args.steps / dt / 1e9
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "int4 decode GEMV O=12288 I=6144 S=1 (one step = one call of the CPU oracle "
                               "on the whole tensor)", "O": O, "I": I, "S": S},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": "full O=12288 I=6144 S=1 int4 matmul per step"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-moe", action="store_true")
    ap.add_argument("--no-mla", action="store_true")
    ap.add_argument("--workload", default="default",
                    choices=["default", "sweep", "decode", "prefill", "moe", "mla", "cpu"])
    ap.add_argument("--fmt", default="i4", choices=["f32", "i8", "i4", "i2"])
    ap.add_argument("--O", type=int, default=12288)
    ap.add_argument("--I", type=int, default=6144)
    ap.add_argument("--S", type=int, default=1)
    ap.add_argument("--gs", type=int, default=0, help="group size of the scales (0: one per row)")
    ap.add_argument("--T", type=int, default=0, help="cached positions of the mla workload (0: its default cases)")
    ap.add_argument("--copies", type=int, default=0, help="distinct weight copies (0: enough for 3x L2)")
    ap.add_argument("--path", default="auto", choices=["auto", "f32", "tc", "tcx", "tcs"],
                    help="matmul path of the decode / prefill workload (auto: the library's choice)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "cpu":
        run_cpu_plan(args)
    elif args.workload == "sweep":
        run_sweep(args)
    elif args.workload in ("decode", "prefill"):
        run_single(args)
    elif args.workload == "moe":
        import torch
        import quantized_weight_quant_gb300 as q
        torch.cuda.set_device(0)
        print(json.dumps(moe_measure(q, args.steps, args.warmup, torch.cuda.Stream())), flush=True)
    elif args.workload == "mla":
        import torch
        import quantized_weight_quant_gb300 as q
        torch.cuda.set_device(0)
        cases = ((args.S, args.T),) if args.T else ((1, 4096), (4, 4096), (1, 32768))
        print(json.dumps(mla_measure(q, args.steps, args.warmup, torch.cuda.Stream(), cases)), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
