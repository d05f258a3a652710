"""Bench: achieved HBM GB/s of the fused epilogue ops on GB300.

One step = one call of every op on its measured workload (SkipLayerNormalization
f16 16384x4096 with bias/residual, f32 (32,2048,1024) with a broadcast skip and
f32 (2,128,768); BiasSoftmax f16 (32,16,512,512) causal, f32 64x262144 and
8x1048576 long rows; BiasAdd f16 (16,1024,4096); QuickGelu f16 67,108,867).

value        = minimum bytes of all ops (every input read once, every output
               written once, reused vectors counted once) / device time of a step
               (every 8th timed step carries one event pair, around the dominant
               op; an event record costs ~2 us of stream time and ends the
               programmatic overlap of the kernels on either side)
ops          = per op: the mean from a separate loop of steps with an event pair
               around every op ("in the step": each op also writes back the
               previous op's dirty L2 lines), and the median / minimum / mean of
               50 launches of the op alone, each after an L2 flush that leaves
               only clean lines ("isolated"); fractions against the measured
               copy bandwidth and against the nominal 8 TB/s
e2e          = the same metric with each step's inputs copied host->device from
               pinned memory and outputs copied back, inside the timed region
roofline     = the dominant kernel's algorithmic bytes / its mean CUDA-event
               duration, against the measured HBM copy bandwidth
cpu_baseline = the float64 CPU oracle on a bounded sample of the same workloads

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workloads on its own GPU
(independent replicas: the ops are row-independent and need no exchange);
timings are max-reduced over ranks.
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gen import synth  # noqa: E402

METRIC = "achieved HBM GB/s per op and % of GB300 HBM roofline; rows/sec for SkipLayerNorm"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal

# Step order: each small workload follows a large streaming one.
K_BREAKDOWN = 50  # steps of the per-op breakdown loop
K_ISOLATED = 50   # launches of each op alone, each after an L2 flush
DOM_EVERY = 8     # timed steps per event-bracketed launch of the dominant op

ORDER = [
    "sln_f16_16384x4096_bias_residual",
    "sln_f32_2x128x768",
    "sln_f32_32x2048x1024_bcast_skip",
    "bias_add_f16_16x1024x4096",
    "bias_softmax_f32_64x262144_cyclic",
    "quick_gelu_f16_67108867",
    "bias_softmax_f16_32x16x512x512_causal",
    "bias_softmax_f32_8x1048576",
]

# DRAM bytes (read + write) per launch from ncu captures of each kernel alone
# (`--profile NAME`: one workload, a few launches), keyed by workload, with the
# hash of the kernel sources' code (comments excluded) they were taken on.  A
# changed source makes the figure stale and it is reported as null.  ncu flushes L2 before each launch,
# so reads are cold (the split-row softmax: pass 2 re-reads from DRAM what a
# step serves from L2), and writes still dirty in L2 when a kernel ends are not
# counted.
NCU_TRAFFIC = {
    "bias_add_f16_16x1024x4096": 356523008,
    "bias_softmax_f16_32x16x512x512_causal": 495178240,
    "bias_softmax_f32_64x262144_cyclic": 153501952,
    "bias_softmax_f32_8x1048576": 75607808,
    "quick_gelu_f16_67108867": 210126592,
    "sln_f16_16384x4096_bias_residual": 479411712,
    "sln_f32_2x128x768": 1608960,
    "sln_f32_32x2048x1024_bcast_skip": 488529664,
}
NCU_TRAFFIC_SOURCE_HASH = "24ff61884dc1d62d"


def _code_only(text: str) -> str:
    """C/C++ source without its comments and blank lines (string and character
    literals kept), so that a comment-only edit leaves the hash unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments excluded)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transformer_epilogue_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# workloads: minimum bytes and calls
# ---------------------------------------------------------------------------

def nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def min_bytes(name, d):
    """Every input read once, every output written once; reused vectors
    (gamma, beta, bias, a broadcast skip, bias rows) count once."""
    w = synth.WORKLOADS[name]
    if w.op == "skip_layer_norm":
        b = sum(nbytes(d[k]) for k in ("input", "skip", "gamma", "beta", "bias"))
        b += nbytes(d["input"]) * (2 if d.get("residual") else 1)
        return b
    if w.op == "bias_softmax":
        return nbytes(d["data"]) * 2 + nbytes(d["bias"])
    if w.op == "bias_add":
        return nbytes(d["X"]) * 2 + nbytes(d["skip"]) + nbytes(d["bias"])
    if w.op == "quick_gelu":
        return nbytes(d["X"]) * 2
    raise KeyError(name)


def rows_of(name, d):
    w = synth.WORKLOADS[name]
    if w.op == "skip_layer_norm":
        return d["input"].numel() // d["input"].shape[-1]
    return None


class DeviceWorkload:
    """Device-resident inputs/outputs of one workload and its op call."""

    def __init__(self, name, host, device):
        import transformer_epilogue_gb300 as te
        self.te = te
        self.name = name
        self.op = synth.WORKLOADS[name].op
        self.host = host
        self.dev = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        d = self.dev
        if self.op == "skip_layer_norm":
            self.outs = {"output": torch.empty_like(d["input"])}
            if host.get("residual"):
                self.outs["sum"] = torch.empty_like(d["input"])
        elif self.op == "bias_softmax":
            self.outs = {"output": torch.empty_like(d["data"])}
            need = te.ep_bias_softmax_workspace_size(d["data"].dtype, d["data"].shape, d["axis"])
            self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device) if need else None
        else:
            self.outs = {"Y": torch.empty_like(d["X"])}
        self.inputs = [k for k, v in self.dev.items() if isinstance(v, torch.Tensor)]

    def call(self):
        te, d, o = self.te, self.dev, self.outs
        if self.op == "skip_layer_norm":
            te.ep_skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"],
                                  output=o["output"], input_skip_bias_sum=o.get("sum"))
        elif self.op == "bias_softmax":
            te.ep_bias_softmax(d["data"], d["bias"], axis=d["axis"], is_inner_broadcast=d["is_inner_broadcast"],
                               output=o["output"], workspace=self.ws)
        elif self.op == "bias_add":
            te.ep_bias_add(d["X"], d["bias"], d["skip"], Y=o["Y"])
        else:
            te.ep_quick_gelu(d["X"], d["alpha"], Y=o["Y"])


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.idx)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t_begin - 0.15 <= r[0] <= t_end + 0.15] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[3][1:5]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------------------
# CPU oracle on bounded samples (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_call(name, d, frac_rows):
    """Run the oracle on the first max(1, frac_rows * rows) rows of a workload;
    returns the minimum bytes of that sample."""
    import oracle
    w = synth.WORKLOADS[name]
    if w.op == "skip_layer_norm":
        H = d["input"].shape[-1]
        R = d["input"].numel() // H
        n = max(1, int(R * frac_rows))
        rows = list(range(n))
        oracle.skip_layer_norm(d["input"], d["skip"], d["gamma"], d["beta"], d["bias"], d["epsilon"], rows=rows)
        if d.get("residual"):
            oracle.skip_bias_sum(d["input"], d["skip"], d["bias"], rows=rows)
        es = d["input"].element_size()
        return n * H * es * (3 + (1 if d.get("residual") else 0))
    if w.op == "bias_softmax":
        dims = oracle.bias_softmax_dims(tuple(d["data"].shape), d["bias"].numel(), d["axis"])
        n = max(1, int(dims["batch"] * frac_rows))
        oracle.bias_softmax(d["data"], d["bias"], d["axis"], d["is_inner_broadcast"], rows=list(range(n)))
        return n * dims["block"] * d["data"].element_size() * 3
    if w.op == "bias_add":
        C = d["X"].shape[-1]
        R = d["X"].numel() // C
        n = max(1, int(R * frac_rows))
        X = d["X"].reshape(-1, C)[:n].reshape(1, n, C)
        S = d["skip"].reshape(-1, C)[:n].reshape(1, n, C)
        oracle.bias_add(X, d["bias"], S)
        return n * C * d["X"].element_size() * 3
    n = max(1, int(d["X"].numel() * frac_rows))
    oracle.quick_gelu(d["X"][:n], d["alpha"])
    return n * d["X"].element_size() * 2


def oracle_step(hosts, frac):
    t0 = time.perf_counter()
    b = sum(oracle_sample_call(n, hosts[n], frac) for n in ORDER)
    return b, time.perf_counter() - t0


def pin_one_core():
    try:
        cpu = sorted(os.sched_getaffinity(0))[0]
        old = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {cpu})
        return old
    except (AttributeError, OSError):
        return None


def calibrate(hosts, target_s, frac=1.0 / 8192):
    """Grow the row fraction until one oracle step takes about target_s."""
    b, t = oracle_step(hosts, frac)
    for _ in range(6):
        if t >= 0.5 * target_s or frac >= 1.0:
            break
        frac = min(1.0, frac * min(16.0, max(1.5, target_s / max(t, 1e-3))))
        b, t = oracle_step(hosts, frac)
    return frac, b, t


def host_cpu() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def cpu_baseline(hosts, budget_s=15.0):
    old = pin_one_core()
    try:
        frac, b, t = calibrate(hosts, budget_s)
    finally:
        if old is not None:
            os.sched_setaffinity(0, old)
    return {"value": b / t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle", "host_cpu": host_cpu(),
            "sample": f"first {frac:.5f} of the rows of every workload (numpy float64, 1 pinned core), "
                      f"{b / 1e6:.1f} MB of minimum traffic in {t:.1f} s; host has {os.cpu_count()} cores"}


# ---------------------------------------------------------------------------

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: torch copy, read+write, burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, no MEASURED_PEAKS.json)"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max_sum(values_max, values_sum, ws):
    """max over ranks of the first list, sum over ranks of the second."""
    if ws == 1:
        return list(values_max), list(values_sum)
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    a = torch.tensor(values_max, dtype=torch.float64, device=dev)
    b = torch.tensor(values_sum, dtype=torch.float64, device=dev)
    dist.all_reduce(a, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return a.cpu().tolist(), b.cpu().tolist()


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def build_hosts():
    hosts = {}
    for n in ORDER:
        hosts[n] = synth.workload(n)
    return hosts


def sliced_workload(name, batch):
    """The named workload with its leading dimension cut to `batch`: every
    tensor whose first dimension equals the data's is sliced (so a causal mask
    follows its data and SkipLayerNorm's skip its input, while a broadcast skip
    or a cyclic bias is kept whole)."""
    d = synth.workload(name)
    if not batch:
        return d
    lead = next(d[k] for k in ("input", "data", "X") if k in d).shape[0]
    if batch > lead:
        raise ValueError(f"batch {batch} > leading dimension {lead} of {name}")
    return {k: (v[:batch].contiguous() if isinstance(v, torch.Tensor) and v.dim() and v.shape[0] == lead else v)
            for k, v in d.items()}


def isolated_times(work, device, reps=K_ISOLATED):
    """Each op alone, `reps` launches, each after an L2 flush outside the event
    pair: write 2x L2 then read 2x L2, so the L2 holds only clean lines when
    the op starts.  Returns per-op lists of durations (ms)."""
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or (132 << 20))
    fw = torch.empty(2 * l2, dtype=torch.uint8, device=device)
    fr = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    out = []
    for w in work:
        ts = []
        for _ in range(reps):
            fw.zero_()
            fr.max()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            w.call()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        out.append(ts)
    del fw, fr
    return out


def run_profile(args):
    """Runs one workload `--reps` times and nothing else (a target for ncu)."""
    import transformer_epilogue_gb300 as te
    te.load_library()
    w = DeviceWorkload(args.profile, sliced_workload(args.profile, args.batch), torch.device("cuda"))
    for _ in range(args.reps):
        w.call()
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "batch": args.batch, "reps": args.reps}), flush=True)
    return 0


def run_profile_shape(args):
    """Runs one shape outside the bench workloads `--reps` times and nothing
    else (a target for ncu): softmax:DTYPE:ROWS:COLS (8 cyclic bias rows) or
    sln:DTYPE:ROWS:H (beta, bias and the residual output)."""
    import transformer_epilogue_gb300 as te
    te.load_library()
    op, dts, rows, cols = args.profile_shape.split(":")
    rows, cols = int(rows), int(cols)
    dt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dts]
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    x = torch.randn(rows, cols, device="cuda", generator=g).to(dt)
    o = torch.empty_like(x)
    if op == "softmax":
        b = torch.randn(8, cols, device="cuda", generator=g).to(dt)
        fn = lambda: te.ep_bias_softmax(x, b, axis=1, is_inner_broadcast=0, output=o)
    elif op == "sln":
        sk = torch.randn(rows, cols, device="cuda", generator=g).to(dt)
        r = torch.empty_like(x)
        gm, bt, bi = (torch.randn(cols, device="cuda", generator=g).to(dt) for _ in range(3))
        fn = lambda: te.ep_skip_layer_norm(x, sk, gm, bt, bi, 1e-12, output=o, input_skip_bias_sum=r)
    else:
        raise ValueError(f"unknown op {op!r} (softmax or sln)")
    for _ in range(args.reps):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"profile_shape": args.profile_shape, "reps": args.reps}), flush=True)
    return 0


def run_reference(args, ws, rank):
    """The reference arm: the float64 CPU oracle, as it stands, on bounded
    samples of the same workloads (rank 0 only)."""
    if rank != 0:
        return 0
    hosts = build_hosts()
    total_steps = args.steps + args.warmup
    budget = min(2.0, 150.0 / max(1, total_steps))
    old = pin_one_core()
    try:
        frac, _, _ = calibrate(hosts, budget)
        for _ in range(args.warmup):
            oracle_step(hosts, frac)
        tb, tt = 0, 0.0
        for _ in range(args.steps):
            b, t = oracle_step(hosts, frac)
            tb += b
            tt += t
    finally:
        if old is not None:
            os.sched_setaffinity(0, old)
    v = tb / tt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; gen/synth.py)",
            "config": {"workload": "all eight epilogue workloads (bounded row samples on the CPU)",
                       "sample_fraction_of_rows": frac},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "host_cpu": host_cpu(),
                             "sample": f"first {frac:.6f} of the rows of every workload per step"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=ORDER, help="run only this workload --reps times (for ncu)")
    ap.add_argument("--batch", type=int, default=0, help="with --profile: cut the leading dimension to this")
    ap.add_argument("--reps", type=int, default=3, help="with --profile: calls of the op")
    ap.add_argument("--profile-shape", help="softmax|sln:DTYPE:ROWS:COLS: run that shape --reps times (for ncu)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    if args.profile:
        return run_profile(args)
    if args.profile_shape:
        return run_profile_shape(args)

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        rc = run_reference(args, ws, rank)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc

    import transformer_epilogue_gb300 as te
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    te.load_library()
    hosts = build_hosts()
    work = [DeviceWorkload(n, hosts[n], device) for n in ORDER]
    bytes_per = [min_bytes(n, hosts[n]) for n in ORDER]
    step_bytes = sum(bytes_per)
    stream = torch.cuda.current_stream(device)

    # warm-up
    for _ in range(args.warmup):
        for w in work:
            w.call()
    torch.cuda.synchronize()

    # per-op breakdown (its own loop, before the timed region): an event pair
    # around every op; each event record adds ~2 us of stream time, so these
    # loops are not the step time
    B = max(5, min(K_BREAKDOWN, args.steps))
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in work]
          for _ in range(B)]
    torch.cuda.synchronize()
    for k in range(B):
        for i, w in enumerate(work):
            ev[k][i][0].record(stream)
            w.call()
            ev[k][i][1].record(stream)
    torch.cuda.synchronize()
    per_op_ms = [statistics.fmean(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(B)) for i in range(len(work))]
    dom = max(range(len(ORDER)), key=lambda i: per_op_ms[i])
    iso_ms = isolated_times(work, device)

    # timed region: K steps; an event pair around the dominant op in every
    # DOM_EVERY-th step (its launch duration for the roofline), no other per-op
    # events: a record between two kernels also ends their programmatic overlap
    K = args.steps
    dom_steps = [k for k in range(K) if k % DOM_EVERY == DOM_EVERY - 1] or [K - 1]
    dom_ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in dom_steps}
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    n_launch0 = te.kernel_launch_count()
    wall0 = time.time()
    t_start.record(stream)
    for k in range(K):
        for i, w in enumerate(work):
            if i == dom and k in dom_ev:
                dom_ev[k][0].record(stream)
                w.call()
                dom_ev[k][1].record(stream)
            else:
                w.call()
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(ws)
    launches = te.kernel_launch_count() - n_launch0
    clk = clocks.stop(wall0, wall1)
    total_ms = t_start.elapsed_time(t_end)
    dom_ms = statistics.fmean(a.elapsed_time(b) for a, b in dom_ev.values())

    # e2e: pinned host inputs -> device, op, outputs -> pinned host, per step.
    # All pinned buffers are views of one page-locked block per direction (two
    # host allocations, not one per tensor).
    def pinned_views(tensors):
        sizes = [(nbytes(t) + 255) // 256 * 256 for t in tensors]
        block = torch.empty(sum(sizes), dtype=torch.uint8, pin_memory=True)
        views, off = [], 0
        for t, sz in zip(tensors, sizes):
            views.append(block[off:off + nbytes(t)].view(t.dtype).view(t.shape))
            off += sz
        return views
    in_src = [(i, k, hosts[n][k]) for i, (n, w) in enumerate(zip(ORDER, work)) for k in w.inputs]
    in_views = pinned_views([t for _, _, t in in_src])
    pinned_in = [{} for _ in work]
    for (i, k, t), v in zip(in_src, in_views):
        v.copy_(t)
        pinned_in[i][k] = v
    out_src = [(i, k, v) for i, w in enumerate(work) for k, v in w.outs.items()]
    out_views = pinned_views([v for _, _, v in out_src])
    pinned_out = [{} for _ in work]
    for (i, k, _), v in zip(out_src, out_views):
        pinned_out[i][k] = v
    h2d = sum(nbytes(t) for p in pinned_in for t in p.values())
    d2h = sum(nbytes(t) for p in pinned_out for t in p.values())

    # Three streams chained by events: op i's inputs go up on s_h2d while op
    # i-1 computes and op i-2's outputs come down on s_d2h (the two copy
    # directions run at the same time).  An upload waits until the previous
    # step's op i has consumed its device inputs; op i waits until the previous
    # step's download of its outputs is done.
    s_h2d = torch.cuda.Stream(device)
    s_d2h = torch.cuda.Stream(device)
    ev_done = [None] * len(work)
    ev_out = [None] * len(work)

    def e2e_step():
        for i, (w, pi, po) in enumerate(zip(work, pinned_in, pinned_out)):
            with torch.cuda.stream(s_h2d):
                if ev_done[i] is not None:
                    s_h2d.wait_event(ev_done[i])
                for k, t in pi.items():
                    w.dev[k].copy_(t, non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_h2d)
            stream.wait_event(e_in)
            if ev_out[i] is not None:
                stream.wait_event(ev_out[i])
            w.call()
            ev_done[i] = torch.cuda.Event()
            ev_done[i].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[i])
                for k, t in po.items():
                    t.copy_(w.outs[k], non_blocking=True)
                ev_out[i] = torch.cuda.Event()
                ev_out[i].record(s_d2h)

    e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    for e in ev_out:
        stream.wait_event(e)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = e0.elapsed_time(e1)

    [total_ms, e2e_ms], [units, e2e_units] = reduce_max_sum(
        [total_ms, e2e_ms], [step_bytes * K, step_bytes * args.e2e_steps], ws)
    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peak, peak_src = measured_peak()
    value = units / (total_ms / 1e3) / 1e9
    ops = {}
    for n, b, ms, iso in zip(ORDER, bytes_per, per_op_ms, iso_ms):
        gbs = b / (ms / 1e3) / 1e9
        med, mn = statistics.median(iso), min(iso)
        o = {"us": ms * 1e3, "min_bytes": b, "gbs": gbs, "frac_of_measured_peak": gbs / peak,
             "frac_nominal": gbs / NOMINAL_HBM_GBS,
             "median_us": med * 1e3, "min_us": mn * 1e3, "mean_us": statistics.fmean(iso) * 1e3,
             "isolated_gbs": b / (med / 1e3) / 1e9,
             "isolated_frac_of_measured_peak": b / (med / 1e3) / 1e9 / peak,
             "isolated_frac_nominal": b / (med / 1e3) / 1e9 / NOMINAL_HBM_GBS}
        r = rows_of(n, hosts[n])
        if r:
            o["rows_per_s"] = r / (ms / 1e3)
        ops[n] = o
    dom_name = ORDER[dom]
    achieved = bytes_per[dom] / (dom_ms / 1e3) / 1e9
    src_hash = kernel_source_hash()
    traffic = NCU_TRAFFIC.get(dom_name) if NCU_TRAFFIC_SOURCE_HASH == src_hash else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded normal/uniform draws and a causal mask; gen/synth.py)",
        "config": {"workload": "one call of each epilogue op per step: " + ", ".join(ORDER),
                   "step_min_bytes": step_bytes, "l2": "inputs larger than L2 (2.8 GB per step; each op "
                   "streams buffers disjoint from the previous op's)", "parallelism": f"replicas x{ws}"},
        "frac_of_measured_peak": value / peak,
        "frac_nominal": value / NOMINAL_HBM_GBS,
        "ops": ops,
        "ops_timing": f"us/gbs/frac_*: in the step, separate loop of {B} steps with an event pair around every "
                      f"op (each record adds ~2 us); median_us/min_us/mean_us/isolated_*: {K_ISOLATED} launches "
                      f"of the op alone, each after an L2 flush leaving only clean lines (event resolution "
                      f"quantises median and minimum)",
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "frac_nominal": achieved / NOMINAL_HBM_GBS, "traffic": traffic,
                     "peak_source": peak_src,
                     "duration_us": dom_ms * 1e3,
                     "duration_source": f"event pair around the op in every {DOM_EVERY}th timed step "
                                        f"({len(dom_steps)} launches), mean"},
        "e2e": {"value": e2e_units / (e2e_ms / 1e3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "pipeline": "uploads, kernels and downloads on three streams, overlapped across ops"},
        "gpu_launches": launches,
        "clocks": clk,
        "kernel_source_hash": src_hash,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(hosts)
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
