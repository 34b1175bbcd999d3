#!/usr/bin/env python3
"""Benchmark: deterministic GEMM throughput on GPT-2-124M linear shapes.

One step = the whole hot path over one synthetic batch: for each GPT-2 layer
shape (K, N) in {(768,2304), (768,768), (768,3072), (3072,768)} at
M = 8192 tokens in bf16, the forward pass Y = X.W + b, dX = dY.W^T and
dW = X^T.dY, on the exact tier (the bits of float64 products summed by
fixed-order KBN, computed from exact integer chunk sums on the tensor cores)
and on the tensor-core tier (tcgen05, fp32 accumulate).  Throughput counts
2*M*K*N useful flops per GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--tiers exact,tc]

Prints one JSON line (rank 0).  Inputs are seeded and synthetic (the pages'
GPT-2 fine-tune needs weights and data that are not available).  L2 is
flushed (a 256 MiB write) between timed steps, outside the timed events.
Under torchrun every rank runs its own replica of the workload (weak
scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("deterministic GEMM GFLOP/s (fwd+dX+dW, GPT-2 shapes) and % of FP64 / "
          "bf16-TC peak")
LAYERS = ((768, 2304), (768, 768), (768, 3072), (3072, 768))
TOKENS = 8192
SEED = 42
PASSES = ("fwd", "dx", "dw")


def _r(x, n=4):
    return None if x is None else float(f"{x:.{n}g}")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------- workload

def pass_dims(pass_, M, K, N):
    """(rows, cols, R) of the pass's output and reduction."""
    return {"fwd": (M, N, K), "dx": (M, K, N), "dw": (K, N, M)}[pass_]


def step_flops(M=TOKENS, layers=LAYERS):
    return sum(2.0 * M * K * N for (K, N) in layers) * len(PASSES)


def make_host_layers(seed, M=TOKENS, layers=LAYERS):
    import seeded_inputs as inputs
    return inputs.gpt2(seed, M=M, layers=layers)


class Workload:
    """Device-resident operands and outputs of one step."""

    def __init__(self, host_layers, device, tiers, only=None):
        import torch
        self.torch = torch
        self.layers = []
        self.tiers = tiers
        self.only = only          # optional set of "tier:pass:KxN" to run alone
        for L in host_layers:
            d = {k: torch.from_numpy(L[k].view(np.int16)).to(device).view(torch.bfloat16)
                 for k in ("X", "W", "b", "dY")}
            M, K, N = L["M"], L["K"], L["N"]
            d.update(M=M, K=K, N=N)
            for t in tiers:
                d[f"Y_{t}"] = torch.empty((M, N), dtype=torch.bfloat16, device=device)
                d[f"dX_{t}"] = torch.empty((M, K), dtype=torch.bfloat16, device=device)
                d[f"dW_{t}"] = torch.empty((K, N), dtype=torch.bfloat16, device=device)
            self.layers.append(d)

    def gemm_list(self, tier):
        """(tier, pass, M, K, N) of every GEMM one step runs on `tier`."""
        out = []
        for d in self.layers:
            for p in PASSES:
                if self.only is None or f"{tier}:{p}:{d['K']}x{d['N']}" in self.only:
                    out.append((tier, p, d["M"], d["K"], d["N"]))
        return out

    def launch_one(self, tier, p, K, N, stream):
        import deterministic_invariant_gemm_fwd_gb300 as cg
        d = next(x for x in self.layers if x["K"] == K and x["N"] == N)
        M, s = d["M"], stream.cuda_stream
        if p == "fwd":
            cg.carbon_gemm_fwd(d[f"Y_{tier}"], d["X"], d["W"], d["b"], M, K, N, "bf16", tier, s)
        elif p == "dx":
            cg.carbon_gemm_dx(d[f"dX_{tier}"], d["dY"], d["W"], M, K, N, "bf16", tier, s)
        else:
            cg.carbon_gemm_dw(d[f"dW_{tier}"], d["X"], d["dY"], M, K, N, "bf16", tier, s)

    def launch(self, tier, stream, events=None):
        """Enqueue the 12 GEMMs of one tier; optional per-launch events."""
        import deterministic_invariant_gemm_fwd_gb300 as cg
        s = stream.cuda_stream
        for d in self.layers:
            M, K, N = d["M"], d["K"], d["N"]
            calls = (
                lambda: cg.carbon_gemm_fwd(d[f"Y_{tier}"], d["X"], d["W"], d["b"], M, K, N, "bf16", tier, s),
                lambda: cg.carbon_gemm_dx(d[f"dX_{tier}"], d["dY"], d["W"], M, K, N, "bf16", tier, s),
                lambda: cg.carbon_gemm_dw(d[f"dW_{tier}"], d["X"], d["dY"], M, K, N, "bf16", tier, s),
            )
            for p, call in zip(PASSES, calls):
                if self.only is not None and f"{tier}:{p}:{K}x{N}" not in self.only:
                    continue
                if events is not None:
                    e0 = self.torch.cuda.Event(enable_timing=True)
                    e1 = self.torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    call()
                    e1.record(stream)
                    events.append((tier, p, M, K, N, e0, e1))
                else:
                    call()


def tc_available():
    import torch
    import deterministic_invariant_gemm_fwd_gb300 as cg
    X = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    try:
        cg.linear_fwd(X, W, None, tier="tc")
        torch.cuda.synchronize()
        return True
    except cg.CarbonError as e:
        if e.status == 2:
            return False
        raise


# ------------------------------------------------------------------- clocks

REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clocks_setting"}


class ClockSampler:
    def __init__(self, index):
        self.proc = None
        self.index = index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], [], set()
        for line in self.out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 4:
                continue
            try:
                s, m = float(parts[0]), float(parts[1])
                bitsv = int(parts[3], 16)
            except ValueError:
                continue
            if bitsv & 0x1:          # idle samples between launches
                continue
            sm.append(s)
            mx.append(m)
            for b, name in REASON_BITS.items():
                if bitsv & b:
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------- fp32 exact tier (FP64 pipe)

def fp32_exact_section(device, stream, fp64_rate, stress=True, repeats=(7, 3)):
    """The fp32 workloads of the exact tier, which run the float64 KBN kernel
    on the FP64 pipe: the toy MLP's nine GEMMs (M = 512 tokens, fwd + dX +
    dW of (K, N) in {(256,512), (512,512), (512,256)}) and the cancellation
    stress dW (65536 tokens, K = 768, N = 3072).  Each is run once untimed,
    then timed `repeats` times with CUDA events on `stream` (the median is
    reported, with the spread).  FP64 utilisation is the
    literal algorithm's floor, 5 FP64 instructions per multiply-add (product,
    sum, two for the exact error, one for the compensation), over the time
    and the measured DFMA rate; the kernel folds the product into the sum's
    FMA and proves whole slices exact, so the figure can pass 1."""
    import torch
    import deterministic_invariant_gemm_fwd_gb300 as cg
    import seeded_inputs as inputs

    def run(calls, macs, reps):
        for c in calls:
            c()
        times = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for c in calls:
                c()
            e1.record(stream)
            stream.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        mac_rate = macs / (ms * 1e-3)
        return {"ms": _r(ms), "ms_min_max": [_r(min(times)), _r(max(times))], "repeats": reps,
                "gflops": _r(2.0 * mac_rate / 1e9),
                "fp64_util_vs_literal": _r(5.0 * mac_rate / fp64_rate)}

    s = stream.cuda_stream
    out = {"unit": "ms, GFLOP/s (2 MNK / t), 5 MNK / (t x measured DFMA rate)",
           "fp64_dfma_rate_tops": _r(fp64_rate / 1e12)}
    calls, macs = [], 0
    torch.cuda.synchronize(device)
    for L in inputs.toy_mlp(SEED):
        M, K, N = L["M"], L["K"], L["N"]
        X, W, b, dY = (torch.from_numpy(L[k]).to(device) for k in ("X", "W", "b", "dY"))
        Y = torch.empty((M, N), dtype=torch.float32, device=device)
        dX = torch.empty((M, K), dtype=torch.float32, device=device)
        dW = torch.empty((K, N), dtype=torch.float32, device=device)
        calls += [lambda Y=Y, X=X, W=W, b=b, M=M, K=K, N=N: cg.carbon_gemm_fwd(Y, X, W, b, M, K, N, "f32", "exact", s),
                  lambda dX=dX, dY=dY, W=W, M=M, K=K, N=N: cg.carbon_gemm_dx(dX, dY, W, M, K, N, "f32", "exact", s),
                  lambda dW=dW, X=X, dY=dY, M=M, K=K, N=N: cg.carbon_gemm_dw(dW, X, dY, M, K, N, "f32", "exact", s)]
        macs += 3 * M * K * N
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        out["toy_mlp_9_gemms"] = run(calls, macs, repeats[0])
        if stress:
            S = inputs.stress_dw(SEED)
            M, K, N = S["M"], S["K"], S["N"]
            X = torch.from_numpy(S["X"]).to(device)
            dY = torch.from_numpy(S["dY"]).to(device)
            dW = torch.empty((K, N), dtype=torch.float32, device=device)
            torch.cuda.synchronize(device)
            out["stress_dw_65536x768x3072"] = run(
                [lambda: cg.carbon_gemm_dw(dW, X, dY, M, K, N, "f32", "exact", s)], M * K * N,
                repeats[1])
            del X, dY, dW
    assert cg.carbon_get_device_status(s) == 0
    return out


# ------------------------------------------- correctly rounded tier (bf16)

def superacc_section(wl, stream, flush, exact_ms, reps=5):
    """The correctly rounded tier (exact sum and bias rounded once) on the
    same 12 GPT-2 GEMMs: one untimed pass, then `reps` passes timed with CUDA
    events on `stream`, L2 flushed before each; the median is reported."""
    import torch
    import deterministic_invariant_gemm_fwd_gb300 as cg
    with torch.cuda.stream(stream):
        wl.launch("superacc", stream)
        stream.synchronize()
        times = []
        for _ in range(reps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            wl.launch("superacc", stream)
            e1.record(stream)
            stream.synchronize()
            times.append(e0.elapsed_time(e1))
    assert cg.carbon_get_device_status(stream.cuda_stream) == 0
    ms = statistics.median(times)
    fl = sum(2.0 * M * K * N for (_, _, M, K, N) in wl.gemm_list("superacc"))
    return {"ms_per_12_gemms": _r(ms), "ms_min_max": [_r(min(times)), _r(max(times))],
            "repeats": reps, "gflops": _r(fl / (ms * 1e-3) / 1e9),
            "vs_exact_tier_time": _r(ms / exact_ms) if exact_ms else None,
            "timing": "CUDA events around the 12 launches, L2 flushed before each pass"}


# ------------------------------------------------------------ CPU baseline

def oracle_sample(host_layers, target_s, threads=None):
    """Time the oracle on a random sample of outputs of every exact-tier GEMM
    of the step.  Returns (useful GFLOP/s, seconds, sampled MACs, threads)."""
    import oracle
    import seeded_inputs as inputs
    threads = threads or oracle.default_threads()

    def run(per_gemm):
        macs, t0 = 0, time.perf_counter()
        for li, L in enumerate(host_layers):
            M, K, N = L["M"], L["K"], L["N"]
            for p, (A, B, bias) in zip(PASSES, ((L["X"], L["W"], L["b"]),
                                               (L["dY"], L["W"], None),
                                               (L["X"], L["dY"], None))):
                rows, cols, R = pass_dims(p, M, K, N)
                ri, ci = inputs.sample_indices(li * 7 + len(p), rows, cols, per_gemm, corners=False)
                oracle.gemm_at(p, "bf16", A, B, bias, M, K, N, ri, ci, threads=threads)
                macs += per_gemm * R
        return macs, time.perf_counter() - t0

    per = 64
    macs, dt = run(per)
    while dt < target_s / 4 and per < 1 << 22:
        per = int(per * min(8.0, max(2.0, target_s / max(dt, 1e-3))))
        macs, dt = run(per)
    return 2.0 * macs / dt / 1e9, dt, macs, threads, per


# -------------------------------------------------------------------- main

def max_over_ranks(ms, pg=None, device=None):
    """The largest of every rank's time (the job ends with its slowest rank);
    the local value when there is no process group."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_gflops(flops_per_rank, world, ms):
    """Whole-job throughput: every rank runs its own replica of the step (weak
    scaling), so the job does world x the flops of one rank in the slowest
    rank's time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e9


# ------------------------------------------------------ recorded DRAM traffic

# The CUDA sources each recorded figure belongs to: the kernel's .cu file and
# the library-internal headers it includes.
KERNEL_SOURCES = {
    "exact_tc_kernel": ("exact_tc.cu", "exact_bf16.cuh", "exact_common.cuh", "tcgen05.cuh",
                        "device_sync.cuh", "carbon_internal.h"),
    "tc_tier": ("tc_gemm.cu", "tcgen05.cuh", "device_sync.cuh", "carbon_internal.h"),
}


def sources_sha256(names, read=None):
    """Hash of the named files of the library's CUDA sources: a traffic figure
    recorded with one hash says nothing about kernels built from other
    sources.  `read(name)` returns a file's bytes (default: the working tree)."""
    import hashlib
    d = os.path.join(ROOT, "deterministic_invariant_gemm_fwd_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(d, name), "rb") as f:
                return f.read()
    h = hashlib.sha256()
    for name in sorted(names):
        h.update(name.encode() + b"\0" + read(name))
    return h.hexdigest()


def recorded_traffic(kernel):
    """DRAM bytes per launch of `kernel` (dram__bytes_read.sum +
    dram__bytes_write.sum, averaged over the launches of one bench step) from
    the ncu summaries in profiles/, when they were taken from the kernel's
    current sources (KERNEL_SOURCES); None otherwise.  A summary records it
    on a line `traffic <kernel> bytes_per_launch=<B> sources_sha256=<hex>`."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d) or kernel not in KERNEL_SOURCES:
        return None
    cur = sources_sha256(KERNEL_SOURCES[kernel])
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name)) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 4 and parts[0] == "traffic" and parts[1] == kernel:
                    kv = dict(p.split("=", 1) for p in parts[2:])
                    if kv.get("sources_sha256") == cur:
                        return int(kv["bytes_per_launch"])
    return None


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reference_arm(args, world, rank):
    """The reference arm: the CPU oracle, timed as it stands, on a bounded
    sample of the same workload in every step."""
    if world > 1 and rank != 0:
        return
    host = make_host_layers(SEED)
    per_step = max(1.0, 90.0 / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        v, dt, macs, threads, per = oracle_sample(host, per_step)
        if i >= args.warmup:
            vals.append((v, dt))
    value = statistics.median(v for v, _ in vals)
    ms = statistics.median(dt for _, dt in vals) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": _r(value), "unit": "GFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": _r(ms), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "gpt2-124m linear layers bf16 M=8192, exact fixed-order KBN "
                               "(CPU oracle on a sample of outputs of every GEMM)",
                   "sample": f"{per} outputs of each of the 12 GEMMs per step"},
        "cpu_baseline": {"value": _r(value), "unit": "GFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": f"{per} outputs x 12 GEMMs, {macs} MACs"},
        "e2e": {"value": _r(value), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tiers", default="auto")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-fp32", action="store_true",
                    help="skip the fp32 exact-tier section (toy MLP and cancellation stress)")
    ap.add_argument("--fp32-only", action="store_true",
                    help="profiling aid: run only the fp32 exact-tier section (toy MLP and, "
                         "unless --no-stress, the cancellation stress dW) and print it")
    ap.add_argument("--no-stress", action="store_true",
                    help="with --fp32-only: leave out the cancellation stress dW")
    ap.add_argument("--no-superacc", action="store_true",
                    help="skip the correctly rounded tier's section (the same 12 GEMMs)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the TC tier eagerly inside the timed region")
    ap.add_argument("--gemm", default=None,
                    help="profiling aid: comma list of tier:pass:KxN to run alone "
                         "(e.g. tc:fwd:768x2304); the JSON line then covers only those")
    args = ap.parse_args()
    world, rank, local = dist_env()

    if args.impl == "reference":
        reference_arm(args, world, rank)
        return

    import torch
    import deterministic_invariant_gemm_fwd_gb300 as cg

    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist

    if args.fp32_only:
        stream = torch.cuda.Stream(device)
        fp64_rate, _ = cg.carbon_measure_fp64_rate(stream.cuda_stream)
        out = fp32_exact_section(device, stream, fp64_rate, stress=not args.no_stress)
        if rank == 0:
            print(json.dumps({"fp32_exact": out}), flush=True)
        return

    tiers = ["exact", "tc"] if args.tiers == "auto" else args.tiers.split(",")
    if "tc" in tiers and not tc_available():
        tiers = [t for t in tiers if t != "tc"]
    host = make_host_layers(SEED + rank)
    only = set(args.gemm.split(",")) if args.gemm else None
    do_superacc = not args.no_superacc and only is None and "exact" in tiers
    wl = Workload(host, device, tiers + (["superacc"] if do_superacc else []), only)
    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def barrier():
        torch.cuda.synchronize(device)
        if pg is not None:
            pg.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for t in tiers:
                wl.launch(t, stream)
        stream.synchronize()
        assert cg.carbon_get_device_status(stream.cuda_stream) == 0

        # The TC tier's twelve ~20-40 us launches are captured once in a CUDA
        # graph and replayed, so host launch overhead does not leak into its
        # timing (the exact tier's ~100 ms launches run eagerly).
        graph, graph_nodes = None, 0
        if "tc" in tiers and not args.no_graph:
            graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(device)
            cap.wait_stream(stream)
            n0 = cg.carbon_debug_launch_count()
            with torch.cuda.graph(graph, stream=cap, capture_error_mode="thread_local"):
                wl.launch("tc", cap)
            graph_nodes = cg.carbon_debug_launch_count() - n0
            stream.wait_stream(cap)
            for _ in range(args.warmup):
                graph.replay()
            stream.synchronize()

        barrier()
        launches0 = cg.carbon_debug_launch_count()
        step_events, kernel_events, graph_events = [], [], []
        if "exact" in tiers:
            cg.carbon_debug_kernel_timing(True)      # events around the exact tier's main kernel
        with ClockSampler(local) as clocks:
            for _ in range(args.steps):
                flush.fill_(1)                                  # L2 flush, outside the events
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for t in tiers:
                    if t == "tc" and graph is not None:
                        g0 = torch.cuda.Event(enable_timing=True)
                        g1 = torch.cuda.Event(enable_timing=True)
                        g0.record(stream)
                        graph.replay()
                        g1.record(stream)
                        graph_events.append((g0, g1))
                    else:
                        wl.launch(t, stream, kernel_events)
                e1.record(stream)
                step_events.append((e0, e1))
            stream.synchronize()
        barrier()
        launches = cg.carbon_debug_launch_count() - launches0 + graph_nodes * len(graph_events)
        assert cg.carbon_get_device_status(stream.cuda_stream) == 0
        main_ms = main_n = main_kg = 0
        phases = None
        repairs = fixups = 0
        if "exact" in tiers:
            main_ms, main_n, main_kg = cg.carbon_debug_kernel_time()
            phases = cg.carbon_debug_exact_phase_time()
            repairs, fixups = cg.carbon_debug_exact_path_counts()
            cg.carbon_debug_kernel_timing(False)

        # per-GEMM kernel time: back-to-back eager launches between two events
        reps = 20
        per_gemm_ms = {}
        for t in tiers:
            if t != "tc":
                continue
            for (_, p, M, K, N) in wl.gemm_list(t):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                wl.launch_one(t, p, K, N, stream)
                a.record(stream)
                for _ in range(reps):
                    wl.launch_one(t, p, K, N, stream)
                b.record(stream)
                stream.synchronize()
                per_gemm_ms[(t, p, K, N)] = a.elapsed_time(b) / reps
        assert cg.carbon_get_device_status(stream.cuda_stream) == 0

    step_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in step_events) / args.steps, pg, device)
    tier_flops = {t: sum(2.0 * M * K * N for (_, _, M, K, N) in wl.gemm_list(t)) for t in tiers}
    flops = sum(tier_flops.values())
    value = whole_job_gflops(flops, world, step_ms)

    tier_info, rooflines = {}, {}
    pk, pk_kind = peaks()
    fp64_rate = None
    for t in tiers:
        fl = tier_flops[t]
        if fl == 0:
            continue
        if t == "tc" and graph is not None:
            ms = sum(g0.elapsed_time(g1) for g0, g1 in graph_events)
            per_gemm = {f"{p}_{K}x{N}": [v] for (tt, p, K, N), v in per_gemm_ms.items() if tt == t}
            how = "CUDA-graph replay of the tier's GEMMs; per-GEMM: 20 back-to-back launches"
        else:
            ev = [e for e in kernel_events if e[0] == t]
            ms = sum(e0.elapsed_time(e1) for *_, e0, e1 in ev)
            per_gemm = {}
            for (_, p, M, K, N, e0, e1) in ev:
                per_gemm.setdefault(f"{p}_{K}x{N}", []).append(e0.elapsed_time(e1))
            how = "CUDA events around every launch"
        fl_all = fl * args.steps
        tier_info[t] = {"ms_per_step": _r(ms / args.steps), "gflops": _r(fl_all / (ms * 1e-3) / 1e9),
                        "timing": how,
                        "ms_per_gemm": {k: _r(sum(v) / len(v)) for k, v in per_gemm.items()}}
        if t == "exact":
            if fp64_rate is None:
                fp64_rate, _ = cg.carbon_measure_fp64_rate(stream.cuda_stream)
            mac_rate = (fl_all / 2.0) / (ms * 1e-3)
            # the dominant kernel runs bf16 digit-plane MMAs on the tensor cores:
            # one plane product = an A plane of 128 rows times a B plane of 64
            # columns over a 256-deep chunk = 2*128*64*256 flops
            kg_flops = main_kg * 2.0 * 128 * 64 * 256
            peak = float(pk["bf16_tflops"])
            achieved = kg_flops / (main_ms * 1e-3) / 1e12 if main_ms > 0 else 0.0
            rooflines["exact"] = {
                "bound": "tensor", "unit": "TFLOP/s", "achieved": _r(achieved), "peak": _r(peak),
                "frac": _r(achieved / peak), "traffic": recorded_traffic("exact_tc_kernel"),
                "traffic_unit": "bytes per launch (ncu, profiles/)", "kernel": "exact_tc_kernel",
                "peak_kind": f"bf16 burst, of {pk_kind}",
                "note": ("algorithmic work = the digit-pair MMAs the kernel issues (counted live: "
                         f"{main_kg} plane products of 2*128*64*256 flops in {main_n} launches), "
                         "over the kernel's own CUDA-event time"),
                "kernel_ms_per_step": _r(main_ms / args.steps),
                "phases_ms_per_step": ({"pre_pass": _r(phases[0] / args.steps),
                                        "exact_tc_kernel": _r(phases[1] / args.steps),
                                        "post_pass": _r(phases[2] / args.steps)}
                                       if phases else None),
                "chunk_repairs_per_step": repairs // args.steps if phases else None,
                "fixups_per_step": fixups // args.steps if phases else None,
                "kernel_share_of_tier": _r(main_ms / ms) if ms > 0 else None,
                "mma_flops_per_useful_flop": _r(kg_flops / fl_all) if fl_all > 0 else None,
                "useful_tflops_kernel": _r(fl_all / (main_ms * 1e-3) / 1e12) if main_ms > 0 else None,
                "useful_gflops_tier": tier_info[t]["gflops"],
                "vs_literal_fp64_floor": _r(mac_rate / (fp64_rate / 5.0)),
                "fp64_dfma_rate_tops": _r(fp64_rate / 1e12)}
        else:
            achieved = fl_all / (ms * 1e-3) / 1e12
            peak = float(pk["bf16_tflops"])
            rooflines["tc"] = {"bound": "tensor", "unit": "TFLOP/s", "achieved": _r(achieved),
                               "peak": _r(peak), "frac": _r(achieved / peak),
                               "traffic": recorded_traffic("tc_tier"),
                               "traffic_unit": "bytes per launch (ncu, profiles/)",
                               "kernel": "tc_gemm_kernel + tc_dw_split_kernel",
                               "peak_kind": f"bf16 burst, of {pk_kind}",
                               "frac_of_sustained": _r(achieved / float(pk.get("bf16_tflops_sustained", peak)))}

    # end to end through the public API: pinned host inputs -> device -> host
    e2e = None
    if not args.no_e2e:
        pinned_in = [{k: torch.from_numpy(L[k].view(np.int16)).pin_memory() for k in ("X", "W", "b", "dY")}
                     for L in host]
        pinned_out = []
        for L in host:
            M, K, N = L["M"], L["K"], L["N"]
            pinned_out.append({f"{n}_{t}": torch.empty(shape, dtype=torch.int16).pin_memory()
                               for t in tiers for n, shape in (("Y", (M, N)), ("dX", (M, K)), ("dW", (K, N)))})
        h2d = sum(v.numel() * 2 for d in pinned_in for v in d.values())
        d2h = sum(v.numel() * 2 for d in pinned_out for v in d.values())
        # Copies overlap the GEMMs, layer by layer: a layer's inputs go up on
        # one copy stream while the previous layer computes, its outputs come
        # down on another while the next one computes.  Every step still moves
        # all of its inputs up and all of its outputs down inside the timed
        # region; events keep a layer's buffers from being overwritten while
        # they are in use (inputs until its GEMMs are done, outputs until
        # they are read back).
        up_s, down_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
        nl = len(wl.layers)
        up_done = [torch.cuda.Event() for _ in range(nl)]
        comp_done = [torch.cuda.Event() for _ in range(nl)]
        down_done = [torch.cuda.Event() for _ in range(nl)]
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up_s.wait_event(e0)
        down_s.wait_event(e0)
        for _ in range(args.steps):
            for li, (d, pi, po) in enumerate(zip(wl.layers, pinned_in, pinned_out)):
                with torch.cuda.stream(up_s):
                    up_s.wait_event(comp_done[li])             # last step's GEMMs have read them
                    for k in ("X", "W", "b", "dY"):
                        d[k].view(torch.int16).copy_(pi[k], non_blocking=True)
                    up_done[li].record(up_s)
                stream.wait_event(up_done[li])
                stream.wait_event(down_done[li])               # last step's outputs are read back
                for t in tiers:
                    for p_ in PASSES:
                        if wl.only is None or f"{t}:{p_}:{d['K']}x{d['N']}" in wl.only:
                            wl.launch_one(t, p_, d["K"], d["N"], stream)
                comp_done[li].record(stream)
                with torch.cuda.stream(down_s):
                    down_s.wait_event(comp_done[li])
                    for t in tiers:
                        for n in ("Y", "dX", "dW"):
                            po[f"{n}_{t}"].copy_(d[f"{n}_{t}"].view(torch.int16), non_blocking=True)
                    down_done[li].record(down_s)
        stream.wait_event(down_done[nl - 1])
        stream.wait_event(up_done[nl - 1])
        e1.record(stream)
        stream.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        e2e_ms = max_over_ranks(e2e_ms, pg, device)
        e2e = {"value": _r(whole_job_gflops(flops, world, e2e_ms)), "unit": "GFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": _r(e2e_ms)}

    superacc = None
    if do_superacc:
        superacc = superacc_section(wl, stream, flush, tier_info.get("exact", {}).get("ms_per_step"))

    fp32 = None
    if "exact" in tiers and not args.no_fp32 and only is None:
        if fp64_rate is None:
            fp64_rate, _ = cg.carbon_measure_fp64_rate(stream.cuda_stream)
        fp32 = fp32_exact_section(device, stream, fp64_rate)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        v, dt, macs, threads, per = oracle_sample(host, args.cpu_seconds)
        cpu = {"value": _r(v), "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{per} outputs of each of the 12 exact-tier GEMMs "
                         f"({macs} MACs, {dt:.1f} s)"}

    if rank == 0:
        dom = "exact" if "exact" in rooflines else "tc"
        if only is not None:
            line_note = {"gemm_filter": sorted(only)}
        else:
            line_note = {}
        line = {
            "metric": METRIC, "value": _r(value), "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": _r(step_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int64" if tiers == ["exact"] else ("f32acc" if tiers == ["tc"] else "int64+f32acc"),
            "data": "synthetic",
            "config": {"workload": "gpt2-124m linear layers, bf16, M=8192 tokens, "
                                   "(K,N) in {(768,2304),(768,768),(768,3072),(3072,768)}, "
                                   "fwd+dX+dW, tiers " + "+".join(tiers),
                       "tiers": tiers, "l2": "flushed between steps (256 MiB write)",
                       "parallelism": f"replicas x{world}", "seed": SEED},
            "tiers": tier_info,
            "roofline": rooflines[dom],
            "rooflines": rooflines,
            "fp32_exact": fp32,
            "superacc": superacc,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            **line_note,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
