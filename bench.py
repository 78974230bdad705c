#!/usr/bin/env python3
"""Benchmark: M=1 quantized GEMV weight GB/s (and us/call) on GB300.

Workload (one "step"): the phi4-14B-shaped 2-bit MatMulNBits decode GEMVs
(bits=2, block 64, fp16 scales, uniform zero point 1.5 passed as a scalar,
fp32 activations and output, M=1) for the five linear shapes qkv (7680x5120),
o (5120x5120), gate_up (35840x5120), down (5120x17920) and lm_head
(100352x5120), one call each.  Inputs are seeded synthetic tensors of those
shapes (the pages measured a real phi4 export that is not available here).

value    = weight bytes (packed codes + fp16 scales) read per step x steps /
           device time, in GB/s, summed over ranks (replicas: every rank runs
           the same step on its own GPU).
Cold weights: every step reads a different replica of all five weight sets;
the replicas total more than three times the 129 MB L2, so no step finds its
weights in L2 (the rotation the pages use for cold timing).

--impl reference times the CPU oracle (the reference arm of the benchmark) on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "M=1 quantized GEMV weight GB/s (% of GB300 HBM peak) and µs/call"
SHAPES = ["qkv", "o", "gate_up", "down", "lm_head"]
BITS, BS, ZP = 2, 64, 1.5
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "mma_gemv_u2_m1_traffic.json")


def weight_bytes(N, K):
    return N * K * BITS // 8 + N * (K // BS) * 2


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("qg_mma_gemv.cu", "qg_device.cuh"):
        with open(os.path.join(ROOT, "gemm_blockwise_dequant_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")


def peaks():
    p = PEAKS_FILE
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------- distributed
def dist_setup(want_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    """Max of a float over ranks (timing only; not on the data path)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------- clocks
class Clocks:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index, log_path=None):
        self.proc = None
        self.gpu = gpu_index
        # raw samples: the --clocks-log file (one per rank), else a temporary file
        self.path = (log_path % gpu_index if log_path and "%d" in log_path else log_path) or \
            os.path.join(tempfile.gettempdir(), "qg_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, loaded_only=False):
        """Median SM clock, maximum clock and the throttle reasons seen.  With
        loaded_only, only samples whose GPU utilisation is at least 50 % count
        (a region that also generates inputs on the host idles in between)."""
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, total = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    mhz = float(parts[1])
                    smax = float(parts[2])
                except ValueError:
                    continue
                total += 1
                if loaded_only:
                    try:
                        if float(parts[9]) < 50.0:
                            continue
                    except (IndexError, ValueError):
                        continue
                sm.append(mhz)
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
               "samples": len(sm)}
        if loaded_only:
            out["samples_total"] = total
            out["samples_rule"] = "samples with GPU utilisation >= 50 %"
        return out


# ------------------------------------------------------------- CPU baseline
class OracleSample:
    """The oracle (as it stands) on a bounded row sample of the workload.

    The five M=1 weight sets are generated once; `run(budget_s)` evaluates an
    evenly spaced row subset of every shape sized from a calibration so that
    one pass takes about `budget_s` seconds (every row when that fits)."""

    def __init__(self):
        import oracle as O
        import workloads as WL

        O.load()
        self.O = O
        self.cores = os.cpu_count() or 1
        self.data = [WL.phi4_u2(s, M=1) for s in SHAPES]
        d = self.data[0]
        self._rows(d, np.arange(64))
        t0 = time.perf_counter()
        self._rows(d, np.arange(512))
        self.per_row_k = (time.perf_counter() - t0) / (512 * d["K"])
        self.full = sum(d["N"] * d["K"] for d in self.data)

    def _rows(self, d, r):
        self.O.qgemm_nbits(d["A"], d["W"], d["scales"], None, M=1, N=d["N"], K=d["K"], bits=BITS, block_size=BS,
                           uniform_zp=ZP, rows=r)

    def run(self, budget_s):
        frac = min(1.0, budget_s / (self.per_row_k * self.full))
        done, secs = 0, 0.0
        for d in self.data:
            r = np.linspace(0, d["N"] - 1, max(16, int(frac * d["N"]))).astype(np.int64)
            t0 = time.perf_counter()
            self._rows(d, r)
            secs += time.perf_counter() - t0
            done += weight_bytes(len(r), d["K"])
        return done, secs, frac


# Arm CPU part numbers of /proc/cpuinfo (implementer 0x41) that this host type may report
ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
             "0xd49": "Arm Neoverse N2"}


def cpu_model():
    """The host CPU's model name from /proc/cpuinfo (an Arm part number is named), else the machine type."""
    import platform

    try:
        with open("/proc/cpuinfo") as f:
            fields = {}
            for line in f:
                key, _, val = line.partition(":")
                fields.setdefault(key.strip(), val.strip())
        if fields.get("model name"):
            return fields["model name"]
        part = fields.get("CPU part", "")
        if part:
            return ARM_PARTS.get(part.lower(), "Arm CPU part " + part) + " (" + platform.machine() + ")"
    except OSError:
        pass
    return platform.machine()


def cpu_baseline(budget_s=12.0, sample=None):
    """Time the oracle on a bounded sample of the workload (about budget_s of CPU work)."""
    S = sample or OracleSample()
    done, secs, passes, frac = 0, 0.0, 0, 0.0
    while secs < 0.8 * budget_s or passes == 0:
        b, t, frac = S.run(min(budget_s, 4.0))
        done, secs, passes = done + b, secs + t, passes + 1
    return {"value": done / secs / 1e9, "unit": "GB/s", "cores": S.cores, "cpu_model": cpu_model(), "kind": "oracle",
            "sample": "%d pass(es) over %.1f%% of the rows of the 5 phi4 shapes, M=1 (%.1f MB of weights, %.1f s, "
                      "OpenMP over rows, %s thread(s))" % (passes, 100 * frac, done / 1e6, secs,
                                                          os.environ.get("OMP_NUM_THREADS", S.cores))}, secs


def oracle_prefill_sample(nrows=64):
    """The oracle on the M=2048 prefill GEMMs, restricted to `nrows` evenly
    spaced activation rows (rows are independent) and every weight row: the
    rows the GPU parity tests check, timed on the host cores (OpenMP)."""
    import oracle as O
    import workloads as WL

    out = {}
    for shape in ("gate_up", "down"):
        d = WL.prefill_u2(shape)
        mrows = np.linspace(0, d["M"] - 1, nrows).astype(np.int64)
        A = np.ascontiguousarray(d["A"][mrows])
        t0 = time.perf_counter()
        O.qgemm_nbits(A, d["W"], d["scales"], None, M=nrows, N=d["N"], K=d["K"], bits=2, block_size=64,
                      uniform_zp=ZP, a_dtype=WL.F16)
        dt = time.perf_counter() - t0
        out["prefill_u2_%s_m2048" % shape] = {"seconds": round(dt, 3), "activation_rows": nrows,
                                              "tflops": round(2.0 * nrows * d["N"] * d["K"] / dt / 1e12, 6)}
    return out


def oracle_single_thread(budget_s=8.0):
    """cpu_baseline with one OpenMP thread, in a child process (the thread count
    is fixed when the oracle library starts its runtime)."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-timing", str(budget_s)], env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d["cores"] = 1
    return d


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on this host's cores.

    Each step is one pass of the oracle over a row sample of the five shapes,
    sized so that the whole run stays near a minute of CPU work.  Under
    torchrun only rank 0 runs it."""
    if rank != 0:
        return 0
    S = OracleSample()
    per_step = max(0.05, 60.0 / max(1, args.steps))
    for _ in range(args.warmup):
        S.run(min(per_step, 0.5))
    done, secs, frac = 0, 0.0, 0.0
    for _ in range(args.steps):
        b, t, frac = S.run(per_step)
        done, secs = done + b, secs + t
    v = done / secs / 1e9
    sample = ("%d steps, each one pass over %.2f%% of the rows of the 5 phi4 shapes, M=1 (%.1f MB of weights in "
              "%.1f s, OpenMP over rows)" % (args.steps, 100 * frac, done / 1e6, secs))
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "phi4-14B u2 decode GEMVs (qkv 7680x5120, o 5120x5120, gate_up 35840x5120, "
                                   "down 5120x17920, lm_head 100352x5120), M=1, bits=2, block 64, fp16 scales, "
                                   "uniform zp 1.5, fp32 A/Y; CPU oracle on a row sample"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": S.cores, "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_ours(args, world, rank, local):
    import torch

    import gemm_blockwise_dequant_gb300 as qg
    import workloads as WL

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    qg.lib()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)

    # weights: one seeded set per shape, replicated so the rotation exceeds 3x L2
    per_step = sum(weight_bytes(*WL.PHI4_SHAPES[s]) for s in SHAPES)
    reps = max(2, -(-3 * L2_BYTES // per_step))
    data = {}
    for s in SHAPES:
        d = WL.phi4_u2(s, M=1, seed=0)
        W = torch.from_numpy(d["W"]).to(dev)
        S = torch.from_numpy(d["scales"].view(np.int16)).to(dev).view(torch.float16)
        A = torch.from_numpy(d["A"]).to(dev)
        data[s] = dict(N=d["N"], K=d["K"], W=[W] + [W.clone() for _ in range(reps - 1)],
                       S=[S] + [S.clone() for _ in range(reps - 1)], A=A,
                       Y=torch.empty(1, d["N"], device=dev), A_host=torch.from_numpy(d["A"]))
    ws_need = max(qg.qgemm_workspace_bytes(0, 1, data[s]["N"], data[s]["K"], BITS, BS) for s in SHAPES)
    ws = torch.empty(max(ws_need, 16), dtype=torch.uint8, device=dev)

    def call(s, r):
        e = data[s]
        qg.qgemm_nbits_uniform_zp(e["A"], e["W"][r], e["S"][r], ZP, e["Y"], bits=BITS, block_size=BS,
                                  workspace=ws, stream=stream)

    def step(r):
        for s in SHAPES:
            call(s, r)

    # CUDA graphs of up to --graph-steps consecutive steps (each step on the next
    # weight replica), like a decode graph that chains the GEMVs of several
    # layers; the library is capture-safe (no sync, no allocation)
    chain = max(1, args.graph_steps)
    graphs = {}

    def graph(n, first):
        key = (n, first % reps)
        if key not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    step((first + i) % reps)
            graphs[key] = g
        return graphs[key]

    def run_steps(n, first):
        done = 0
        while done < n:
            c = min(chain, n - done)
            graph(c, first + done).replay()
            done += c

    with torch.cuda.stream(stream):
        for r in range(reps):
            step(r)
        stream.synchronize()
        for first, n in ((0, args.warmup), (args.warmup, args.steps)):
            for j in range(0, n, chain):
                graph(min(chain, n - j), first + j)
    torch.cuda.synchronize()

    # ---- timed region: K steps (5 GEMV launches each) as graph replays
    with torch.cuda.stream(stream):
        run_steps(args.warmup, 0)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local, getattr(args, "clocks_log", None)) as clk:
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            run_steps(args.steps, args.warmup)
            end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    step_ms = start.elapsed_time(end) / args.steps
    step_ms = max_over_ranks(step_ms, world)
    clocks = clk.summary()

    # ---- per-launch duration of each shape: a graph of back-to-back launches of
    # that shape, each on its own weight replica (more than 3x L2 per graph, so
    # every launch reads cold weights), timed with events around the replay
    per_shape_us, isolated_us = {}, {}
    dom_bytes, dom_time = 0, 0.0
    for s in SHAPES:
        e = data[s]
        nb = weight_bytes(*WL.PHI4_SHAPES[s])
        n = max(reps, -(-3 * L2_BYTES // nb), 8)
        Ws = e["W"] + [e["W"][0].clone() for _ in range(n - len(e["W"]))]
        Ss = e["S"] + [e["S"][0].clone() for _ in range(n - len(e["S"]))]

        def one(i):
            qg.qgemm_nbits_uniform_zp(e["A"], Ws[i], Ss[i], ZP, e["Y"], bits=BITS, block_size=BS,
                                      workspace=ws, stream=stream)

        with torch.cuda.stream(stream):
            for i in range(n):
                one(i)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    one(i)
            g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(3):
                g.replay()
            b.record(stream)
            # the same launches one at a time, events around each (launch latency included)
            evs = []
            for i in range(8):
                a1, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a1.record(stream)
                one(i % n)
                b1.record(stream)
                evs.append((a1, b1))
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (3 * n)
        per_shape_us[s] = us
        isolated_us[s] = statistics.median(x.elapsed_time(y) * 1e3 for x, y in evs)
        del Ws, Ss, g
        if WL.PHI4_SHAPES[s][1] == 5120:  # the K=5120 launches share one kernel instantiation
            dom_bytes += nb
            dom_time += us

    # ---- end to end through the API with host buffers: every step copies its
    # inputs (the five activation rows, one pinned host buffer) to the device,
    # runs the 5 GEMVs eagerly and reads its results (the five output rows, one
    # device buffer) back to pinned host memory
    Ks = [data[s]["K"] for s in SHAPES]
    Ns = [data[s]["N"] for s in SHAPES]
    A_host = torch.cat([data[s]["A_host"].reshape(-1) for s in SHAPES]).pin_memory()
    Y_host = torch.empty(sum(Ns)).pin_memory()
    A_all = torch.empty(sum(Ks), device=dev)
    Y_all = torch.empty(sum(Ns), device=dev)
    A_v = dict(zip(SHAPES, (v.view(1, -1) for v in torch.split(A_all, Ks))))
    Y_v = dict(zip(SHAPES, (v.view(1, -1) for v in torch.split(Y_all, Ns))))
    h2d = A_host.numel() * 4
    d2h = Y_host.numel() * 4

    def step_e2e(r):
        A_all.copy_(A_host, non_blocking=True)
        for s in SHAPES:
            e = data[s]
            qg.qgemm_nbits_uniform_zp(A_v[s], e["W"][r], e["S"][r], ZP, Y_v[s], bits=BITS, block_size=BS,
                                      workspace=ws, stream=stream)
        Y_host.copy_(Y_all, non_blocking=True)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step_e2e(i % reps)
        stream.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            step_e2e(i % reps)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    for s in SHAPES:  # the e2e outputs are the device path's (same inputs, same weights)
        if not torch.equal(Y_v[s], data[s]["Y"]):
            raise SystemExit("bench.py: end-to-end output differs from the device-resident run (%s)" % s)

    peak, peak_kind = peaks()
    value = world * per_step / (step_ms * 1e-3) / 1e9
    achieved = dom_bytes / (dom_time * 1e-6) / 1e9
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_source_hash") == kernel_source_hash():
            traffic = tr.get("bytes_per_launch")
    # ---- every configuration of the hot path (one GPU): the suite's timing of
    # each, with its own clock record over the loaded samples
    configs, cclocks = None, None
    if world == 1 and not args.no_configs:
        with Clocks(local, None) as clk2:
            recs = run_suite(groups=CONFIG_GROUPS, echo=False)
        configs = {r.pop("config"): r for r in recs}
        cclocks = clk2.summary(loaded_only=True)
    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb, _ = cpu_baseline()
        cb["single_thread"] = oracle_single_thread()
        cb["prefill_sample"] = oracle_prefill_sample()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "phi4-14B u2 decode GEMVs (qkv 7680x5120, o 5120x5120, gate_up 35840x5120, "
                               "down 5120x17920, lm_head 100352x5120), M=1, bits=2, block 64, fp16 scales, "
                               "uniform zp 1.5, fp32 A/Y",
                   "weight_bytes_per_step": per_step, "l2": "weights rotate over %d replicas (%.0f MB > 3x L2)" % (
                       reps, reps * per_step / 1e6),
                   "step": "the 5 GEMV launches; steps replayed as CUDA graphs of up to %d steps" % chain,
                   "pct_of_hbm_peak": round(100 * value / world / peak, 1),
                   "us_per_call": {s: round(v, 2) for s, v in per_shape_us.items()},
                   "us_per_call_isolated": {s: round(v, 2) for s, v in isolated_us.items()},
                   "per_launch": "us_per_call: graph of back-to-back launches of one shape, cold weights; "
                                 "us_per_call_isolated: one launch between two events",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "mma_gemv_kernel u2 M=1 (K=5120 launches: qkv, o, gate_up, lm_head)",
                     "peak_kind": peak_kind},
        "e2e": {"value": round(world * per_step / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": len(SHAPES) * args.steps,
        "clocks": clocks,
        "cpu_baseline": cb,
    }
    if configs is not None:
        line["config"]["configs"] = configs
        line["config"]["configs_clocks"] = cclocks
        line["config"]["configs_method"] = (
            "each configuration through the public API after the timed steps: a CUDA graph of back-to-back calls "
            "whose weights rotate over copies (QMoE: disjoint expert sets) totalling more than 3x L2, replayed for "
            "about 60 ms; us_per_call = event time / calls; gbs over weight bytes (codes + block parameters); "
            "hbm_frac / tensor_frac against the measured copy / bf16 peaks; prefill and ragged reuse one weight set")
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- config suite
# the groups the benchmark line carries (the N sweep only runs under --suite)
CONFIG_GROUPS = ("tiny_u4", "phi4_u2", "nf4", "qmoe", "prefill", "f32_large_m", "phi4_u8", "packed_zp", "ragged",
                 "gather")


def run_suite(only=None, groups=None, echo=True):
    """Time every configuration of the hot path through the public API (one
    JSON line each): tiny u4 GEMV; the phi4 u2 decode shapes at M=1 and M=4;
    8-bit codes on two of those shapes;
    the NF4 codebook shapes at M=1, 4, 16, 64 (bf16 activations); the QMoE
    decode (128 experts, top-8, 2880/2880, u4 block 32) with and without zero
    points, with fp16 and with int8 activations; the two M=2048 prefill GEMMs; the
    phi4 gate_up projection with fp32 activations at M=64 and M=2048; the
    ragged expert GEMM of a 128-expert top-8 2048/768 layer over a 2048-token prompt; an N sweep
    around two decode shapes (partition-camping outliers);
    the block-quantized embedding gather
    (u4, u8, E4M3 tables).  Each figure is the mean over a CUDA
    graph of R back-to-back calls whose weights rotate over copies (or expert
    sets) totalling more than three times the L2, so every call reads cold
    weights; prefill is compute-bound and reuses one weight set.

    `groups` restricts the run to those groups; every record is also returned
    (a list of dicts), and printed as one JSON line when `echo` is set."""
    import torch

    import gemm_blockwise_dequant_gb300 as qg
    import workloads as WL

    if not torch.cuda.is_available():
        raise SystemExit("bench.py --suite: no CUDA device (the library has no CPU path)")
    qg.lib()
    peak_gbs, _ = peaks()
    tf_peak = None
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            tf_peak = json.load(f).get("bf16_tflops")
    st = torch.cuda.Stream()
    dev = torch.device("cuda")

    def t16(a, dt):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(dt)

    def timed(call, n):
        with torch.cuda.stream(st):
            for i in range(min(n, 4)):
                call(i)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for i in range(n):
                    call(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            g.replay()
            b.record(st)
            st.synchronize()
            # enough replays for about 60 ms of back-to-back work (at least 5)
            reps = int(min(2000, max(5, 60.0 / max(1e-3, a.elapsed_time(b)))))
            a.record(st)
            for _ in range(reps):
                g.replay()
            b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * n)

    def emit(name, us, nbytes=None, flops=None, **extra):
        line = {"config": name, "us_per_call": round(us, 2)}
        if nbytes:
            gbs = nbytes / (us * 1e-6) / 1e9
            line.update(weight_bytes=int(nbytes), gbs=round(gbs, 1), hbm_frac=round(gbs / peak_gbs, 4))
        if flops:
            tfs = flops / (us * 1e-6) / 1e12
            line.update(tflops=round(tfs, 1))
            if tf_peak:
                line.update(tensor_frac=round(tfs / tf_peak, 4))
        line.update(extra)
        records.append(line)
        if echo:
            print(json.dumps(line), flush=True)

    def reps_for(nbytes):
        return max(2, -(-3 * L2_BYTES // max(1, nbytes)))

    def want(group):
        if groups is not None:
            return group in groups
        return only is None or only in group

    records = []

    # tiny u4 (M=1, 128 x 256, block 64, zero-point tensor)
    if want("tiny_u4"):
        d = WL.tiny_u4()
        A, W, S, Z = torch.from_numpy(d["A"]).to(dev), torch.from_numpy(d["W"]).to(dev), t16(d["scales"], torch.float16), \
            t16(d["zero_points"], torch.float16)
        Y = torch.empty(1, 128, device=dev)
        emit("tiny_u4_m1", timed(lambda i: qg.qgemm_nbits(A, W, S, Z, Y, bits=4, block_size=64, stream=st), 50))

    # phi4 u2 decode, M = 1 and 4
    if want("phi4_u2"):
        for M in (1, 4):
            for shape in SHAPES:
                d = WL.phi4_u2(shape, M=M)
                wb = d["W"].nbytes + d["scales"].nbytes
                r = reps_for(wb)
                Ws = [torch.from_numpy(d["W"]).to(dev) for _ in range(r)]
                Ss = [t16(d["scales"], torch.float16) for _ in range(r)]
                A = torch.from_numpy(d["A"]).to(dev)
                Y = torch.empty(M, d["N"], device=dev)
                ws = torch.empty(max(16, qg.qgemm_workspace_bytes(0, M, d["N"], d["K"], 2, 64)), dtype=torch.uint8, device=dev)
                us = timed(lambda i: qg.qgemm_nbits_uniform_zp(A, Ws[i % r], Ss[i % r], ZP, Y, bits=2, block_size=64,
                                                               workspace=ws, stream=st), 2 * r)
                emit("phi4_u2_%s_m%d" % (shape, M), us, nbytes=wb)
                del Ws, Ss

    # 8-bit MatMulNBits codes on two of the phi4 shapes, M = 1
    if want("phi4_u8"):
        for shape in ("qkv", "lm_head"):
            d = WL.phi4_u8(shape, M=1)
            wb = d["W"].nbytes + d["scales"].nbytes
            r = reps_for(wb)
            Ws = [torch.from_numpy(d["W"]).to(dev) for _ in range(r)]
            S = t16(d["scales"], torch.float16)
            A = torch.from_numpy(d["A"]).to(dev)
            Y = torch.empty(1, d["N"], device=dev)
            ws = torch.empty(max(16, qg.qgemm_workspace_bytes(0, 1, d["N"], d["K"], 8, 64)), dtype=torch.uint8, device=dev)
            us = timed(lambda i: qg.qgemm_nbits_uniform_zp(A, Ws[i % r], S, 128.0, Y, bits=8, block_size=64,
                                                           workspace=ws, stream=st), 2 * r)
            emit("phi4_u8_%s_m1" % shape, us, nbytes=wb)
            del Ws

    # u4 block 32 with packed integer zero points, and the same GEMV with an fp16 zero-point tensor
    if want("packed_zp"):
        for shape in ("qkv", "lm_head"):
            N, K = WL.PHI4_SHAPES[shape]
            d = WL.packed_zp(N, K, M=1, bits=4, block_size=32)
            z16 = WL.fp16_uniform_int(WL.rng(1), (N, K // 32), 0, 15)
            A = torch.from_numpy(d["A"]).to(dev)
            Y = torch.empty(1, N, device=dev)
            for packed in (True, False):
                zb = d["zp_packed"] if packed else z16
                wb = d["W"].nbytes + d["scales"].nbytes + zb.nbytes
                r = reps_for(wb)
                Ws = [torch.from_numpy(d["W"]).to(dev) for _ in range(r)]
                Ss = [t16(d["scales"], torch.float16) for _ in range(r)]
                Zs = [torch.from_numpy(zb).to(dev) if packed else t16(zb, torch.float16) for _ in range(r)]
                if packed:
                    ws = torch.empty(max(16, qg.qgemm_nbits_packed_zp_workspace_bytes(0, 1, N, K, 4, 32)),
                                     dtype=torch.uint8, device=dev)
                    call = lambda i: qg.qgemm_nbits_packed_zp(A, Ws[i % r], Ss[i % r], Zs[i % r], Y, bits=4,
                                                              block_size=32, workspace=ws, stream=st)
                else:
                    ws = torch.empty(max(16, qg.qgemm_workspace_bytes(0, 1, N, K, 4, 32)), dtype=torch.uint8,
                                     device=dev)
                    call = lambda i: qg.qgemm_nbits(A, Ws[i % r], Ss[i % r], Zs[i % r], Y, bits=4, block_size=32,
                                                    workspace=ws, stream=st)
                emit("u4_bs32_%s_zp_%s_m1" % ("packed" if packed else "fp16", shape), timed(call, 2 * r), nbytes=wb)
                del Ws, Ss, Zs

    # fp32 activations at prefill sizes: the phi4 gate_up projection, M = 64 and 2048
    if want("f32_large_m"):
        d = WL.phi4_u2("gate_up", M=2048)
        W, S = torch.from_numpy(d["W"]).to(dev), t16(d["scales"], torch.float16)
        for M in (64, 2048):
            A = torch.from_numpy(np.ascontiguousarray(d["A"][:M])).to(dev)
            Y = torch.empty(M, d["N"], device=dev)
            ws = torch.empty(max(16, qg.qgemm_workspace_bytes(0, M, d["N"], d["K"], 2, 64)), dtype=torch.uint8,
                             device=dev)
            us = timed(lambda i: qg.qgemm_nbits_uniform_zp(A, W, S, ZP, Y, bits=2, block_size=64, workspace=ws,
                                                           stream=st), 2)
            emit("phi4_u2_gate_up_f32_m%d" % M, us, nbytes=d["W"].nbytes + d["scales"].nbytes,
                 flops=2.0 * M * d["N"] * d["K"])

    # NF4 codebook, bf16 activations
    if want("nf4"):
        for ad, tdt, tag in ((2, torch.bfloat16, "bf16"), (1, torch.float16, "f16")):
            for shape in ("square", "gqa_kv", "up", "down"):
                for M in (1, 4, 16, 64):
                    d = WL.nf4(shape, M=M, a_dtype=ad)
                    wb = d["W"].nbytes + d["absmax"].nbytes
                    r = reps_for(wb)
                    Ws = [torch.from_numpy(d["W"]).to(dev) for _ in range(r)]
                    am = torch.from_numpy(d["absmax"]).to(dev)
                    cb = torch.from_numpy(d["codebook"]).to(dev)
                    A = t16(d["A"], tdt)
                    Y = torch.empty(M, d["N"], device=dev, dtype=tdt)
                    ws = torch.empty(max(16, qg.qgemm_workspace_bytes(ad, M, d["N"], d["K"], 4, 64)), dtype=torch.uint8,
                                     device=dev)
                    us = timed(lambda i: qg.qgemm_codebook4(A, Ws[i % r], cb, am, Y, block_size=64, workspace=ws,
                                                            stream=st), 2 * r)
                    emit("nf4_%s_%s_%dx%d_m%d" % (tag, shape, d["N"], d["K"], M), us, nbytes=wb,
                         flops=2.0 * M * d["N"] * d["K"])
                    del Ws

    # NF4 with a nested (double-quantized) absmax, M = 1, bf16: the expansion plus the codebook GEMV;
    # bytes = codes + 8-bit absmax codes + second-level scales
    if want("nf4"):
        d = WL.nf4_nested("square", M=1, a_dtype=2)
        wb = d["W"].nbytes + d["absmax_q"].nbytes + d["absmax2"].nbytes
        r = reps_for(wb)
        Ws = [torch.from_numpy(d["W"]).to(dev) for _ in range(r)]
        qa = torch.from_numpy(d["absmax_q"]).to(dev)
        tab, a2 = torch.from_numpy(d["absmax_table"]).to(dev), torch.from_numpy(d["absmax2"]).to(dev)
        cb = torch.from_numpy(d["codebook"]).to(dev)
        A = t16(d["A"], torch.bfloat16)
        Y = torch.empty(1, d["N"], device=dev, dtype=torch.bfloat16)
        ws = torch.empty(qg.qgemm_codebook4_nested_workspace_bytes(2, 1, d["N"], d["K"], 64), dtype=torch.uint8,
                         device=dev)
        us = timed(lambda i: qg.qgemm_codebook4_nested(A, Ws[i % r], cb, qa, tab, a2, d["absmax_offset"], Y,
                                                       block_size=64, workspace=ws, stream=st), 2 * r)
        emit("nf4_nested_square_4096x4096_m1", us, nbytes=wb)
        del Ws

    # QMoE decode: rotate over disjoint expert sets (128 experts, top-8)
    if want("qmoe"):
        for with_zp in (False, True):
            d = WL.qmoe(with_zp=with_zp)
            h = lambda a: None if a is None else t16(a, torch.float16)
            kw = dict(num_experts=d["num_experts"], fc1_w=torch.from_numpy(d["fc1_w"]).to(dev), fc1_scales=h(d["fc1_scales"]),
                      fc1_zp=h(d["fc1_zp"]), fc1_bias=h(d["fc1_bias"]), fc2_w=torch.from_numpy(d["fc2_w"]).to(dev),
                      fc2_scales=h(d["fc2_scales"]), fc2_zp=h(d["fc2_zp"]), fc2_bias=h(d["fc2_bias"]), bits=4, block_size=32)
            k, E = d["k"], d["num_experts"]
            sets = [torch.arange(j * k, (j + 1) * k, dtype=torch.int32, device=dev) for j in range(E // k)]
            wts = torch.from_numpy(d["weights"]).to(dev)
            x = h(d["x"])
            y = torch.empty(d["hidden"], dtype=torch.float16, device=dev)
            ws = torch.empty(qg.qmoe_decode_workspace_bytes(k, d["hidden"], d["inter"]), dtype=torch.uint8, device=dev)
            per_expert = (d["fc1_w"][0].nbytes + d["fc1_scales"][0].nbytes + d["fc2_w"][0].nbytes + d["fc2_scales"][0].nbytes
                          + (d["fc1_zp"][0].nbytes + d["fc2_zp"][0].nbytes if with_zp else 0))
            us = timed(lambda i: qg.qmoe_decode_fused(x, sets[i % len(sets)], wts, y=y, workspace=ws, stream=st, **kw),
                       len(sets))
            emit("qmoe_top8_2880_u4_bs32_%s" % ("zp" if with_zp else "nozp"), us, nbytes=k * per_expert)
            us = timed(lambda i: qg.qmoe_decode_fused_dp4a(x, sets[i % len(sets)], wts, y=y, workspace=ws, stream=st,
                                                           **kw), len(sets))
            emit("qmoe_dp4a_top8_2880_u4_bs32_%s" % ("zp" if with_zp else "nozp"), us, nbytes=k * per_expert)
            del kw

    # prefill u2, M = 2048, fp16 activations, fp32 out
    if want("prefill"):
        for shape in ("gate_up", "down"):
            d = WL.prefill_u2(shape, M=2048)
            A, W, S = t16(d["A"], torch.float16), torch.from_numpy(d["W"]).to(dev), t16(d["scales"], torch.float16)
            Y = torch.empty(d["M"], d["N"], device=dev)
            ws = torch.empty(max(16, qg.qgemm_workspace_bytes(1, d["M"], d["N"], d["K"], 2, 64)), dtype=torch.uint8, device=dev)
            us = timed(lambda i: qg.qgemm_nbits_uniform_zp(A, W, S, ZP, Y, bits=2, block_size=64, workspace=ws, stream=st), 4)
            emit("prefill_u2_%s_m2048" % shape, us, flops=2.0 * d["M"] * d["N"] * d["K"])
            del A, W, S, Y

    # ragged expert GEMM: fc1 (1536 x 2048 per expert) of the 128-expert top-8 "2048 / 768" MoE layer over a
    # 2048-token prompt (16384 rows, ~128 per expert), u4 block 32, fp16 in and out; one weight set
    # (compute-bound)
    if want("ragged"):
        for NK in ((1536, 2048), (5760, 2880)):  # the 2048/768 layer; a 2880-wide layer (90 blocks per row)
            d = WL.ragged(N=NK[0], K=NK[1])
            X = t16(d["X"], torch.float16)
            W = torch.from_numpy(d["W"]).to(dev)
            S = t16(d["scales"], torch.float16)
            T = int(d["offsets"][-1])
            Y = torch.empty(T, d["N"], dtype=torch.float16, device=dev)
            off = d["offsets"]
            ws = torch.empty(max(16, qg.qmoe_ragged_mm_workspace_bytes(1, off, d["N"], d["K"], 4, 32)),
                             dtype=torch.uint8, device=dev)
            us = timed(lambda i: qg.qmoe_ragged_mm(X, off, W, S, None, Y, bits=4, block_size=32, workspace=ws,
                                                   stream=st), 4)
            emit("ragged_fc1_128x%dx%d_u4_bs32_tokens2048_top8" % NK, us, flops=2.0 * T * d["N"] * d["K"],
                 rows=T, experts_min_rows=int(np.diff(off).min()), experts_max_rows=int(np.diff(off).max()))
            if NK == (1536, 2048):  # the same with the offsets in device memory (no host copy of them)
                off_d = torch.from_numpy(np.asarray(off, np.int64)).to(dev)
                wsd = torch.empty(qg.qmoe_ragged_mm_device_offsets_workspace_bytes(len(off) - 1), dtype=torch.uint8,
                                  device=dev)
                us = timed(lambda i: qg.qmoe_ragged_mm_device_offsets(X, off_d, W, S, None, Y, bits=4, block_size=32,
                                                                      workspace=wsd, stream=st), 4)
                emit("ragged_fc1_128x%dx%d_u4_bs32_tokens2048_top8_device_offsets" % NK, us,
                     flops=2.0 * T * d["N"] * d["K"], rows=T)
            del X, W, S, Y

    # N sweep around the decode shapes (u2 M=1, K = 5120 around qkv's N and K = 17920 around down's N, steps
    # of 64 rows): a row count that maps badly onto the HBM channels would show as an outlier against its
    # neighbours (more than 15 % below the median GB/s of the two on each side).
    if want("nsweep"):
        for K, centre in ((5120, 7680), (17920, 5120)):
            pts = []
            for N in range(centre - 8 * 64, centre + 8 * 64 + 1, 64):
                g = np.random.Generator(np.random.PCG64(N))
                W0 = g.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
                S0 = g.uniform(0.01, 0.05, size=(N, K // 64)).astype(np.float16).view(np.int16)
                wb = W0.nbytes + S0.nbytes
                r = reps_for(wb)
                Ws = [torch.from_numpy(W0).to(dev) for _ in range(r)]
                S = torch.from_numpy(S0).to(dev).view(torch.float16)
                A = torch.from_numpy(g.standard_normal((1, K)).astype(np.float32)).to(dev)
                Y = torch.empty(1, N, device=dev)
                ws = torch.empty(max(16, qg.qgemm_workspace_bytes(0, 1, N, K, 2, 64)), dtype=torch.uint8, device=dev)
                us = timed(lambda i: qg.qgemm_nbits_uniform_zp(A, Ws[i % r], S, ZP, Y, bits=2, block_size=64,
                                                               workspace=ws, stream=st), 2 * r)
                pts.append((N, us, wb / (us * 1e-6) / 1e9))
                del Ws
            for j, (N, us, gbs) in enumerate(pts):
                nbr = [q[2] for q in pts[max(0, j - 2):j] + pts[j + 1:j + 3]]
                med = statistics.median(nbr)
                emit("nsweep_u2_m1_k%d_n%d" % (K, N), us, nbytes=N * K // 4 + N * (K // 64) * 2,
                     neighbour_median_gbs=round(med, 1), outlier=bool(gbs < 0.85 * med))

    # block-quantized embedding gather: phi4 table 100352 x 5120, block 32, 2048 token ids, fp16 out.
    # 16 index sets, each drawn from its own sixteenth of the vocabulary, so a row read by one call
    # is not read again for 15 calls (over 3x the L2 of traffic in between).
    if want("gather"):
        for fmt, name in ((1, "u4"), (2, "u8"), (3, "e4m3")):
            d = WL.embedding(fmt)
            n, D, V, bs = d["n"], d["D"], d["V"], d["block_size"]
            W = torch.from_numpy(d["W"]).to(dev)
            S = t16(d["scales"], torch.float16)
            Z = None if d["zero_points"] is None else t16(d["zero_points"], torch.float16)
            g = np.random.Generator(np.random.PCG64(1))
            sets = [torch.from_numpy(g.integers(j * (V // 16), (j + 1) * (V // 16), size=n, dtype=np.int64)).to(dev)
                    for j in range(16)]
            Y = torch.empty(n, D, dtype=torch.float16, device=dev)
            nbytes = n * (8 + D * WL.EMBED_BITS[fmt] // 8 + (D // bs) * 2 * (1 if Z is None else 2) + D * 2)
            us = timed(lambda i: qg.qg_gather_block_quantized(sets[i % 16], W, S, Z, Y, w_format=fmt, block_size=bs,
                                                              stream=st), 32)
            emit("gather_%s_phi4_embed_n2048_bs32_f16" % name, us, nbytes=nbytes, bytes_include="indices, codes, "
                 "scales, zero points, fp16 output")
            del W, S, Z, Y
    return records


# ------------------------------------------------------------- ncu probes
def run_probe(name):
    """Small fixed workloads for profiler captures (no timing, no JSON line).

    gemv_k5120   3 warm-up calls, then one call, of each K=5120 phi4 u2 M=1 shape
                 (qkv, o, gate_up, lm_head): the launches of the dominant kernel
    gemv_lm_head 4 calls of the lm_head shape (100352 x 5120, u2, M=1)
    gemv_down    4 calls of the down shape (5120 x 17920, u2, M=1)
    tc_prefill   4 calls of a prefill-sized u2 GEMM on the tensor cores
                 (M=2048, N=K=5120, fp16 activations, fp32 out)
    tc_prefill_gate_up, tc_prefill_down
                 3 calls of the phi4-14B prefill GEMMs (M=2048; 35840 x 5120,
                 5120 x 17920)
    tc_nf4_m64   4 calls of the NF4 codebook GEMM 14336 x 4096 at M=64 (bf16, tensor cores)
    qmoe         4 calls of the 128-expert top-8 2880/2880 block-32 QMoE decode
    qmoe_dp4a    the same with int8 activations
    ragged       4 calls of the ragged expert GEMM (128 experts, 16384 rows, 1536 x 2048 u4 block 32)
    gather       4 calls of the u4 embedding gather (100352 x 5120 table, block 32,
                 2048 token ids, fp16 out)
    """
    import torch

    import gemm_blockwise_dequant_gb300 as qg
    import workloads as WL

    def nbits(d):
        ad = d["a_dtype"]
        A = torch.from_numpy(d["A"] if ad == 0 else d["A"].view(np.int16)).cuda()
        if ad == 1:
            A = A.view(torch.float16)
        W = torch.from_numpy(d["W"]).cuda()
        S = torch.from_numpy(d["scales"].view(np.int16)).cuda().view(torch.float16)
        Y = torch.empty(d["M"], d["N"], device="cuda")
        ws = torch.empty(max(16, qg.qgemm_workspace_bytes(ad, d["M"], d["N"], d["K"], 2, 64)), dtype=torch.uint8,
                         device="cuda")
        return lambda: qg.qgemm_nbits_uniform_zp(A, W, S, ZP, Y, bits=2, block_size=64, workspace=ws)

    if name == "gemv_k5120":
        calls = [nbits(WL.phi4_u2(s, M=1)) for s in ("qkv", "o", "gate_up", "lm_head")]
        for c in calls:
            for _ in range(3):
                c()
        for c in calls:
            c()
    elif name in ("gemv_lm_head", "gemv_down"):
        c = nbits(WL.phi4_u2(name[5:], M=1))
        for _ in range(4):
            c()
    elif name == "tc_prefill":
        c = nbits(WL.prefill_u2((5120, 5120), M=2048))
        for _ in range(4):
            c()
    elif name in ("tc_prefill_gate_up", "tc_prefill_down"):
        c = nbits(WL.prefill_u2(name[len("tc_prefill_"):], M=2048))
        for _ in range(3):
            c()
    elif name in ("qmoe", "qmoe_dp4a"):
        d = WL.qmoe()
        h = lambda a: None if a is None else torch.from_numpy(a.view(np.int16)).cuda().view(torch.float16)
        y = torch.empty(d["hidden"], dtype=torch.float16, device="cuda")
        kw = dict(num_experts=d["num_experts"], fc1_w=torch.from_numpy(d["fc1_w"]).cuda(), fc1_scales=h(d["fc1_scales"]),
                  fc1_zp=None, fc1_bias=h(d["fc1_bias"]), fc2_w=torch.from_numpy(d["fc2_w"]).cuda(),
                  fc2_scales=h(d["fc2_scales"]), fc2_zp=None, fc2_bias=h(d["fc2_bias"]), bits=4, block_size=32, y=y)
        x, ids, w = h(d["x"]), torch.from_numpy(d["ids"]).cuda(), torch.from_numpy(d["weights"]).cuda()
        for _ in range(4):
            (qg.qmoe_decode_fused_dp4a if name == "qmoe_dp4a" else qg.qmoe_decode_fused)(x, ids, w, **kw)
    elif name == "tc_nf4_m64":
        d = WL.nf4("up", M=64, a_dtype=2)
        A = torch.from_numpy(d["A"].view(np.int16)).cuda().view(torch.bfloat16)
        W = torch.from_numpy(d["W"]).cuda()
        cb, am = torch.from_numpy(d["codebook"]).cuda(), torch.from_numpy(d["absmax"]).cuda()
        Y = torch.empty(64, d["N"], dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(max(16, qg.qgemm_workspace_bytes(2, 64, d["N"], d["K"], 4, 64)), dtype=torch.uint8,
                         device="cuda")
        for _ in range(4):
            qg.qgemm_codebook4(A, W, cb, am, Y, block_size=64, workspace=ws)
    elif name == "ragged":
        d = WL.ragged()
        X = torch.from_numpy(d["X"].view(np.int16)).cuda().view(torch.float16)
        W = torch.from_numpy(d["W"]).cuda()
        S = torch.from_numpy(d["scales"].view(np.int16)).cuda().view(torch.float16)
        Y = torch.empty(int(d["offsets"][-1]), d["N"], dtype=torch.float16, device="cuda")
        for _ in range(4):
            qg.qmoe_ragged_mm(X, d["offsets"], W, S, None, Y, bits=4, block_size=32)
    elif name == "gather":
        d = WL.embedding(1)
        W = torch.from_numpy(d["W"]).cuda()
        S = torch.from_numpy(d["scales"].view(np.int16)).cuda().view(torch.float16)
        Z = torch.from_numpy(d["zero_points"].view(np.int16)).cuda().view(torch.float16)
        idx = torch.from_numpy(d["indices"]).cuda()
        Y = torch.empty(d["n"], d["D"], dtype=torch.float16, device="cuda")
        for _ in range(4):
            qg.qg_gather_block_quantized(idx, W, S, Z, Y, w_format=1, block_size=d["block_size"])
    else:
        raise SystemExit("unknown probe %r" % name)
    torch.cuda.synchronize()
    print("probe %s done" % name)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration timings that follow the benchmark step")
    ap.add_argument("--oracle-timing", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--graph-steps", type=int, default=8,
                    help="steps per CUDA graph in the timed region (each step is 5 GEMV launches)")
    ap.add_argument("--clocks-log", default=None,
                    help="file for the raw nvidia-smi samples of the timed region (%%d: GPU index); default a temp file")
    ap.add_argument("--probe", choices=["gemv_k5120", "gemv_lm_head", "gemv_down", "tc_prefill", "tc_prefill_gate_up",
                                        "tc_prefill_down", "tc_nf4_m64", "qmoe",
                                        "qmoe_dp4a", "ragged", "gather"],
                    help="run a small fixed workload for a profiler capture instead of the benchmark")
    ap.add_argument("--suite", action="store_true",
                    help="time every configuration (one JSON line each) instead of the benchmark")
    ap.add_argument("--only", choices=["tiny_u4", "phi4_u2", "phi4_u8", "packed_zp", "nf4", "qmoe", "prefill",
                                       "f32_large_m", "ragged", "gather", "nsweep"],
                    help="with --suite: time one group of configurations only")
    args = ap.parse_args()
    if args.oracle_timing is not None:  # child of oracle_single_thread()
        cb, _ = cpu_baseline(budget_s=args.oracle_timing)
        print(json.dumps(cb), flush=True)
        return 0
    if args.probe:
        return run_probe(args.probe)
    if args.suite or args.only:
        run_suite(args.only)
        return 0
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
