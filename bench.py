#!/usr/bin/env python
"""Benchmark of the GB300 block-scaled MXFP4 GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--split-k S]
    python bench.py --impl reference ...     # the CPU oracle on a bounded sample
    python bench.py --profile-shape M,N,K [--calls C] [--format F]   # for profilers

One step is the whole hot path on one batch of resident inputs: one
mxfp4_gemm call, as a user makes it -- for compute-bound shapes the scale
relayout of A and B (one launch) and the GEMM on the relaid scales, launched
as its programmatic dependent; otherwise the GEMM alone, which builds the
tcgen05 scale layout itself and sums its split-K partials in-kernel.  Steps
rotate over copies of the inputs whose total exceeds three times the L2, so
no step finds its operands in L2, and K steps run back to back between one
pair of CUDA events on the launching stream (each launch waits in-kernel for
the one before it).  The roofline's kernel time is the GEMM alone on relaid
scales, timed the same way in a second loop that runs for at least a second
while nvidia-smi samples the clocks.  The default run (the large 8192^3
workload) also times the bandwidth-bound decode (1 x 8192 x 8192) and skinny
(64 x 7168 x 16384) workloads and reports them under "hbm_bound", each next
to a plain streaming read of its bytes timed the same way.  Rank 0 prints one
JSON line.  With N > 1 (torchrun) every rank runs an independent replica of
the workload (the GEMM needs no exchange), the barrier + max over ranks
times the job, and value counts all ranks' FLOPs.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 GEMM TFLOPS (device-timed, 1 GB300) and % of dense FP4 peak / HBM roofline"
UNIT = "TFLOP/s"
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense FP4 / dense bf16 tensor rate
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def max_over_ranks(values, dist, device):
    """Element-wise max of a list of floats over all ranks (the job's time is
    the slowest replica's); the values themselves without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def replica_throughput(world, flops_per_step, steps, total_ms):
    """Whole-job TFLOP/s: each of `world` replicas ran `steps` GEMMs of
    `flops_per_step`, and the job took the slowest rank's `total_ms`."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


# Device code and launchers of the GEMM kernels: a DRAM counter capture stays
# valid while these are unchanged and the plan launches the same configuration.
KERNEL_SOURCES = ("gemm_pair.cuh", "gemm_sm103.cu", "ptx.cuh", "internal.h")


def plan_key(plan):
    """The launch configuration a traffic capture was taken with."""
    return (f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k} stages {plan.stages} split "
            f"{plan.split_k} swap {plan.swap_ab} pair {plan.pair} "
            f"relayout {plan.relayout_pass} grid {plan.grid_x}x{plan.grid_y}x{plan.grid_z}")


def kernel_sources_sha1(names=KERNEL_SOURCES):
    """Hash of the kernels' sources (the GEMM's by default): DRAM counters
    taken for one version are only reported while the sources are unchanged."""
    import hashlib
    h = hashlib.sha1()
    for name in names:
        with open(os.path.join(ROOT, "block_scaled_mxfp4_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(workload, kernel, plan=None):
    """DRAM bytes (read + write) of one launch of `kernel` on `workload` from
    profiles/traffic.json (an ncu counter capture), or None if there is no
    capture for these sources and, when the record names one, this plan."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel") != kernel:
        return None
    if rec.get("sources_sha1") != kernel_sources_sha1(tuple(rec.get("sources", KERNEL_SOURCES))):
        return None
    if plan is not None and "plan" in rec and rec["plan"] != plan_key(plan):
        return None
    return rec["dram_bytes_read"] + rec["dram_bytes_write"]


def split_note(plan):
    if plan.split_k <= 1:
        return ""
    if plan.split_k <= 8:
        return (f" (K split {plan.split_k} ways; the splits of a tile form one cluster and sum "
                "their partials in split order over distributed shared memory)")
    return (f" (K split {plan.split_k} ways; the CTA that finishes a tile last sums its "
            "partials from the workspace in split order)")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large",
                    choices=["tiny", "decode", "mid", "large", "skinny", "quantize", "quantize8",
                             "quantize6",
                             "large8", "decode8", "mixed8", "large6", "mixed6", "large_nv",
                             "decode_nv", "skinny_nv"])
    ap.add_argument("--split-k", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prepacked", action="store_true",
                    help="step = scale relayout A + B kernels + GEMM on relaid scales")
    ap.add_argument("--hbm-steps", type=int, default=0,
                    help="calls per timed loop of the decode / skinny sub-benchmarks "
                         "(default: max(steps, 1000))")
    ap.add_argument("--no-hbm-bound", action="store_true",
                    help="skip the decode / skinny sub-benchmarks of the default run")
    ap.add_argument("--sustained-s", type=float, default=1.2,
                    help="seconds of the sustained GEMM-alone loop (0: skip it)")
    ap.add_argument("--profile-shape", default=None,
                    help="M,N,K: run a few GEMMs of a random shape for a profiler, no timing")
    ap.add_argument("--calls", type=int, default=3, help="--profile-shape: GEMM calls")
    ap.add_argument("--format", default="mxfp4",
                    choices=["mxfp4", "e4m3", "e5m2", "e2m3", "e3m2", "e2m1", "nvfp4"],
                    help="--profile-shape: element format")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def workload_geometry(p):
    flops = 2.0 * p.M * p.N * p.K
    algo_bytes = (p.M * p.K // 2 + p.N * p.K // 2 + p.M * p.K // 32 + p.N * p.K // 32
                  + 2 * p.M * p.N + (2 * p.M * p.N if p.beta != 0.0 else 0))
    return flops, algo_bytes


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx_ = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        # Samples "under load": SM clock within the upper part of its range.
        loaded = [s for s in sm if s >= 0.5 * (max(mx_) if mx_ else 1)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i - 5] for r in rows for i in range(5, 9)
                          if r[i].lower() in ("active", "1")})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx_) if mx_ else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "reasons": reasons}


def oracle_throughput(p, seconds, seed):
    """Time the CPU oracle (as it stands) on sampled outputs of the workload:
    returns (TFLOP/s, threads, sample description)."""
    import numpy as np

    import oracle
    from block_scaled_mxfp4_gb300 import inputs
    rng = np.random.default_rng(seed)

    def run(count):
        pairs = np.stack([rng.integers(0, p.M, count), rng.integers(0, p.N, count)], axis=1)
        t0 = time.perf_counter()
        if hasattr(p, "fmt_a"):          # MXFP8 problem
            fmt = inputs.BYTE_FORMATS
            oracle.gemm8_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K, fmt[p.fmt_a], fmt[p.fmt_b],
                                 pairs, alpha=p.alpha, beta=p.beta, C=p.C)
        elif p.SA.shape[1] == p.K // 16:  # NVFP4 problem (one scale per 16 K)
            oracle.gemm_nv_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K, pairs, alpha=p.alpha,
                                   beta=p.beta, C=p.C)
        else:
            oracle.gemm_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K, pairs, alpha=p.alpha,
                                beta=p.beta, C=p.C)
        return time.perf_counter() - t0

    cores = oracle.host_cores()
    count = max(cores * 4, 64)
    t = run(count)
    # A small probe is dominated by thread start-up, so scale up until the
    # timed sample itself lasts most of the requested time.
    for _ in range(4):
        if t >= 0.7 * seconds:
            break
        count = int(max(2 * count, count * seconds / max(t, 1e-6)))
        t = run(count)
    flops = 2.0 * p.K * count
    desc = (f"{count} random (m, n) outputs of the {p.M}x{p.N}x{p.K} workload, full K each "
            f"({flops / 2:.3g} MACs, {t:.1f} s)")
    return flops / t / 1e12, cores, desc, t


def run_reference(args, rank):
    """Reference arm: the CPU oracle, timed on the host cores, rank 0 only."""
    if rank != 0:
        return
    from block_scaled_mxfp4_gb300 import inputs
    if args.workload in ("quantize", "quantize8", "quantize6"):
        run_reference_quantize(args)
        return
    fp8 = args.workload in inputs.WORKLOADS8
    if args.workload in NV_WORKLOADS:
        p = nvfp4_problem(args.workload)
    else:
        p = inputs.workload8(args.workload) if fp8 else inputs.workload(args.workload)
    # About 100 s of oracle time in all (2.5 - 4 minutes with the per-step
    # overheads on 16 host cores), at most 4 s per step.
    per_step = min(4.0, 100.0 / max(1, args.steps))
    for i in range(args.warmup):
        oracle_throughput(p, min(per_step, 1.0), 1000 + i)
    vals, times, desc, cores = [], [], "", 0
    for i in range(args.steps):
        v, cores, desc, t = oracle_throughput(p, per_step, 2000 + i)
        vals.append(v)
        times.append(t)
    value = len(vals) / sum(1.0 / v for v in vals)        # total FLOPs / total time
    line = {
        "impl": "reference",
        "metric": ((METRIC6 if args.workload.endswith("6") else METRIC8) if fp8 else
                   METRIC_NV if args.workload in NV_WORKLOADS else METRIC),
        "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload} M={p.M} N={p.N} K={p.K}",
                   "M": p.M, "N": p.N, "K": p.K},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "per step: " + desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# --workload -> (format name, ABI code, oracle code, kernel) of mxfp8_quantize runs.
QUANT_BYTE = {"quantize8": ("mxfp8 e4m3", 0, 1, "quantize8_kernel<0>"),
              "quantize6": ("mxfp6 e2m3 (padded)", 3, 3, "quantize8_kernel<3>")}


def quant_metric(workload):
    if workload == "quantize8":
        return "MXFP8 quantiser bandwidth (bf16 -> E4M3 codes + E8M0 scales)"
    if workload == "quantize6":
        return "MXFP6 quantiser bandwidth (bf16 -> padded E2M3 codes + E8M0 scales)"
    return "MXFP4 quantiser bandwidth (bf16 -> E2M1 codes + E8M0 scales)"


METRIC8 = "MXFP8 GEMM TFLOPS (device-timed, 1 GB300) and % of dense FP8 peak / HBM roofline"
METRIC6 = "MXFP6 GEMM TFLOPS (device-timed, 1 GB300) and % of dense FP6 peak (the FP8 rate)"
FP8_PER_BF16 = 2.0                   # nominal dense FP8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


def run_mxfp8(args, world, rank, local_rank):
    """--workload large8 | decode8 | mixed8 | large6 | mixed6: one mxfp8_gemm
    call per step (FP6 operands in the padded 16-codes-per-16-bytes form)
    (scale relayout + one-tile tcgen05 GEMM, or the split-K GEMM), device
    timed with L2 flushed between steps; each rank of a multi-GPU launch runs
    the whole problem as a replica."""
    import numpy as np
    import torch

    import block_scaled_mxfp4_gb300 as mx
    from block_scaled_mxfp4_gb300 import build, inputs

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    build.build()
    dev = torch.device("cuda", local_rank)
    p = inputs.workload8(args.workload)
    M, N, K = p.M, p.N, p.K
    fmt = {"e4m3": mx.MXFP8_E4M3, "e5m2": mx.MXFP8_E5M2, "e2m3": mx.MXFP6_E2M3,
           "e3m2": mx.MXFP6_E3M2}
    fp6 = p.fmt_a in inputs.FP6_FORMATS or p.fmt_b in inputs.FP6_FORMATS
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    A, B, SA, SB = d(p.A), d(p.B), d(p.SA), d(p.SB)
    C = d(p.C.view(np.int16)).view(torch.bfloat16) if p.C is not None else None
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    split = args.split_k
    plan = mx.mxfp8_plan_gemm(M, N, K, split, 0)
    ws_bytes = mx.mxfp8_gemm_workspace_size(M, N, K, split)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    Cs = C if p.beta != 0.0 else None

    def step():
        mx.mxfp8_gemm(D, N, Cs, 0 if Cs is None else N, A, K, B, K, SA, K // 32, SB, K // 32,
                      fmt[p.fmt_a], fmt[p.fmt_b], p.alpha, p.beta, M, N, K, split,
                      ws if ws_bytes else None, ws_bytes, stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    tot_ms = max_over_ranks([sum(e[0].elapsed_time(e[1]) for e in ev)], dist, dev)[0]
    ms = tot_ms / args.steps
    flops = 2.0 * M * N * K
    nbytes = M * K + N * K + (M + N) * K // 32 + 2 * M * N + (2 * M * N if p.beta != 0.0 else 0)
    value = world * flops * args.steps / (tot_ms * 1e-3) / 1e12
    # end to end: host buffers through mxfp8_gemm_host (pinned host memory,
    # copies pipelined against the block GEMMs, all inside the timed region)
    pin = lambda t: t.cpu().pin_memory()
    hA, hB, hSA, hSB = pin(A), pin(B), pin(SA), pin(SB)
    hC = pin(C) if Cs is not None else None
    hD = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    arena_b = mx.mxfp8_gemm_host_arena_size(M, N, K, split, p.beta != 0.0)
    arena = torch.empty(arena_b, dtype=torch.uint8, device=dev)

    def e2e_step():
        mx.mxfp8_gemm_host(hD, hC, hA, hB, hSA, hSB, fmt[p.fmt_a], fmt[p.fmt_b], p.alpha, p.beta,
                           M, N, K, split, arena, arena_b, stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / args.e2e_steps], dist, dev)[0]
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    hbm_bound = M <= 64
    kernels = ("scale_relayout_kernel + " if plan.relayout_pass else "") + \
        f"gemm_mxf4_kernel<{plan.tile_n}, {plan.stages}, {'true' if plan.swap_ab else 'false'}, 1>"
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_source": f"{peak_src} HBM copy bandwidth"}
    else:
        peak = peaks["bf16_tflops"] * FP8_PER_BF16
        roof = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": peak,
                "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16 burst {peaks['bf16_tflops']:.1f} TFLOP/s x "
                               f"{FP8_PER_BF16:g} (nominal dense FP8/bf16 ratio"
                               + ("; FP6 runs at the FP8 rate in kind::mxf8f6f4)" if fp6 else ")")}
    traffic = recorded_traffic(args.workload, "gemm_mxf4_kernel", plan)
    roof.update({"frac": roof["achieved"] / roof["peak"], "traffic": traffic,
                 "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one GEMM "
                                    "launch (profiles/traffic.json)") if traffic else
                                   "no capture for these sources",
                 "kernel": kernels + " (one mxfp8_gemm call, timed together)", "kernel_ms": ms,
                 "algorithmic_bytes": nbytes, "flops": flops})
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_throughput(p, 10.0, 77)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    h2d = sum(t.numel() * t.element_size() for t in (hA, hB, hSA, hSB) + ((hC,) if hC is not None else ()))
    line = {
        "metric": METRIC6 if fp6 else METRIC8, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": f"{'mxfp6' if fp6 else 'mxfp8'} ({p.fmt_a} x {p.fmt_b})", "data": "synthetic",
        "config": {"workload": f"{args.workload} M={M} N={N} K={K}", "M": M, "N": N, "K": K,
                   "fmt_a": p.fmt_a, "fmt_b": p.fmt_b, "alpha": p.alpha, "beta": p.beta,
                   "seed": p.seed, "split_k": plan.split_k, "swap_ab": plan.swap_ab,
                   "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}", "stages": plan.stages,
                   "grid": [plan.grid_x, plan.grid_y, plan.grid_z],
                   "l2": "flushed between timed steps (512 MiB write outside the events)",
                   "step": "one mxfp8_gemm call" + split_note(plan),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": M * N * 2, "ms_per_step": e2e_ms,
                "api": "mxfp8_gemm_host (pinned host buffers)"},
        "gpu_launches": args.steps * (1 + plan.relayout_pass),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


METRIC_NV = "NVFP4 GEMM TFLOPS (device-timed, 1 GB300) and % of dense FP4 peak / HBM roofline"

# NVFP4 workloads: the MXFP4 large, decode and skinny shapes (alpha, beta and
# C as there) with E2M1 codes uniform over all 16 and UE4M3 scales uniform
# over 0x28..0x48 (0.25 .. 4).
NV_WORKLOADS = {
    "large_nv": (8192, 8192, 8192, 13, 1.0, 0.0, None),
    "decode_nv": (1, 8192, 8192, 14, 1.0, 0.0, None),
    "skinny_nv": (64, 7168, 16384, 15, 1.0, 1.0, 0.1),
}


def nvfp4_problem(name="large_nv"):
    from block_scaled_mxfp4_gb300 import inputs
    M, N, K, seed, alpha, beta, c_sigma = NV_WORKLOADS[name]
    return inputs.make_problem_nv(name, M, N, K, seed=seed, alpha=alpha, beta=beta,
                                  c_sigma=c_sigma)


def run_nvfp4(args, world, rank, local_rank):
    """--workload large_nv | decode_nv | skinny_nv: one nvfp4_gemm call per
    step (large: the NVFP4 scale relayout + the CTA-pair kernel launched as
    its dependent; decode / skinny: the one-tile kernel with split-K in the
    launch), steps back to back over rotating input copies, as the MXFP4
    headline is timed; each rank of a multi-GPU launch runs a replica."""
    import torch

    import block_scaled_mxfp4_gb300 as mx
    from block_scaled_mxfp4_gb300 import build

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    build.build()
    dev = torch.device("cuda", local_rank)
    p = nvfp4_problem(args.workload)
    M, N, K = p.M, p.N, p.K
    in_bytes = M * K // 2 + N * K // 2 + (M + N) * K // 16 + (2 * M * N if p.beta != 0.0 else 0)
    copies = rotation_copies(in_bytes)
    ops = Operands(p, copies, dev)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    wsb = mx.nvfp4_gemm_workspace_size(M, N, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def launch(i):
        c = i % copies
        C = ops.C[c] if p.beta != 0.0 else None
        mx.nvfp4_gemm(D, N, C, N if C is not None else 0, ops.A[c], K, ops.B[c], K, ops.SA[c],
                      K // 16, ops.SB[c], K // 16, p.alpha, p.beta, M, N, K, ws, wsb, stream)

    for i in range(max(3, args.warmup)):
        launch(i)
    sampler = ClockSampler(local_rank)
    sampler.start()
    tot_ms = max_over_ranks([timed_back_to_back(stream, args.steps, launch, dist, dev)], dist,
                            dev)[0]
    clocks = sampler.stop()
    ms = tot_ms / args.steps
    flops = 2.0 * M * N * K
    nbytes = in_bytes + 2 * M * N
    value = world * flops * args.steps / (tot_ms * 1e-3) / 1e12
    # End to end through the same entry point from pinned host buffers: the
    # inputs' copies in, the call, D's copy out, all inside the timed region.
    pin = lambda t: t.cpu().pin_memory()
    hA, hB, hSA, hSB = pin(ops.A[0]), pin(ops.B[0]), pin(ops.SA[0]), pin(ops.SB[0])
    copies_in = [(hA, ops.A[0]), (hB, ops.B[0]), (hSA, ops.SA[0]), (hSB, ops.SB[0])]
    if p.beta != 0.0:
        copies_in.append((pin(ops.C[0]), ops.C[0]))
    hD = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        for h, d in copies_in:
            d.copy_(h, non_blocking=True)
        launch(0)
        hD.copy_(D, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / args.e2e_steps], dist, dev)[0]
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    skinny = M <= 64
    if skinny:
        achieved = nbytes / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{peak_src} HBM copy bandwidth",
                "kernel": "gemm_mxf4_kernel<64, 4, true, 2, 2> (one nvfp4_gemm call)"}
    else:
        achieved = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"] * FP4_OVER_BF16, "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16 burst {peaks['bf16_tflops']:.1f} TFLOP/s x "
                               f"{FP4_OVER_BF16:g} (nominal dense FP4/bf16 ratio; NVFP4 runs at "
                               "the FP4 rate)",
                "kernel": "scale_relayout_kernel + gemm_mxf4_pair<5, true> (one nvfp4_gemm "
                          "call, timed together)"}
    traffic = recorded_traffic(args.workload, "gemm_mxf4_kernel" if skinny else "gemm_mxf4_pair")
    roof.update({"frac": achieved / roof["peak"], "traffic": traffic,
                 "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one GEMM "
                                   "launch (profiles/traffic.json); null when the sources changed "
                                   "since",
                 "kernel_ms": ms, "algorithmic_bytes": nbytes, "flops": flops})
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_throughput(p, 10.0, 78)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    h2d = sum(h.numel() * h.element_size() for h, _ in copies_in)
    line = {
        "metric": METRIC_NV, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1, ue4m3 per 16)", "data": "synthetic",
        "config": {"workload": f"{args.workload} M={M} N={N} K={K}", "M": M, "N": N, "K": K,
                   "alpha": p.alpha, "beta": p.beta, "seed": p.seed,
                   "tile": "128x64x256 (swap-AB)" if skinny else "256x256x256",
                   "stages": 4 if skinny else 5,
                   "l2": f"inputs larger than L2: steps rotate over {copies} copies of the "
                         "inputs, back to back between one pair of events",
                   "step": ("one nvfp4_gemm call: the one-tile GEMM, K split across a cluster "
                            "summed in the launch") if skinny else
                           ("one nvfp4_gemm call: NVFP4 scale relayout of A and B (one launch) + "
                            "CTA-pair GEMM launched as its dependent"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": M * N * 2, "ms_per_step": e2e_ms,
                "api": "nvfp4_gemm with its inputs copied in and D copied out (pinned host "
                       "memory) on the same stream"},
        "gpu_launches": (1 if skinny else 2) * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


QUANT_ROWS, QUANT_K = 8192, 8192     # the large GEMM's activations, bf16


def run_reference_quantize(args):
    """Reference arm of --workload quantize: the oracle quantiser on one host
    thread, each step a bounded sample of rows of the same input."""
    import numpy as np

    import oracle
    from block_scaled_mxfp4_gb300 import inputs
    rows, K = QUANT_ROWS, QUANT_K
    xbits = inputs.f32_to_bf16_bits(
        np.random.default_rng(5).standard_normal((rows, K), dtype=np.float32))
    nrows = 64
    fp8 = args.workload in QUANT_BYTE
    name, _, ofmt, _ = QUANT_BYTE.get(args.workload, (None, None, None, None))
    per_elem = 2 + (1 if fp8 else 0.5) + 1 / 32

    def one(i):
        chunk = xbits[(i * nrows) % rows:][:nrows]
        if fp8:
            oracle.quantize8(chunk, nrows, K, ofmt)
        else:
            oracle.quantize(chunk, nrows, K)

    for i in range(args.warmup):
        one(i)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        one(i)
        times.append(time.perf_counter() - t0)
    value = args.steps * nrows * K * per_elem / sum(times) / 1e9
    line = {
        "impl": "reference",
        "metric": quant_metric(args.workload),
        "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.workload} rows={rows} K={K}", "rows": rows,
                                        "K": K},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step: {nrows} rows of the {rows}x{K} input"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_quantize(args, world, rank, local_rank):
    """--workload quantize: mxfp4_quantize of bf16 [8192, 8192] N(0,1)
    activations into the GEMM's operand format; bandwidth-bound, reported in
    GB/s of algorithmic bytes (2 in, 17/32 out per element) against the HBM
    copy peak, with the CPU oracle on a bounded sample beside it."""
    import numpy as np
    import torch

    import block_scaled_mxfp4_gb300 as mx
    from block_scaled_mxfp4_gb300 import build, inputs

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    build.build()
    dev = torch.device("cuda", local_rank)
    rows, K = QUANT_ROWS, QUANT_K
    rng = np.random.default_rng(5)
    xbits = inputs.f32_to_bf16_bits(rng.standard_normal((rows, K), dtype=np.float32))
    X = torch.from_numpy(xbits.view(np.int16)).to(dev)
    fp8 = args.workload in QUANT_BYTE           # one byte per element (8-bit or padded 6-bit)
    name, afmt, ofmt, kname = QUANT_BYTE.get(args.workload, (None, None, None, "quantize_kernel"))
    qcols = K if fp8 else K // 2
    Q = torch.empty((rows, qcols), dtype=torch.uint8, device=dev)
    S = torch.empty((rows, K // 32), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    nbytes = rows * K * 2 + rows * qcols + rows * K // 32

    def step():
        if fp8:
            mx.mxfp8_quantize(Q, K, S, K // 32, X, K, rows, K, afmt, stream)
        else:
            mx.mxfp4_quantize(Q, K, S, K // 32, X, K, rows, K, stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    tot_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    tot_ms = max_over_ranks([tot_ms], dist, dev)[0]
    ms = tot_ms / args.steps
    value = world * nbytes * args.steps / (tot_ms * 1e-3) / 1e9
    # end to end: host bf16 in, host codes and scales out, copies timed
    hX = torch.from_numpy(xbits.view(np.int16)).pin_memory()
    hQ = torch.empty((rows, qcols), dtype=torch.uint8).pin_memory()
    hS = torch.empty((rows, K // 32), dtype=torch.uint8).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        X.copy_(hX, non_blocking=True)
        step()
        hQ.copy_(Q, non_blocking=True)
        hS.copy_(S, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / args.e2e_steps], dist, dev)[0]
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        nrows = 256
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 10.0:
            if fp8:
                oracle.quantize8(xbits[reps * nrows % rows:][:nrows], nrows, K, ofmt)
            else:
                oracle.quantize(xbits[reps * nrows % rows:][:nrows], nrows, K)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": reps * nbytes / rows * nrows / dt / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"{reps} x {nrows} rows of the {rows}x{K} input "
                                           f"({dt:.1f} s, one thread)"}
    line = {
        "metric": quant_metric(args.workload),
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": f"bf16->{name}" if fp8 else "bf16->mxfp4",
        "data": "synthetic",
        "config": {"workload": f"{args.workload} rows={rows} K={K}", "rows": rows, "K": K,
                   "l2": "flushed between timed steps (512 MiB write outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": recorded_traffic(args.workload, "quantize8_kernel" if fp8
                                                 else "quantize_kernel"),
                     "kernel": kname, "kernel_ms": ms,
                     "algorithmic_bytes": nbytes, "peak_source": f"{peak_src} HBM copy bandwidth"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": rows * K * 2, "d2h_bytes_per_step": rows * qcols + rows * K // 32,
                "ms_per_step": e2e_ms,
                "api": f"{'mxfp8' if fp8 else 'mxfp4'}_quantize (pinned host copies around it)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


L2_BYTES = 129 * 1024 * 1024          # GB300 L2; rotation keeps > 3x this in flight


def rotation_copies(nbytes):
    """Input copies a rotation needs so that their total exceeds 3 x L2."""
    return max(2, -(-3 * L2_BYTES // max(1, nbytes)) + 1)


class Operands:
    """`copies` device copies of a problem's inputs (each its own allocation,
    so every step of a rotation reads bytes that no recent step touched)."""

    def __init__(self, p, copies, dev):
        import numpy as np
        import torch
        to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.A = [to_dev(p.A) for _ in range(copies)]
        self.B = [to_dev(p.B) for _ in range(copies)]
        self.SA = [to_dev(p.SA) for _ in range(copies)]
        self.SB = [to_dev(p.SB) for _ in range(copies)]
        self.C = None if p.C is None else \
            [to_dev(p.C.view(np.int16)).view(torch.bfloat16) for _ in range(copies)]
        self.copies = copies


def timed_back_to_back(stream, n, launch, dist=None, device=None):
    """Total ms of n launches (launch(i)) enqueued back to back between one
    pair of CUDA events on `stream`, bracketed by a barrier + synchronize."""
    import torch
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        launch(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return e0.elapsed_time(e1)


def probe_lib():
    """The benchmark's streaming-read helper (not part of the library)."""
    import ctypes
    from block_scaled_mxfp4_gb300 import build
    L = ctypes.CDLL(build.build_probe())
    L.mxfp4_probe_stream_read.restype = ctypes.c_int
    L.mxfp4_probe_stream_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                          ctypes.c_int, ctypes.c_void_p]
    return L


def stream_floor(nbytes, steps, stream, dev):
    """A plain streaming read of nbytes, over a rotation of buffers like the
    GEMM's, launched back to back (mode 1: each read waits for the one before
    it, as mxfp4_gemm does; mode 2: reads overlap, as with MXFP4_FLAG_B_STATIC)."""
    import torch
    L = probe_lib()
    per = -(-nbytes // 4096) * 4096
    copies = rotation_copies(per)
    pool = torch.empty(per * copies, dtype=torch.uint8, device=dev)
    pool.fill_(1)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {"what": "one streaming read of the algorithmic bytes (16-byte loads, every SM), "
                   f"rotating over {copies} buffers, back to back between one event pair"}
    for mode, key in ((1, "ordered"), (2, "overlapped")):
        def launch(i):
            rc = L.mxfp4_probe_stream_read(pool.data_ptr() + (i % copies) * per, nbytes,
                                           sink.data_ptr(), mode, stream.cuda_stream)
            assert rc == 0, rc
        for i in range(20):
            launch(i)
        ms = timed_back_to_back(stream, steps, launch) / steps
        out[key] = {"us": ms * 1e3, "GB/s": nbytes / (ms * 1e-3) / 1e9}
    del pool
    return out


def hbm_bound_run(name, steps, dev, stream, peaks, peak_src, dist=None):
    """Decode / skinny sub-benchmark of the default run: K back-to-back
    mxfp4_gemm calls over rotating input copies, plain and with
    MXFP4_FLAG_B_STATIC, against the HBM copy peak and a streaming read of
    the same bytes timed the same way; plus one cold call after a flush."""
    import torch

    import block_scaled_mxfp4_gb300 as mx
    from block_scaled_mxfp4_gb300 import inputs
    p = inputs.workload(name)
    flops, algo_bytes = workload_geometry(p)
    M, N, K = p.M, p.N, p.K
    copies = rotation_copies(algo_bytes)
    ops = Operands(p, copies, dev)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    plan = mx.mxfp4_plan_gemm(M, N, K, 0, 0)
    wsb = mx.mxfp4_gemm_workspace_size(M, N, K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)

    def launch(i, flags):
        c = i % copies
        C = ops.C[c] if p.beta != 0.0 else None
        mx.mxfp4_gemm_ex(D, N, C, N, ops.A[c], K, ops.B[c], K, ops.SA[c], K // 32, ops.SB[c],
                         K // 32, p.alpha, p.beta, M, N, K, 0, flags, ws, wsb, stream)

    res = {"workload": f"{name} M={M} N={N} K={K}", "split_k": plan.split_k,
           "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}", "swap_ab": plan.swap_ab,
           "grid": [plan.grid_x, plan.grid_y, plan.grid_z], "rotation_copies": copies,
           "algorithmic_bytes": algo_bytes, "steps": steps}
    for flags, key in ((0, "default"), (mx.MXFP4_FLAG_B_STATIC, "b_static")):
        for i in range(max(20, steps // 10)):
            launch(i, flags)
        ms = max_over_ranks([timed_back_to_back(stream, steps, lambda i: launch(i, flags), dist,
                                                dev) / steps], dist, dev)[0]
        gbs = algo_bytes / (ms * 1e-3) / 1e9
        res[key] = {"us_per_gemm": ms * 1e3, "TFLOP/s": flops / (ms * 1e-3) / 1e12,
                    "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                                 "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                                 "peak_source": f"{peak_src} HBM copy bandwidth",
                                 "traffic": recorded_traffic(name, "gemm_mxf4_kernel", plan)}}
    res["b_static"]["api"] = ("mxfp4_gemm_ex(..., MXFP4_FLAG_B_STATIC): B and its scales are "
                              "loaded without the in-kernel wait on the previous call")
    res["default"]["api"] = "mxfp4_gemm"
    floor = stream_floor(algo_bytes, steps, stream, dev)
    floor["default_over_ordered"] = res["default"]["us_per_gemm"] / floor["ordered"]["us"]
    floor["b_static_over_overlapped"] = res["b_static"]["us_per_gemm"] / floor["overlapped"]["us"]
    res["stream_floor"] = floor
    # One call alone after a 512 MiB flush (launch latency included).
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    cold = []
    for i in range(13):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch(i, 0)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            cold.append(e0.elapsed_time(e1))
    res["cold_single_call_us"] = statistics.median(cold) * 1e3
    del flush, ops
    return res


def profile_shape(args):
    """Run a few GEMMs of a seeded random shape for a profiler (no timing,
    nothing checked): mxfp4 = random fp4x2 codes and E8M0 scales in
    [120, 127], then --calls mxfp4_gemm calls (--prepacked: scales relaid
    once, then mxfp4_gemm_prepacked calls) with the heuristic's plan; the
    byte formats = random codes (the 8-bit formats' NaN codes avoided; every
    byte is a valid padded 6- or 4-bit group), then --calls mxfp8_gemm calls;
    nvfp4 = random fp4x2 codes and UE4M3 scales in [0x30, 0x40], then --calls
    nvfp4_gemm calls."""
    import torch

    import block_scaled_mxfp4_gb300 as mx
    from block_scaled_mxfp4_gb300 import build
    build.build()
    M, N, K = (int(x) for x in args.profile_shape.split(","))
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(0)
    SA = torch.randint(120, 128, (M, K // 32), dtype=torch.uint8, device=dev, generator=g)
    SB = torch.randint(120, 128, (N, K // 32), dtype=torch.uint8, device=dev, generator=g)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if args.format == "nvfp4":
        A = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev, generator=g)
        B = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=g)
        SA = torch.randint(0x30, 0x41, (M, K // 16), dtype=torch.uint8, device=dev, generator=g)
        SB = torch.randint(0x30, 0x41, (N, K // 16), dtype=torch.uint8, device=dev, generator=g)
        wsb = mx.nvfp4_gemm_workspace_size(M, N, K)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        for _ in range(args.calls):
            mx.nvfp4_gemm(D, N, None, 0, A, K, B, K, SA, K // 16, SB, K // 16, 1.0, 0.0, M, N, K,
                          ws, wsb)
        torch.cuda.synchronize()
        print(f"{M}x{N}x{K} nvfp4: {args.calls} calls")
        return
    if args.format != "mxfp4":
        fmt = {"e4m3": mx.MXFP8_E4M3, "e5m2": mx.MXFP8_E5M2, "e2m3": mx.MXFP6_E2M3,
               "e3m2": mx.MXFP6_E3M2, "e2m1": mx.MXFP4_E2M1_PADDED}[args.format]
        top = 0x70 if args.format in ("e4m3", "e5m2") else 256
        A = torch.randint(0, top, (M, K), dtype=torch.uint8, device=dev, generator=g)
        B = torch.randint(0, top, (N, K), dtype=torch.uint8, device=dev, generator=g)
        wsb = mx.mxfp8_gemm_workspace_size(M, N, K, 0)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        for _ in range(args.calls):
            mx.mxfp8_gemm(D, N, None, N, A, K, B, K, SA, K // 32, SB, K // 32, fmt, fmt, 1.0, 0.0,
                          M, N, K, 0, ws if wsb else None, wsb)
        plan = mx.mxfp8_plan_gemm(M, N, K, 0, 0)
    else:
        A = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev, generator=g)
        B = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=g)
        if args.prepacked:
            sfa = torch.empty(mx.mxfp4_scale_relayout_size(M, K), dtype=torch.uint8, device=dev)
            sfb = torch.empty(mx.mxfp4_scale_relayout_size(N, K), dtype=torch.uint8, device=dev)
            mx.mxfp4_scale_relayout(sfa, SA, M, K, K // 32)
            mx.mxfp4_scale_relayout(sfb, SB, N, K, K // 32)
            wsb = mx.mxfp4_gemm_prepacked_workspace_size(M, N, K, 0)
            ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
            for _ in range(args.calls):
                mx.mxfp4_gemm_prepacked(D, N, None, N, A, K, B, K, sfa, sfb, 1.0, 0.0, M, N, K,
                                        0, ws if wsb else None, wsb)
        else:
            wsb = mx.mxfp4_gemm_workspace_size(M, N, K, 0)
            ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
            for _ in range(args.calls):
                mx.mxfp4_gemm(D, N, None, N, A, K, B, K, SA, K // 32, SB, K // 32, 1.0, 0.0,
                              M, N, K, 0, ws if wsb else None, wsb)
        plan = mx.mxfp4_plan_gemm(M, N, K, 0, 0)
    torch.cuda.synchronize()
    print(f"{M}x{N}x{K} {args.format}: {args.calls} calls, plan {plan.as_dict()}")


def run_mxfp4(args, world, rank, local_rank):
    import numpy as np
    import torch

    import block_scaled_mxfp4_gb300 as mx
    from block_scaled_mxfp4_gb300 import build, inputs

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    build.build()
    mx.lib()

    p = inputs.workload(args.workload)
    flops, algo_bytes = workload_geometry(p)
    dev = torch.device("cuda", local_rank)
    M, N, K = p.M, p.N, p.K
    in_bytes = M * K // 2 + N * K // 2 + (M + N) * K // 32 + (2 * M * N if p.C is not None else 0)
    copies = rotation_copies(in_bytes)
    ops = Operands(p, copies, dev)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    plan = mx.mxfp4_plan_gemm(M, N, K, args.split_k, 0)
    wsb = mx.mxfp4_gemm_workspace_size(M, N, K, args.split_k)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    wpb = mx.mxfp4_gemm_prepacked_workspace_size(M, N, K, args.split_k)
    wp = torch.empty(max(wpb, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Relaid scales of every copy, for the GEMM-alone loop (and --prepacked).
    sfa = [torch.empty(mx.mxfp4_scale_relayout_size(M, K), dtype=torch.uint8, device=dev)
           for _ in range(copies)]
    sfb = [torch.empty(mx.mxfp4_scale_relayout_size(N, K), dtype=torch.uint8, device=dev)
           for _ in range(copies)]
    for c in range(copies):
        mx.mxfp4_scale_relayout2(sfa[c], ops.SA[c], M, K // 32, sfb[c], ops.SB[c], N, K // 32, K,
                                 stream)
    Cs = lambda c: ops.C[c] if p.beta != 0.0 else None
    gemm_alone = args.prepacked or plan.relayout_pass

    def step(i):
        c = i % copies
        if args.prepacked:
            mx.mxfp4_scale_relayout2(sfa[c], ops.SA[c], M, K // 32, sfb[c], ops.SB[c], N,
                                     K // 32, K, stream)
            mx.mxfp4_gemm_prepacked(D, N, Cs(c), N, ops.A[c], K, ops.B[c], K, sfa[c], sfb[c],
                                    p.alpha, p.beta, M, N, K, args.split_k, wp, wpb, stream)
        else:
            mx.mxfp4_gemm(D, N, Cs(c), N, ops.A[c], K, ops.B[c], K, ops.SA[c], K // 32, ops.SB[c],
                          K // 32, p.alpha, p.beta, M, N, K, args.split_k, ws, wsb, stream)

    def gemm_kernel(i):
        c = i % copies
        mx.mxfp4_gemm_prepacked(D, N, Cs(c), N, ops.A[c], K, ops.B[c], K, sfa[c], sfb[c], p.alpha,
                                p.beta, M, N, K, args.split_k, wp, wpb, stream)

    for i in range(max(3, args.warmup)):
        step(i)
        if gemm_alone:
            gemm_kernel(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    t_wall = time.perf_counter()
    tot_ms = timed_back_to_back(stream, args.steps, step, dist, dev)
    t_wall = time.perf_counter() - t_wall
    # The GEMM kernel alone (relaid scales) for the roofline, timed the same
    # way: a burst as long as the timed steps (against the burst peak), then
    # a loop of at least a second (against the sustained peak) so that the
    # clock sampler sees the GPU under sustained load.
    per = tot_ms / args.steps
    n_sus = max(1, int(args.sustained_s * 1e3 / max(per, 1e-3))) if args.sustained_s > 0 else 0
    if gemm_alone:
        n_alone = args.steps
        gemm_avg = timed_back_to_back(stream, n_alone, gemm_kernel, dist, dev) / n_alone
        sus_tot = timed_back_to_back(stream, n_sus, gemm_kernel, dist, dev) if n_sus else 0.0
    else:
        n_alone = 0
        gemm_avg = tot_ms / args.steps
        sus_tot = timed_back_to_back(stream, n_sus, step, dist, dev) if n_sus else 0.0
    sus_avg = sus_tot / n_sus if n_sus else gemm_avg
    gemm_tot = sus_tot
    clocks = sampler.stop()
    tot_ms, gemm_avg, sus_avg = max_over_ranks([tot_ms, gemm_avg, sus_avg], dist, dev)
    ms_per_step = tot_ms / args.steps
    value = replica_throughput(world, flops, args.steps, tot_ms)
    launches_per_step = 2 if plan.relayout_pass or args.prepacked else 1

    # ---- end to end: host buffers through the C ABI, copies in the timed region
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hA, hB, hSA, hSB = pin(p.A), pin(p.B), pin(p.SA), pin(p.SB)
    hC = pin(p.C.view(np.int16)) if p.C is not None else None
    hD = torch.empty((M, N), dtype=torch.int16).pin_memory()
    arena_b = mx.mxfp4_gemm_host_arena_size(M, N, K, args.split_k, p.beta != 0.0)
    arena = torch.empty(arena_b, dtype=torch.uint8, device=dev)

    def e2e_step(i):
        mx.mxfp4_gemm_host(hD, hC, hA, hB, hSA, hSB, p.alpha, p.beta, M, N, K, args.split_k,
                           arena, arena_b, stream)

    for i in range(3):
        e2e_step(i)
    e2e_ms = timed_back_to_back(stream, args.e2e_steps, e2e_step, dist, dev) / args.e2e_steps
    e2e_ms = max_over_ranks([e2e_ms], dist, dev)[0]
    h2d = hA.numel() + hB.numel() + hSA.numel() + hSB.numel() + (hC.numel() * 2 if hC is not None else 0)
    d2h = hD.numel() * 2
    del arena

    peaks, peak_src = load_peaks()
    # The bandwidth-bound workloads of the target, in the same process.
    hbm = None
    if args.workload == "large" and not args.no_hbm_bound and not args.prepacked:
        del ops, sfa, sfb
        torch.cuda.empty_cache()
        hbm_steps = args.hbm_steps if args.hbm_steps > 0 else max(args.steps, 1000)
        hbm = {w: hbm_bound_run(w, hbm_steps, dev, stream, peaks, peak_src, dist)
               for w in ("decode", "skinny")}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    if args.workload in ("large", "mid", "tiny"):
        peak = peaks["bf16_tflops"] * FP4_OVER_BF16
        roof = {"bound": "tensor", "achieved": flops / (gemm_avg * 1e-3) / 1e12, "peak": peak,
                "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16 burst {peaks['bf16_tflops']:.1f} TFLOP/s x "
                               f"{FP4_OVER_BF16:g} (nominal dense FP4/bf16 ratio)"}
    else:
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": algo_bytes / (gemm_avg * 1e-3) / 1e9, "peak": peak,
                "unit": "GB/s", "peak_source": f"{peak_src} HBM copy bandwidth"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor" and n_sus:
        sus_peak = peaks["bf16_tflops_sustained"] * FP4_OVER_BF16
        sus_ach = flops / (sus_avg * 1e-3) / 1e12
        roof["sustained"] = {
            "achieved": sus_ach, "peak": sus_peak, "frac": sus_ach / sus_peak, "unit": "TFLOP/s",
            "kernel_ms": sus_avg, "launches": n_sus,
            "peak_source": f"{peak_src} bf16 sustained {peaks['bf16_tflops_sustained']:.1f} "
                           f"TFLOP/s x {FP4_OVER_BF16:g}",
            "what": "the same kernel back to back for over a second (power-capped clocks)"}
    kname = "gemm_mxf4_pair" if plan.pair else "gemm_mxf4_kernel"
    roof["traffic"] = recorded_traffic(args.workload, kname, plan)
    roof["traffic_source"] = ("profiles/traffic.json (ncu dram__bytes_read.sum + "
                              "dram__bytes_write.sum of one launch, same kernel sources "
                              "and launch configuration)"
                              if roof["traffic"] is not None else None)
    roof["kernel"] = kname + (f" (GEMM alone on relaid scales: {n_alone} launches back to back)"
                              if gemm_alone else " (scale layout built in-kernel)")
    roof["kernel_ms"] = gemm_avg
    roof["algorithmic_bytes"] = algo_bytes
    roof["flops"] = flops

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_throughput(p, 12.0, 7)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4", "data": "synthetic",
        "config": {"workload": f"{args.workload} M={M} N={N} K={K}", "M": M, "N": N, "K": K,
                   "alpha": p.alpha, "beta": p.beta, "seed": p.seed,
                   "split_k": plan.split_k, "swap_ab": plan.swap_ab,
                   "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}", "stages": plan.stages,
                   "grid": [plan.grid_x, plan.grid_y, plan.grid_z],
                   "l2": f"inputs larger than L2: steps rotate over {copies} copies of the "
                         f"inputs ({copies * in_bytes / 2**20:.0f} MiB > 3 x L2), back to back "
                         "between one pair of events",
                   "step": ("mxfp4_scale_relayout2 + mxfp4_gemm_prepacked"
                            if args.prepacked else
                            "one mxfp4_gemm call: scale relayout of A and B (one launch) + GEMM "
                            "on relaid scales (launched as its dependent)"
                            if plan.relayout_pass else
                            "one mxfp4_gemm call: GEMM with in-kernel scale layout")
                           + split_note(plan),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": replica_throughput(world, flops, 1, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "api": "mxfp4_gemm_host (pinned host buffers)"},
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_note": ("our kernels in the timed step loop; the roofline's GEMM-alone "
                              f"loops ({n_alone} + {n_sus} launches) run after it" if gemm_alone else
                              f"our kernels in the timed step loop; a sustained loop of {n_sus} "
                              "steps runs after it"),
        "clocks": clocks,
        "clocks_window": ("nvidia-smi every 50 ms over the timed steps and the GEMM-alone "
                          f"loops ({(t_wall * 1e3 + gemm_tot) / 1e3:.2f} s of GPU work)"),
        "wall_s_timed_loop": t_wall,
    }
    if hbm is not None:
        line["hbm_bound"] = hbm
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.profile_shape:
        profile_shape(args)
        return
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.workload in ("quantize", "quantize8", "quantize6"):
        run_quantize(args, world, rank, local_rank)
        return
    if args.workload in ("large8", "decode8", "mixed8", "large6", "mixed6"):
        run_mxfp8(args, world, rank, local_rank)
        return
    if args.workload in NV_WORKLOADS:
        run_nvfp4(args, world, rank, local_rank)
        return
    run_mxfp4(args, world, rank, local_rank)


if __name__ == "__main__":
    main()
