#!/usr/bin/env python3
"""Benchmark of the tcgen05 GEMM on synthetic, seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Prints ONE JSON line (rank 0). A step is one GEMM D = alpha*A*B + beta*C of
the workload, inputs resident in HBM; `value` is whole-job TFLOP/s
(2*M*N*K per step, summed over ranks, over the slowest rank's time). The
default workload is the 8192^3 bf16 GEMM (A K-major, B MN-major, fp32 out,
beta = 1 over a seeded C, CTA pairs, persistent scheduler); its operands
(768 MB) are larger than L2, so no flush is needed between steps.

`--impl reference` times the fp64 CPU oracle on a bounded row sample of the
same workload instead (the only other place this script runs the oracle is
the `cpu_baseline` leg of the default run).

Multi-GPU: the GEMM does not shard here; N ranks run N independent replicas
(one process per GPU, NCCL only for the barrier and the max-over-ranks time).
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

# name -> (M, N, K, in, a_major, b_major, out, alpha, beta, dist, scale, options, description)
WORKLOADS = {
    "square8192_pair_f32_beta1": dict(
        M=8192, N=8192, K=8192, a_major="K", b_major="MN", out="f32", alpha=1.0, beta=1.0, dist="uniform",
        scale=1.0, seed=20, options=dict(cta_group=2, tile_n=256),
        desc="8192^3 bf16, A K-major, B MN-major, U[-1,1], fp32 out, beta=1 over seeded C, "
             "cta_group::2 CTA pairs, persistent tile scheduler"),
    "square4096_bf16": dict(
        M=4096, N=4096, K=4096, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="normal",
        scale=0.1, seed=10, options=dict(cta_group=1, tile_n=256),
        desc="4096^3 bf16, A and B K-major, N(0,1)*0.1, bf16 out, SW128, cta_group::1"),
    "skinny_m16384_n128_k8192": dict(
        M=16384, N=128, K=8192, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="normal",
        scale=1.0, seed=30, options=None, desc="M=16384 N=128 K=8192 bf16, N(0,1), bf16 out"),
    "skinny_m128_n16384_k4096": dict(
        M=128, N=16384, K=4096, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="normal",
        scale=1.0, seed=31, options=None, desc="M=128 N=16384 K=4096 bf16, N(0,1), bf16 out"),
    "single_tile_128x128x32_f16": dict(
        M=128, N=128, K=32, a_major="K", b_major="MN", out="f32", alpha=1.0, beta=0.0, dist="uniform",
        scale=1.0, seed=0, options=None, in_fmt="f16",
        desc="D[128x128] fp32 = A[128x32] fp16 K-major x B[32x128] fp16 MN-major, two m128n128k16 MMAs"),
}
DEFAULT_WORKLOAD = "square8192_pair_f32_beta1"
GROUPED = "grouped64_n4096_k2048"


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


KERNEL_SOURCES = ("gemm_kernel.cuh", "ptx.cuh", "descriptors.cuh")


def _source_hash():
    """Hash of the device-code sources; a stored ncu traffic figure is valid only for this hash."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "smem_swizzle_layouts_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current sources."""
    path = os.path.join(ROOT, "profiles", f"{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != _source_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi samples (every 20 ms); only those taken inside the timed region count."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t_start", 0.0), getattr(self, "t_end", float("inf"))
        inside = [ln for t, ln in self.lines if t0 <= t <= t1 + 0.02]
        for ln in inside:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                mx = float(parts[3])
            except ValueError:
                continue
            for name, val in zip(names, parts[6:10]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi sample fell inside the timed region"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, device) -> float:
    """The slowest rank's time: all-reduce MAX over the process group."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world_size: int, max_ms: float) -> float:
    """Whole-job rate: the units all ranks processed over the slowest rank's time (per second)."""
    return units_per_rank * world_size / (max_ms / 1e3)


def _torch_inputs(wl, dev, pinned=False):
    import torch
    in_fmt = wl.get("in_fmt", "bf16")
    M, N, K = wl["M"], wl["N"], wl["K"]
    A = si.matrix_bits(wl["seed"], M, K, wl["dist"], in_fmt, scale=wl["scale"], transpose=wl["a_major"] == "MN")
    B = si.matrix_bits(wl["seed"] + 1, K, N, wl["dist"], in_fmt, scale=wl["scale"], transpose=wl["b_major"] == "K")
    C = (si.matrix_bits(wl["seed"] + 2, M, N, wl["dist"], wl["out"], scale=wl["scale"])
         if wl["beta"] != 0.0 else None)
    host = [si.torch_from_bits(A, in_fmt), si.torch_from_bits(B, in_fmt),
            si.torch_from_bits(C, wl["out"]) if C is not None else None]
    if pinned:
        host = [h.pin_memory() if h is not None else None for h in host]
    devt = [h.to(dev) if h is not None else None for h in host]
    return (A, B, C), host, devt


def _run_ours(args, wl_name, wl, ws, rank, local):
    import torch
    import smem_swizzle_layouts_gb300 as g

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wl["out"]]
    M, N, K = wl["M"], wl["N"], wl["K"]
    in_type = 1 if wl.get("in_fmt", "bf16") == "bf16" else 0
    bits, host, (At, Bt, Ct) = _torch_inputs(wl, dev, pinned=True)
    D = torch.empty(M, N, dtype=tdt, device=dev)
    lda, ldb = At.stride(0), Bt.stride(0)
    am, bm = (0 if wl["a_major"] == "K" else 1), (0 if wl["b_major"] == "K" else 1)
    dt = {"f32": 0, "bf16": 1, "f16": 2}[wl["out"]]

    def step(Aa, Bb, Cc, Dd):
        g.gemm_ex(in_type, M, N, K, Aa, am, lda, Bb, bm, ldb, Cc, N if Cc is not None else 0, Dd, N, dt,
                  wl["alpha"], wl["beta"], options=wl["options"], stream=stream)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(At, Bt, Ct, D)
    st, word = g.gemm_last_device_status(stream)
    if st != g.OK:
        raise RuntimeError(f"device status {st} ({word:#x}) during warm-up")

    # ---- device-resident timing: per-launch events on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier()
    sampler.start()
    time.sleep(0.5)  # nvidia-smi is up and sampling before the timed region starts
    launches0 = g.gemm_launch_count()
    sampler.mark("t_start")
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_begin.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step(At, Bt, Ct, D)
            ends[i].record(stream)
        t_end.record(stream)
    barrier()
    sampler.mark("t_end")
    launches = g.gemm_launch_count() - launches0
    clocks = sampler.stop()
    st, word = g.gemm_last_device_status(stream)
    if st != g.OK:
        raise RuntimeError(f"device status {st} ({word:#x}) in the timed region")
    total_ms = t_begin.elapsed_time(t_end)
    per_launch = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if ws > 1:
        total_ms = max_over_ranks(total_ms, dev)

    # ---- end to end through the public API with host buffers
    hA, hB, hC = host
    hD = torch.empty(M, N, dtype=tdt).pin_memory()
    e2e_steps = max(1, min(args.steps, 10))
    barrier()
    with torch.cuda.stream(stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            At.copy_(hA, non_blocking=True)
            Bt.copy_(hB, non_blocking=True)
            if Ct is not None:
                Ct.copy_(hC, non_blocking=True)
            step(At, Bt, Ct, D)
            hD.copy_(D, non_blocking=True)
        e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = At.numel() * At.element_size() + Bt.numel() * Bt.element_size() + (
        Ct.numel() * Ct.element_size() if Ct is not None else 0)
    d2h = D.numel() * D.element_size()
    return dict(total_ms=total_ms, per_launch=per_launch, launches=launches, clocks=clocks, e2e_ms=e2e_ms,
                h2d=h2d, d2h=d2h, bits=bits)


def _oracle_rows_rate(wl, bits, target_s, max_rows=None, fixed_rows=None):
    """Time the oracle on the first R rows of the workload; returns (flop/s, rows, seconds, threads)."""
    from oracle import gemm as og
    A, B, C = bits
    M, N, K = wl["M"], wl["N"], wl["K"]
    in_fmt = wl.get("in_fmt", "bf16")
    threads = og.num_threads()

    def rows_of(R):
        if wl["a_major"] == "K":
            return A[:R], K
        return A, M  # MN-major A: all columns stay; rows are picked by the M extent below

    def run(R):
        Ar, lda = rows_of(R)
        Cr = C[:R] if C is not None else None
        t0 = time.perf_counter()
        og.gemm(R, N, K, Ar, B, in_fmt=in_fmt, a_major=wl["a_major"], b_major=wl["b_major"], lda=lda,
                C=Cr, c_fmt=wl["out"], ldc=N, alpha=wl["alpha"], beta=wl["beta"], threads=threads)
        return time.perf_counter() - t0

    if fixed_rows:
        t = run(fixed_rows)
        return 2.0 * fixed_rows * N * K / t, fixed_rows, t, threads
    R = min(M, max(1, threads))
    t = run(R)
    if t < target_s and R < M:
        R = min(M, max(R + 1, int(R * target_s / max(t, 1e-6))))
        if max_rows:
            R = min(R, max_rows)
        t = run(R)
    return 2.0 * R * N * K / t, R, t, threads


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    ws, rank, local = _dist_env()
    wl = WORKLOADS[args.workload]
    flops = 2.0 * wl["M"] * wl["N"] * wl["K"]
    config = {"workload": args.workload, "desc": wl["desc"], "M": wl["M"], "N": wl["N"], "K": wl["K"],
              "a_major": wl["a_major"], "b_major": wl["b_major"], "out": wl["out"], "alpha": wl["alpha"],
              "beta": wl["beta"], "inputs": f"{wl['dist']} x{wl['scale']}, seed {wl['seed']}",
              "l2": "operands larger than L2 (no flush)" if flops >= 2 * 4096 ** 3 else
                    "operands resident; no flush between steps",
              "parallelism": f"replicas x{max(ws, args.gpus)}"}
    metric = "GEMM TFLOP/s (bf16 in, fp32 accum)"

    if args.impl == "reference":
        if rank != 0:
            return
        bits = _torch_inputs_host_only(wl)
        # calibrate a row sample so that warm-up + timed steps take about two minutes
        per_step = max(0.5, 120.0 / (args.warmup + args.steps))
        _, R, _, threads = _oracle_rows_rate(wl, bits, target_s=per_step)
        rates = []
        for i in range(args.warmup + args.steps):
            rate, R, t, threads = _oracle_rows_rate(wl, bits, target_s=0.0, fixed_rows=R)
            if i >= args.warmup:
                rates.append(rate)
        value = statistics.median(rates) / 1e12
        sample = f"first {R} of {wl['M']} rows of the workload per step ({2.0 * R * wl['N'] * wl['K']:.3e} flop)"
        line = {"impl": "reference", "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    r = _run_ours(args, args.workload, wl, ws, rank, local)
    value = job_throughput(flops * args.steps, ws, r["total_ms"]) / 1e12
    kernel_ms = statistics.mean(r["per_launch"])
    achieved = flops / (kernel_ms / 1e3) / 1e12
    peaks, peak_src = _peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    traffic = _profiled_traffic(args.workload)
    line = {"metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["total_ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
            "e2e": {"value": flops / (r["e2e_ms"] / 1e3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "ms_per_step": r["e2e_ms"]},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
                         "traffic": traffic, "kernel_ms": kernel_ms},
            "gpu_launches": r["launches"], "clocks": r["clocks"]}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, R, t, threads = _oracle_rows_rate(wl, r["bits"], target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {R} of {wl['M']} rows of the same workload, {t:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def _torch_inputs_host_only(wl):
    in_fmt = wl.get("in_fmt", "bf16")
    M, N, K = wl["M"], wl["N"], wl["K"]
    A = si.matrix_bits(wl["seed"], M, K, wl["dist"], in_fmt, scale=wl["scale"], transpose=wl["a_major"] == "MN")
    B = si.matrix_bits(wl["seed"] + 1, K, N, wl["dist"], in_fmt, scale=wl["scale"], transpose=wl["b_major"] == "K")
    C = (si.matrix_bits(wl["seed"] + 2, M, N, wl["dist"], wl["out"], scale=wl["scale"])
         if wl["beta"] != 0.0 else None)
    return A, B, C


if __name__ == "__main__":
    main()
