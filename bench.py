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
        scale=0.1, seed=10, options=dict(cta_group=1, workspace=True),
        desc="4096^3 bf16, A and B K-major, N(0,1)*0.1, bf16 out, SW128, cta_group::1 with the library's default "
             "tile for the shape (256x224 on one CTA, two M=128 MMAs per B slice: 304 tiles, two full rounds, "
             "unsplit); the stream-K workspace it is given would split the ragged last wave of 128-row tiles"),
    "skinny_m16384_n128_k8192": dict(
        M=16384, N=128, K=8192, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="normal",
        scale=1.0, seed=30, options=None, bound="hbm", desc="M=16384 N=128 K=8192 bf16, N(0,1), bf16 out"),
    "skinny_m128_n16384_k4096": dict(
        M=128, N=16384, K=4096, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="normal",
        scale=1.0, seed=31, options=None, bound="hbm", desc="M=128 N=16384 K=4096 bf16, N(0,1), bf16 out"),
    "smallm_m32_n16384_k8192": dict(
        M=32, N=16384, K=8192, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="normal",
        scale=1.0, seed=32, options=None, bound="hbm",
        desc="M=32 N=16384 K=8192 bf16 (a decode-like small-M shape: B streamed from HBM), N(0,1), bf16 out, "
             "default plan: weight-stationary tcgen05.mma.ws tiles of 64 x 128"),
    "grouped64_n4096_k2048": dict(
        kind="grouped", M=0, N=4096, K=2048, problems=64, m_seed=5, a_major="K", b_major="K", out="bf16",
        alpha=1.0, beta=0.0, dist="uniform", scale=1.0, seed=100, options=None,
        desc="64 independent bf16 problems, M_i uniform in {128..4096} step 128 (rng 5), N=4096, K=2048, "
             "U[-1,1], bf16 out, one launch over a device-side problem list"),
    "square8192_fp8_pair": dict(
        M=8192, N=8192, K=8192, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="uniform",
        scale=1.0, seed=40, options=dict(cta_group=2, tile_n=256), in_fmt="e4m3", b_fmt="e4m3", peak_ratio=2.0,
        desc="8192^3 fp8 E4M3 x E4M3 (kind::f8f6f4), A and B K-major, U[-1,1], fp32 accumulate, bf16 out, "
             "cta_group::2 CTA pairs"),
    "square8192_mxfp8": dict(
        M=8192, N=8192, K=8192, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="uniform",
        scale=1.0, seed=50, options=None, in_fmt="e4m3", b_fmt="e4m3", mx=True, peak_ratio=2.0,
        desc="8192^3 block-scaled fp8 (MXFP8: E4M3 with one E8M0 scale per 32 elements of K, codes U{124..130}; "
             "tcgen05 kind::mxf8f6f4), A and B K-major, U[-1,1], fp32 accumulate, bf16 out, 256x256 CTA-pair tiles"),
    "square8192_nvfp4": dict(
        M=8192, N=8192, K=8192, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="fp4",
        scale=1.0, seed=60, options=None, fp4="nvfp4", peak_ratio=6.0,
        desc="8192^3 block-scaled fp4 (NVFP4: packed E2M1, all sixteen codes, one UE4M3 scale per 16 elements "
             "of K from {1/4..6}; tcgen05 kind::mxf4nvf4), A and B K-major, fp32 accumulate, bf16 out, "
             "256x256 CTA-pair tiles"),
    "square8192_mxfp4": dict(
        M=8192, N=8192, K=8192, a_major="K", b_major="K", out="bf16", alpha=1.0, beta=0.0, dist="fp4",
        scale=1.0, seed=70, options=None, fp4="mxfp4", peak_ratio=6.0,
        desc="8192^3 block-scaled fp4 (MXFP4: packed E2M1, all sixteen codes, one E8M0 scale per 32 elements "
             "of K, codes U{124..130}; tcgen05 kind::mxf4), A and B K-major, fp32 accumulate, bf16 out, "
             "256x256 CTA-pair tiles"),
    "single_tile_128x128x32_f16": dict(
        M=128, N=128, K=32, a_major="K", b_major="MN", out="f32", alpha=1.0, beta=0.0, dist="uniform",
        scale=1.0, seed=0, options=None, in_fmt="f16",
        desc="D[128x128] fp32 = A[128x32] fp16 K-major x B[32x128] fp16 MN-major, two m128n128k16 MMAs"),
}
DEFAULT_WORKLOAD = "square8192_pair_f32_beta1"


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


# Published (not measured) per-GPU figures, reported beside the measured
# denominators: NVIDIA's HGX B300 sheet gives 36 PFLOP/s bf16 per 8 GPUs with
# 2:4 sparsity, i.e. 2.25 PFLOP/s dense per GPU, and 8 TB/s of HBM3e.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_BF16_SOURCE = "nominal dense bf16 2250 TFLOP/s (NVIDIA HGX B300: 36 PFLOP/s sparse per 8 GPUs)"
NOMINAL_HBM_GBS = 8000.0
NOMINAL_HBM_SOURCE = "nominal HBM3e 8000 GB/s (NVIDIA GB300 sheet)"

KERNEL_SOURCES = ("gemm_kernel.cuh", "ptx.cuh", "descriptors.cuh")


def _code_lines(text):
    """The source without its // comments and blank lines (what the compiler sees of it)."""
    out = []
    for line in text.splitlines():
        code = re.sub(r"//.*$", "", line).rstrip()
        if code.strip():
            out.append(code)
    return "\n".join(out)


def _source_hash(read=None):
    """Hash of the device-code sources, comments left out; a stored ncu traffic figure is valid
    only for this hash. `read(name)` returns a source's text (default: the working tree)."""
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "smem_swizzle_layouts_gb300", "csrc", name)) as f:
                return f.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(name.encode())
        h.update(_code_lines(read(name)).encode())
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
            # the region was shorter than the sampling period: report the
            # nearest sample on each side of it, labelled as such
            before = [(t, ln) for t, ln in self.lines if t < t0]
            after = [(t, ln) for t, ln in self.lines if t > t1 + 0.02]
            near = {}
            for label, pick in (("before", before[-1:]), ("after", after[:1])):
                for t, ln in pick:
                    parts = [p.strip() for p in ln.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        near[label] = {"sm_mhz": float(parts[2]), "sm_max_mhz": float(parts[3]),
                                       "ms_from_region": round(1e3 * (t - t0 if label == "before" else t - t1), 1),
                                       "reasons": [n for n, v in zip(names, parts[6:10])
                                                   if v.lower() in ("active", "1")]}
                    except ValueError:
                        continue
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi sample fell inside the timed region; nearest samples outside it follow",
                    "nearest_outside": near}
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


FP4_KINDS = {"nvfp4": (0, 16, "ue4m3"), "mxfp4": (1, 32, "e8m0")}
UE4M3_POOL = np.array([(e << 3) | m for e in (5, 6, 7, 8, 9) for m in (0, 4)], np.uint8)  # 1/4 .. 6


def _fp4_inputs(wl):
    """Packed E2M1 operands (M x K/2, N x K/2 bytes) and row-major scale codes of an fp4 workload."""
    code, block, scale = FP4_KINDS[wl["fp4"]]
    M, N, K = wl["M"], wl["N"], wl["K"]
    A = si.pack_fp4(si.fp4_codes(wl["seed"], M, K))
    B = si.pack_fp4(si.fp4_codes(wl["seed"] + 1, N, K))
    nb = (K + block - 1) // block
    if scale == "ue4m3":
        z = si.scale_codes(wl["seed"] + 2, M + N, nb, 0, len(UE4M3_POOL) - 1)
        sa, sb = UE4M3_POOL[z[:M]], UE4M3_POOL[z[M:]]
    else:
        sa, sb = si.scale_codes(wl["seed"] + 2, M, nb), si.scale_codes(wl["seed"] + 3, N, nb)
    return A, B, sa, sb


def _mx_codes(wl):
    """Seeded E8M0 scale codes of a block-scaled workload (row-major, one per 32 elements of K)."""
    nb = (wl["K"] + 31) // 32
    return si.scale_codes(wl["seed"] + 3, wl["M"], nb), si.scale_codes(wl["seed"] + 4, wl["N"], nb)


def _torch_inputs(wl, dev, pinned=False):
    import torch
    in_fmt = wl.get("in_fmt", "bf16")
    M, N, K = wl["M"], wl["N"], wl["K"]
    b_fmt = wl.get("b_fmt", in_fmt)
    A = si.matrix_bits(wl["seed"], M, K, wl["dist"], in_fmt, scale=wl["scale"], transpose=wl["a_major"] == "MN")
    B = si.matrix_bits(wl["seed"] + 1, K, N, wl["dist"], b_fmt, scale=wl["scale"], transpose=wl["b_major"] == "K")
    C = (si.matrix_bits(wl["seed"] + 2, M, N, wl["dist"], wl["out"], scale=wl["scale"])
         if wl["beta"] != 0.0 else None)
    host = [si.torch_from_bits(A, in_fmt), si.torch_from_bits(B, b_fmt),
            si.torch_from_bits(C, wl["out"]) if C is not None else None]
    if pinned:
        host = [h.pin_memory() if h is not None else None for h in host]
    devt = [h.to(dev) if h is not None else None for h in host]
    return (A, B, C), host, devt


class _DeviceSet:
    """Device buffers and a launch for one slot of the end-to-end pipeline."""

    def __init__(self, pairs, step, outs):
        self.pairs, self.step, self._outs = pairs, step, outs

    def outputs(self):
        return self._outs


class GemmJob:
    """One GEMM per step through gemm_ex."""

    def __init__(self, wl, dev, stream, options):
        import torch
        import smem_swizzle_layouts_gb300 as g
        self.g, self.wl, self.stream = g, wl, stream
        tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wl["out"]]
        self.M, self.N, self.K = wl["M"], wl["N"], wl["K"]
        self.in_type = 1 if wl.get("in_fmt", "bf16") == "bf16" else 0
        fp4_scales = None
        if wl.get("fp4"):
            code, block, scale = FP4_KINDS[wl["fp4"]]
            A4, B4, sa, sb = _fp4_inputs(wl)
            fill = 0x38 if scale == "ue4m3" else 127
            host = [torch.from_numpy(A4.reshape(-1)).pin_memory(), torch.from_numpy(B4.reshape(-1)).pin_memory(), None]
            devt = [h.to(dev) if h is not None else None for h in host]
            host_s = [torch.from_numpy(si.mx_scale_atoms(c, n, self.K, block, fill)).pin_memory()
                      for c, n in ((sa, self.M), (sb, self.N))]
            fp4_scales = [h.to(dev) for h in host_s]
            self.bits = (A4, B4, None, sa, sb)
        else:
            self.bits, host, devt = _torch_inputs(wl, dev, pinned=True)
        self.A, self.B, self.C = devt
        self.D = torch.empty(self.M, self.N, dtype=tdt, device=dev)
        self.hD = torch.empty(self.M, self.N, dtype=tdt).pin_memory()
        self.pairs = [(h, d) for h, d in zip(host, devt) if h is not None]
        self.am = 0 if wl["a_major"] == "K" else 1
        self.bm = 0 if wl["b_major"] == "K" else 1
        self.dt = {"f32": 0, "bf16": 1, "f16": 2}[wl["out"]]
        if options and options.get("workspace") is True:
            # stream-K workspace, zeroed once ("workspace": true in the options)
            options = dict(options, workspace=torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8,
                                                          device=dev))
        self.options = options
        self.flops = 2.0 * self.M * self.N * self.K
        # arguments marshalled once; each step is one call into the C ABI
        fp8 = None
        if wl.get("in_fmt") in ("e4m3", "e5m2"):
            codes = {"e4m3": g.FP8_E4M3, "e5m2": g.FP8_E5M2}
            fp8 = (codes[wl["in_fmt"]], codes[wl.get("b_fmt", wl["in_fmt"])])
        scales = None
        if fp4_scales is not None:
            self.pairs += list(zip(host_s, fp4_scales))
            scales = fp4_scales
        if wl.get("mx"):
            sa, sb = _mx_codes(wl)
            self.bits = self.bits + (sa, sb)
            host_s = [torch.from_numpy(si.mx_scale_atoms(c, n, self.K)).pin_memory()
                      for c, n in ((sa, self.M), (sb, self.N))]
            scales = [h.to(dev) for h in host_s]
            self.pairs += list(zip(host_s, scales))
        lda = self.K if wl.get("fp4") else self.A.stride(0)
        ldb = self.K if wl.get("fp4") else self.B.stride(0)
        fp4 = FP4_KINDS[wl["fp4"]][0] if wl.get("fp4") else None

        def make_call(A, B, C, D, sc):
            return g.GemmCall(self.in_type, self.M, self.N, self.K, A, self.am, lda, B, self.bm, ldb, C,
                              self.N if C is not None else 0, D, self.N, self.dt, wl["alpha"], wl["beta"],
                              options=options, stream=stream, fp8=fp8, scales=sc, fp4=fp4)

        self._make_call, self._scales = make_call, scales
        self.call = make_call(self.A, self.B, self.C, self.D, scales)

    def step(self):
        self.call()

    def outputs(self):
        return [(self.D, self.hD)]

    def second_set(self):
        """A second set of device buffers (same host buffers) with its own pre-marshalled call."""
        import torch
        twin = {id(d): torch.empty_like(d) for _, d in self.pairs}
        D2 = torch.empty_like(self.D)
        call = self._make_call(twin[id(self.A)], twin[id(self.B)],
                               twin[id(self.C)] if self.C is not None else None, D2,
                               [twin[id(s)] for s in self._scales] if self._scales else None)
        return _DeviceSet([(h, twin[id(d)]) for h, d in self.pairs], call, [(D2, self.hD)])

    def oracle_rate(self, target_s, fixed_rows=None):
        return _oracle_rows_rate(self.wl, self.bits, target_s, fixed_rows=fixed_rows)


class GroupedJob:
    """One grouped launch over a 64-problem list per step (gemm_bf16_grouped)."""

    def __init__(self, wl, dev, stream, options):
        import torch
        import smem_swizzle_layouts_gb300 as g
        self.g, self.wl, self.stream = g, wl, stream
        N, K = wl["N"], wl["K"]
        rng = np.random.default_rng(wl["m_seed"])
        self.Ms = [int(x) * 128 for x in rng.integers(1, 33, wl["problems"])]
        self.N, self.K = N, K
        self.hA, self.hB, self.hD, self.probs, self.bits = [], [], [], [], []
        self.pairs, self.outs = [], []
        for i, M in enumerate(self.Ms):
            A = si.matrix_bits(wl["seed"] + 3 * i, M, K, wl["dist"], "bf16")
            B = si.matrix_bits(wl["seed"] + 3 * i + 1, K, N, wl["dist"], "bf16", transpose=True)
            hA = si.torch_from_bits(A, "bf16").pin_memory()
            hB = si.torch_from_bits(B, "bf16").pin_memory()
            dA, dB = hA.to(dev), hB.to(dev)
            dD = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            hD = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
            self.pairs += [(hA, dA), (hB, dB)]
            self.outs.append((dD, hD))
            self.bits.append((A, B))
            self.probs.append(dict(M=M, N=N, K=K, A=dA, B=dB, C=None, D=dD, lda=K, ldb=K, ldc=0, ldd=N))
        self.ws_bytes = g.gemm_grouped_workspace_size(len(self.Ms))
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.flops = float(sum(2.0 * M * N * K for M in self.Ms))
        self.options = options

    def _launch(self, probs, ws):
        if self.options:
            self.g.gemm_grouped_ex(1, probs, 0, 0, 1, self.wl["alpha"], self.wl["beta"], ws, self.ws_bytes,
                                   options=self.options, stream=self.stream)
        else:
            self.g.gemm_bf16_grouped(probs, 0, 0, 1, self.wl["alpha"], self.wl["beta"], ws, self.ws_bytes,
                                     stream=self.stream)

    def step(self):
        self._launch(self.probs, self.ws)

    def outputs(self):
        return self.outs

    def second_set(self):
        """A second set of device buffers (same host buffers) with its own problem list and workspace."""
        import torch
        twin = {id(d): torch.empty_like(d) for _, d in self.pairs}
        outs = [(torch.empty_like(d), h) for d, h in self.outs]
        probs = [dict(q, A=twin[id(q["A"])], B=twin[id(q["B"])], D=o[0]) for q, o in zip(self.probs, outs)]
        ws = torch.empty_like(self.ws)

        def call():
            self._launch(probs, ws)
        return _DeviceSet([(h, twin[id(d)]) for h, d in self.pairs], call, outs)

    def oracle_rate(self, target_s, fixed_rows=None):
        A, B = self.bits[0]
        sub = dict(self.wl, M=self.Ms[0], a_major="K", b_major="K", out="bf16", beta=0.0)
        return _oracle_rows_rate(sub, (A, B, None), target_s, fixed_rows=fixed_rows)


def _run_ours(args, wl_name, wl, ws, rank, local):
    import torch
    import smem_swizzle_layouts_gb300 as g

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    options = wl.get("options")
    if args.options:
        options = dict(options or {}, **json.loads(args.options))
    job = (GroupedJob if wl.get("kind") == "grouped" else GemmJob)(wl, dev, stream, options)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            job.step()
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
            job.step()
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
    # ---- end to end: every step uploads its inputs from pinned host memory,
    # runs the GEMM and reads its result back. Steps are pipelined the way a
    # stream of independent GEMMs would be: uploads, compute and downloads on
    # three streams over two device buffer sets, so step i+1 uploads while
    # step i computes and step i-1 downloads (events guard each set's reuse).
    e2e_steps = max(2, min(args.steps, 20))
    sets = [job, job.second_set()]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    ev_in, ev_cmp, ev_out = ([ev() for _ in range(e2e_steps)] for _ in range(3))
    for S in sets:  # first use of the second set's call outside the timed region
        with torch.cuda.stream(stream):
            S.step()
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        S = sets[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_cmp[i - 2])  # this set's inputs are free once its last GEMM ran
            for h, d in S.pairs:
                d.copy_(h, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])  # its output buffer has been read back
        S.step()
        ev_cmp[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[i])
            for d, h in S.outputs():
                h.copy_(d, non_blocking=True)
            ev_out[i].record(s_out)
    s_out.wait_event(ev_in[e2e_steps - 1])
    e1.record(s_out)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = sum(d.numel() * d.element_size() for _, d in job.pairs)
    d2h = sum(d.numel() * d.element_size() for d, _ in job.outputs())
    return dict(total_ms=total_ms, per_launch=per_launch, launches=launches, clocks=clocks, e2e_ms=e2e_ms,
                h2d=h2d, d2h=d2h, job=job, options=options)


def _oracle_rows_rate(wl, bits, target_s, max_rows=None, fixed_rows=None):
    """Time the oracle on the first R rows of the workload; returns (flop/s, rows, seconds, threads)."""
    from oracle import gemm as og
    A, B, C = bits[:3]
    scales = bits[3:] if len(bits) > 3 else None
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
        kw = dict(in_fmt=in_fmt, b_fmt=wl.get("b_fmt", in_fmt), a_major=wl["a_major"], b_major=wl["b_major"],
                  lda=lda, C=Cr, c_fmt=wl["out"], ldc=N, alpha=wl["alpha"], beta=wl["beta"], threads=threads)
        t0 = time.perf_counter()
        if wl.get("fp4"):
            _, block, scale = FP4_KINDS[wl["fp4"]]
            og.gemm_fp4(R, N, K, A[:R], B, scales[0][:R], scales[1], block=block, scale=scale, C=None,
                        alpha=wl["alpha"], beta=wl["beta"], threads=threads)
        elif scales is not None:
            og.gemm_mx(R, N, K, Ar, B, scales[0][:R], scales[1], **kw)
        else:
            og.gemm(R, N, K, Ar, B, **kw)
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


def _algorithmic_bytes(wl, job):
    """Minimum HBM bytes of one step: read A, B (and C), write D once."""
    ob = 4 if wl["out"] == "f32" else 2
    if wl.get("kind") == "grouped":
        N, K = wl["N"], wl["K"]
        return float(sum((M * K + K * N) * 2 + M * N * ob for M in job.Ms))
    M, N, K = wl["M"], wl["N"], wl["K"]
    eb = 1 if wl.get("in_fmt") in ("e4m3", "e5m2") else 0.5 if wl.get("fp4") else 2
    block = FP4_KINDS[wl["fp4"]][1] if wl.get("fp4") else 32
    sf = (M + N) * ((K + block - 1) // block) if (wl.get("mx") or wl.get("fp4")) else 0  # one scale byte per block
    return float((M * K + K * N) * eb + sf + M * N * ob * (2 if wl["beta"] != 0.0 else 1))


def _reference_line(args, wl, config, metric):
    """The oracle timed on the host cores on a bounded row sample of the workload."""
    if wl.get("kind") == "grouped":
        rng = np.random.default_rng(wl["m_seed"])
        M0 = int(rng.integers(1, 33, wl["problems"])[0]) * 128
        sub = dict(wl, M=M0)
        A = si.matrix_bits(wl["seed"], M0, wl["K"], wl["dist"], "bf16")
        B = si.matrix_bits(wl["seed"] + 1, wl["K"], wl["N"], wl["dist"], "bf16", transpose=True)
        bits, rows_of = (A, B, None), f"problem 0 (M={M0})"
    else:
        sub, bits, rows_of = wl, _host_bits(wl), f"{wl['M']} rows"
    # calibrate a row sample so that warm-up + timed steps take about two minutes
    per_step = max(0.5, 120.0 / (args.warmup + args.steps))
    _, R, _, threads = _oracle_rows_rate(sub, bits, target_s=per_step)
    rates = []
    for i in range(args.warmup + args.steps):
        rate, R, t, threads = _oracle_rows_rate(sub, bits, target_s=0.0, fixed_rows=R)
        if i >= args.warmup:
            rates.append(rate)
    value = statistics.median(rates) / 1e12
    sample = f"first {R} of {rows_of} per step ({2.0 * R * sub['N'] * sub['K']:.3e} flop)"
    return {"impl": "reference", "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--options", default="", help="JSON overrides of the workload's gemm options (ablations)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    ws, rank, local = _dist_env()
    wl = WORKLOADS[args.workload]
    config = {"workload": args.workload, "desc": wl["desc"], "M": wl["M"], "N": wl["N"], "K": wl["K"],
              "a_major": wl["a_major"], "b_major": wl["b_major"], "out": wl["out"], "alpha": wl["alpha"],
              "beta": wl["beta"], "inputs": f"{wl['dist']} x{wl['scale']}, seed {wl['seed']}",
              "parallelism": f"replicas x{max(ws, args.gpus)}"}
    if args.options:
        config["options"] = json.loads(args.options)
    metric = "GEMM TFLOP/s (bf16 in, fp32 accum) and % of GB300 dense BF16 tensor peak"
    if wl.get("in_fmt") in ("e4m3", "e5m2"):
        metric = "GEMM TFLOP/s (fp8 in, fp32 accum) and % of GB300 dense FP8 tensor peak"
    if wl.get("mx"):
        metric = "GEMM TFLOP/s (MXFP8 block-scaled fp8 in, fp32 accum) and % of GB300 dense FP8 tensor peak"
    if wl.get("fp4"):
        metric = (f"GEMM TFLOP/s ({wl['fp4'].upper()} block-scaled fp4 in, fp32 accum) and % of GB300 dense "
                  "FP4 tensor peak")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(_reference_line(args, wl, config, metric)))
        return

    import torch
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    r = _run_ours(args, args.workload, wl, ws, rank, local)
    job = r["job"]
    flops = job.flops
    bytes_alg = _algorithmic_bytes(wl, job)
    config["l2"] = ("operands larger than L2 (129 MB): no flush between steps" if bytes_alg > 129e6 else
                    "operands fit in L2; steps run back to back without a flush")
    value = job_throughput(flops * args.steps, ws, r["total_ms"]) / 1e12
    # the roofline's achieved rate uses the mean launch time; median and min
    # over the same launches are reported beside it
    kernel_ms = statistics.mean(r["per_launch"])
    kernel_stats = {"kernel_ms_median": statistics.median(r["per_launch"]), "kernel_ms_min": min(r["per_launch"]),
                    "launches_timed": len(r["per_launch"])}
    peaks, peak_src = _peaks()
    traffic = _profiled_traffic(args.workload) if not args.options else None
    if wl.get("bound") == "hbm":
        achieved = bytes_alg / (kernel_ms / 1e3) / 1e9
        peak = float(peaks.get("hbm_gbs", 6800.0))
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_src} hbm_gbs", "traffic": traffic, "kernel_ms": kernel_ms, **kernel_stats,
                "algorithmic_bytes": bytes_alg,
                "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "nominal_source": NOMINAL_HBM_SOURCE}
    else:
        achieved = flops / (kernel_ms / 1e3) / 1e12
        ratio = float(wl.get("peak_ratio", 1.0))  # nominal dense peaks over bf16: fp8 4.5/2.25, fp4 13.5/2.25
        peak = float(peaks.get("bf16_tflops", 1900.0)) * ratio
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peak_src} bf16_tflops (burst)" + (
                    f" x {ratio:g} (nominal {'fp4' if wl.get('fp4') else 'fp8'}/bf16 dense ratio)" if ratio != 1.0 else ""),
                "frac_of_sustained": achieved / (float(peaks.get("bf16_tflops_sustained", peak)) * ratio),
                "frac_of_nominal": achieved / (NOMINAL_BF16_TFLOPS * ratio),
                "nominal_source": NOMINAL_BF16_SOURCE + (f" x {ratio:g}" if ratio != 1.0 else ""),
                "traffic": traffic, "kernel_ms": kernel_ms, **kernel_stats, "algorithmic_bytes": bytes_alg}
    line = {"metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["total_ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e2m1" if wl.get("fp4") else wl.get("in_fmt", "bf16"),
            "data": "synthetic",
            "config": config,
            "e2e": {"value": flops / (r["e2e_ms"] / 1e3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "ms_per_step": r["e2e_ms"]},
            "roofline": roof, "gpu_launches": r["launches"], "clocks": r["clocks"]}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, R, t, threads = job.oracle_rate(args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {R} rows of the same workload ({t:.1f} s)"}
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def _torch_inputs_host_only(wl):
    in_fmt = wl.get("in_fmt", "bf16")
    M, N, K = wl["M"], wl["N"], wl["K"]
    A = si.matrix_bits(wl["seed"], M, K, wl["dist"], in_fmt, scale=wl["scale"], transpose=wl["a_major"] == "MN")
    B = si.matrix_bits(wl["seed"] + 1, K, N, wl["dist"], wl.get("b_fmt", in_fmt), scale=wl["scale"],
                       transpose=wl["b_major"] == "K")
    C = (si.matrix_bits(wl["seed"] + 2, M, N, wl["dist"], wl["out"], scale=wl["scale"])
         if wl["beta"] != 0.0 else None)
    if wl.get("mx"):
        return (A, B, C) + _mx_codes(wl)
    return A, B, C


def _host_bits(wl):
    """Host-side inputs of a workload for the oracle legs."""
    if wl.get("fp4"):
        A4, B4, sa, sb = _fp4_inputs(wl)
        return (A4, B4, None, sa, sb)
    return _torch_inputs_host_only(wl)


if __name__ == "__main__":
    main()
