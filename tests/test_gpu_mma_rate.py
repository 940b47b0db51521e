"""Tensor-pipe instruction rates on the GPU, from the stand-alone probe in
smem_swizzle_layouts_gb300/csrc/probes/mma_rate.cu: back-to-back tcgen05.mma
of 128 rows per SM x N = 256 with operands fixed in shared memory.

These pin the per-clock ratios behind the roofline denominators the bench
uses: every kind completes one such MMA per SM in about 128 cycles, so per
clock fp8 (K = 32) does twice and fp4 (K = 64) four times the bf16 (K = 16)
work, single CTAs and CTA pairs alike; copying three scale atoms into TMEM
before every NVFP4 MMA (the tcgen05.cp of a 128-byte stage) slows it down.
"""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "smem_swizzle_layouts_gb300", "csrc", "probes", "mma_rate.cu")


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    pytest.skip("nvcc not found")


def test_mma_instruction_rates(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = str(tmp_path / "mma_rate")
    subprocess.run([_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", SRC, "-o", exe],
                   check=True, capture_output=True, text=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    rates = {}
    for line in run.stdout.splitlines():
        kind, cg, cp, cycles, flop = line.split()
        rates[(kind, int(cg[2:]), int(cp[2:]))] = (float(cycles), float(flop))
    for key, (cycles, _) in rates.items():
        if key[2] == 0:
            assert 120.0 <= cycles <= 141.0, (key, cycles)   # one 128x256 MMA per SM per ~128 cycles
    bf16 = rates[("bf16", 1, 0)][1]
    assert abs(bf16 / 8192.0 - 1.0) < 0.08, bf16
    for kind, cg, ratio in (("bf16", 2, 1), ("e4m3", 1, 2), ("e4m3", 2, 2), ("mxfp8", 2, 2), ("mxfp4", 2, 4),
                            ("nvfp4", 2, 4)):
        assert abs(rates[(kind, cg, 0)][1] / bf16 / ratio - 1.0) < 0.05, (kind, cg, rates[(kind, cg, 0)])
    # three tcgen05.cp of scale atoms before every MMA cost the pipe time
    assert rates[("nvfp4", 2, 1)][0] > 1.2 * rates[("nvfp4", 2, 0)][0]
