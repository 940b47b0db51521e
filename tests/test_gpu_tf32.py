"""GPU parity of the TF32 GEMM (gemm_ex in_type 2, tcgen05 kind::tf32) against the oracle.

The operands are fp32 words; kind::tf32 multiplies their TF32 part. MN-major
operands are staged in the 128-byte swizzle with 32-byte atoms (descriptor
code 1, "LBO, SBO and SWZ for a tcgen05 tile", section 4), the layout the
oracle reads as Swizzle(2, 5, 2) with 4-row K bands: an exact GEMM through
it checks that reading of the page's raw value 1 on the hardware. Integer
inputs are bit-exact; normal inputs (TF32-representable) are held to the
parity tolerance; one case pins the oracle's TF32 reading (truncation).
"""
import numpy as np
import pytest

import seeded_inputs as si
from oracle import gemm as og
from oracle import layouts as L
from test_gpu_parity import SWZ_PARAM, TDT, _out_bits, run_case, sample_entries

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("K", "MN"), ("MN", "K"), ("MN", "MN")])
@pytest.mark.parametrize("opts", [dict(cta_group=1, tile_n=256), dict(cta_group=1, tile_n=128),
                                  dict(cta_group=2, tile_n=256)], ids=["cg1n256", "cg1n128", "pairs"])
def test_tf32_majors_integer_exact(g, a_major, b_major, opts):
    # MN-major operands go through descriptor code 1 (32-byte atoms)
    run_case(g, 384, 520, 256, in_fmt="tf32", a_major=a_major, b_major=b_major, dist="int4", exact=True,
             options=opts)


@pytest.mark.parametrize("M,N,K", [(128, 128, 8), (100, 300, 200), (640, 384, 520), (1000, 1000, 1000), (7, 264, 40)])
def test_tf32_ragged_shapes_exact(g, M, N, K):
    run_case(g, M, N, K, in_fmt="tf32", a_major="K", b_major="MN", dist="int4", exact=True, seed=M + N + K)


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_tf32_normal_inputs_alpha_beta_within_tolerance(g, out):
    run_case(g, 512, 600, 768, in_fmt="tf32", a_major="MN", b_major="K", dist="normal", out=out, alpha=0.5,
             beta=-1.25, seed=19)


def test_tf32_reads_the_truncated_operand(g):
    # A holds values in [1, 2) on the TF32 grid plus junk in the 13 dropped fraction bits; B small
    # integers. Every product and sum is exact in fp32, so D is bit-exact against the oracle's
    # truncating reading -- and differs from it wherever the junk is at least half a TF32 unit
    M, N, K = 256, 256, 64
    rng = np.random.default_rng(7)
    a = (1.0 + rng.integers(0, 1024, (M, K)) / 1024.0).astype(np.float32).view(np.uint32)
    a = a | rng.integers(0, 0x2000, (M, K)).astype(np.uint32)
    b = si.matrix_bits(8, K, N, "int4", "tf32", transpose=True)
    At = torch.from_numpy(a.view(np.int32)).view(torch.float32).to(DEV)
    Bt = torch.from_numpy(b.view(np.int32)).view(torch.float32).to(DEV)
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    g.gemm_ex(2, M, N, K, At, 0, K, Bt, 0, K, None, 0, D, N, 0, 1.0, 0.0)
    ref, _ = og.gemm(M, N, K, a, b, in_fmt="tf32", a_major="K", b_major="K")
    rounded, _ = og.gemm(M, N, K, si.to_storage(si.bits_to_float64(a, "f32"), "tf32"), b, in_fmt="tf32",
                         a_major="K", b_major="K")
    assert (ref != rounded).mean() > 0.5           # the two readings differ here
    assert np.array_equal(_out_bits(D, "f32"), og.round_bits(ref, "f32"))


@pytest.mark.parametrize("rows,bk", [(128, 32), (256, 32), (128, 64)])
def test_tf32_code1_descriptor_words_match_oracle(g, rows, bk):
    n = bk // 8
    out = torch.zeros(n + 1, dtype=torch.int64, device=DEV)
    base = 8 * 1024
    g.gemm_debug_descriptors(1, SWZ_PARAM[L.ATOM32], rows, bk, base, n, 1, 256, 4, 0, 1, out)
    words = [int(x) & (2 ** 64 - 1) for x in out.cpu().tolist()]
    for j in range(n):
        assert words[j] == L.encode_smem_desc(L.stage_slice_desc("MN", L.ATOM32, rows, bk, 4, j, base)), j


def test_tf32_square_4096_sampled(g):
    M = N = K = 4096
    run_case(g, M, N, K, in_fmt="tf32", a_major="K", b_major="MN", dist="normal", out="f32", seed=23,
             sample=sample_entries(M, N, 2048, seed=6))
