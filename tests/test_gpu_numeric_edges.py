"""GPU parity at the numeric edges of the method, bit for bit against the oracle.

* Output rounding at the ends of the 16-bit output types: integer-valued
  operands make the fp32 accumulator exact, and a power-of-two alpha moves it
  past the largest finite bf16/f16 value (the result must be +-inf, and the
  largest finite value itself must survive) or into the subnormal range (the
  result must be rounded to nearest-even on the subnormal grid, not flushed).
  The reference is the exact value rounded once by ``oracle.round_bits``.
* Block-scaled operands ("06 Blackwell Tensor Core - tcgen05 MMA",
  "Block-Scaled MMA"): E8M0 scale codes at both ends of the finite range
  (0 = 2^-127 against 254 = 2^127, paired so the scaled products stay finite),
  UE4M3 subnormal scales (exponent field 0) and UE4M3's largest finite code
  0x7E (448). Operand values and scales are chosen so that every product and
  partial sum stays exact in fp32, so these cases are bit-exact too.

Each case first checks, on the oracle side, that its inputs really reach the
edge it is named for (some +-inf, some subnormal outputs, ...).
"""
import numpy as np
import pytest

import seeded_inputs as si
from oracle import gemm as og
from test_gpu_fp4 import run_fp4
from test_gpu_mx import run_mx
from test_gpu_parity import TDT, _out_bits, _ru, _to_dev

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
OUT = {"f32": 0, "bf16": 1, "f16": 2}
# smallest normal and largest finite value of each output type
MIN_NORMAL = {"bf16": 2.0 ** -126, "f16": 2.0 ** -14, "f32": 2.0 ** -126}
MAX_FINITE = {"bf16": 255 * 2.0 ** 120, "f16": 65504.0}


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


def _edge_gemm(g, M, N, K, out, alpha, *, seed, options=None, in_fmt="bf16"):
    """Integer-valued operands in [-4, 4] through gemm_ex; returns (got bits, oracle value)."""
    lda, ldb, ldd = _ru(K, 8), _ru(K, 8), _ru(N, 8)
    A = si.matrix_bits(seed, M, K, "int4", in_fmt, ld=lda)
    B = si.matrix_bits(seed + 1, K, N, "int4", in_fmt, transpose=True, ld=ldb)
    At, Bt = _to_dev(A, in_fmt), _to_dev(B, in_fmt)
    Dt = torch.full((M, ldd), float("nan"), dtype=TDT[out], device=DEV)
    g.gemm_ex(1 if in_fmt == "bf16" else 0, M, N, K, At, 0, lda, Bt, 0, ldb, None, 0, Dt, ldd, OUT[out],
              alpha, 0.0, options=options)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, f"device status word {word:#x}"
    ref, _ = og.gemm(M, N, K, A, B, in_fmt=in_fmt, a_major="K", b_major="K", lda=lda, ldb=ldb, alpha=alpha)
    return _out_bits(Dt, out)[:, :N], ref


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("out,alpha", [("bf16", 2.0 ** 120), ("f16", 2.0 ** 8)])
def test_output_overflows_to_inf(g, out, alpha, cta_group):
    # |acc| >= 256 overflows to +-inf; for bf16, |acc| = 255 is exactly the largest finite value
    got, ref = _edge_gemm(g, 384, 320, 1024, out, alpha, seed=900 + cta_group, options=dict(cta_group=cta_group))
    want = og.round_bits(ref, out)
    dec = si.bits_to_float64(want, out)
    assert np.isinf(dec).sum() > 1000 and (dec == np.inf).any() and (dec == -np.inf).any()
    assert np.isfinite(dec).sum() > 1000
    if out == "bf16":
        assert (np.abs(dec) == MAX_FINITE["bf16"]).any()
    assert np.array_equal(got, want)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("out,alpha", [("bf16", 2.0 ** -140), ("f16", 2.0 ** -30), ("f32", 2.0 ** -140)])
def test_output_subnormal_range_rounds_to_nearest_even(g, out, alpha, cta_group):
    # alpha * acc lands below the smallest normal value of the output type; for the
    # 16-bit types most results need rounding on the subnormal grid, ties included
    got, ref = _edge_gemm(g, 256, 264, 512, out, alpha, seed=910 + cta_group, options=dict(cta_group=cta_group))
    want = og.round_bits(ref, out)
    dec = si.bits_to_float64(want, out)
    sub = (dec != 0) & (np.abs(dec) < MIN_NORMAL[out])
    assert sub.sum() > 0.5 * dec.size
    if out != "f32":
        assert (dec != ref).sum() > 0.25 * dec.size   # rounding really happens
    assert np.array_equal(got, want)


def test_output_edges_on_fp16_inputs_and_64_row_tiles(g):
    # the same overflow edge through fp16 operands and the M = 64 (Layout F) epilogue
    got, ref = _edge_gemm(g, 64, 384, 1024, "f16", 2.0 ** 8, seed=920, in_fmt="f16", options=dict(tile_m=64))
    want = og.round_bits(ref, "f16")
    assert np.isinf(si.bits_to_float64(want, "f16")).any()
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- block-scaled scale codes at their edges

@pytest.mark.parametrize("options", [None, dict(cta_group=2)])
@pytest.mark.parametrize("a_rng,b_rng", [((0, 3), (251, 254)), ((251, 254), (0, 3))])
def test_mxfp8_e8m0_codes_at_both_ends(g, a_rng, b_rng, options):
    # 2^-127 .. 2^-124 against 2^124 .. 2^127: the scale products stay within 2^+-3
    run_mx(g, 384, 320, 512, exact=True, seed=930, lo=a_rng[0], hi=a_rng[1], b_lo=b_rng[0], b_hi=b_rng[1],
           options=options)


def test_mxfp8_e8m0_extremes_on_256_wide_pairs_with_bf16_output(g):
    # the single-accumulator 256 x 256 pair tiles and their early-release epilogue
    run_mx(g, 2048, 2048, 512, exact=True, seed=931, out="bf16", lo=0, hi=3, b_lo=251, b_hi=254)


UE4M3_SUBNORMAL = np.arange(1, 8, dtype=np.uint8)          # exponent field 0: m * 2^-9
UE4M3_TOP = np.array([0x7E, 0x7C, 0x78, 0x70], np.uint8)   # 448 (largest finite), 384, 256, 128


@pytest.mark.parametrize("options", [None, dict(cta_group=2)])
@pytest.mark.parametrize("a_pool,b_pool", [(UE4M3_SUBNORMAL, UE4M3_TOP), (UE4M3_TOP, UE4M3_SUBNORMAL),
                                           (UE4M3_SUBNORMAL, UE4M3_SUBNORMAL)])
def test_nvfp4_ue4m3_subnormal_and_largest_scales(g, a_pool, b_pool, options):
    run_fp4(g, 384, 320, 512, "nvfp4", seed=940, a_pool=a_pool, b_pool=b_pool, options=options)


def test_nvfp4_ue4m3_edges_with_bf16_output(g):
    run_fp4(g, 2048, 2048, 256, "nvfp4", seed=941, out="bf16", a_pool=UE4M3_SUBNORMAL, b_pool=UE4M3_TOP)


@pytest.mark.parametrize("options", [None, dict(cta_group=2)])
def test_mxfp4_e8m0_codes_at_both_ends(g, options):
    run_fp4(g, 384, 320, 512, "mxfp4", seed=950, a_pool=np.arange(0, 4), b_pool=np.arange(251, 255),
            options=options)
