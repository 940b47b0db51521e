"""GPU parity of the weight-stationary tiles (tcgen05.mma.ws) against the oracle.

"06 Blackwell Tensor Core - tcgen05 MMA", "How cta_group Sets the Operation
Scope": .ws is one of the four choices that fix the accumulator layout. The
library runs it on single-CTA tiles of 32 rows (M = 32 exists only in the
.ws form) and, when asked, 64 rows; the epilogue reads the accumulator back
through the column-part map the oracle states as ``layouts.tmem_ws``. A wrong
map would put results in the wrong rows or columns, so the integer cases
compare bit for bit; normal inputs are held to the parity tolerance.
"""
import numpy as np
import pytest

from test_gpu_parity import run_case, sample_entries

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

WS32 = dict(tile_m=32)
WS64 = dict(tile_m=64, mma_ws=1)
WS64W = dict(tile_m=64, tile_n=256, mma_ws=1)


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


@pytest.mark.parametrize("opts", [WS32, WS64, WS64W], ids=["m32", "m64", "m64n256"])
def test_ws_single_tile_exact(g, opts):
    M = opts["tile_m"]
    run_case(g, M, opts.get("tile_n", 256 if M == 32 else 128), 128, dist="int4", exact=True, options=opts)


@pytest.mark.parametrize("opts", [WS32, WS64, WS64W], ids=["m32", "m64", "m64n256"])
@pytest.mark.parametrize("M,N,K", [(20, 1000, 520), (32, 512, 256), (64, 384, 192), (100, 300, 200), (7, 264, 72),
                                   (130, 520, 1000)])
def test_ws_ragged_shapes_exact(g, opts, M, N, K):
    # several row tiles, ragged N and K tails
    run_case(g, M, N, K, dist="int4", exact=True, seed=M + N + K, options=opts)


@pytest.mark.parametrize("opts", [WS32, WS64], ids=["m32", "m64"])
@pytest.mark.parametrize("a_major,b_major", [("K", "MN"), ("MN", "K"), ("MN", "MN")])
def test_ws_operand_majors_exact(g, opts, a_major, b_major):
    run_case(g, 96, 512, 256, a_major=a_major, b_major=b_major, dist="int4", exact=True, options=opts)


@pytest.mark.parametrize("opts", [WS32, WS64], ids=["m32", "m64"])
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_ws_outputs_alpha_beta_within_tolerance(g, opts, out):
    run_case(g, 72, 600, 384, dist="normal", out=out, alpha=0.75, beta=-1.5, seed=11, options=opts)


@pytest.mark.parametrize("opts", [WS32, WS64], ids=["m32", "m64"])
def test_ws_in_place_and_fp16(g, opts):
    run_case(g, 40, 520, 136, in_fmt="f16", dist="uniform", out="f32", beta=1.0, inplace=True, options=opts)


@pytest.mark.parametrize("opts", [WS32, WS64], ids=["m32", "m64"])
def test_ws_k_zero_gives_beta_c(g, opts):
    run_case(g, 48, 300, 0, dist="uniform", out="f32", beta=0.5, options=opts)


def test_ws_is_chosen_for_tiny_m_when_asked(g):
    # mma_ws 1 with no tile_m: 32-row tiles for M <= 32
    run_case(g, 16, 2048, 512, dist="int4", exact=True, options=dict(mma_ws=1))


@pytest.mark.parametrize("opts", [WS32, WS64], ids=["m32", "m64"])
def test_ws_decode_shape_sampled(g, opts):
    # a small-M, wide-N, long-K shape (32 x 16384 x 4096) on sampled entries
    M, N, K = 32, 16384, 4096
    run_case(g, M, N, K, dist="normal", out="bf16", seed=21, options=opts, sample=sample_entries(M, N, 2048, seed=3))
