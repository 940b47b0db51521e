"""GPU parity of the epilogue's direct paths: C read from global memory into
registers instead of staged in shared memory by TMA (flags bit 4), and D
written from registers instead of staged and stored by TMA (flags bit 6,
which reads C into registers too).

Integer-valued inputs make every result exact, so the cases compare bit for
bit against the oracle. They cover the chunk at the N edge (partial 16-byte
units, 4- and 2-byte outputs), rows past M, padded leading dimensions, D
aliasing C, K = 0, stream-K heads, single CTAs, two-half tiles and pairs.
"""
import pytest

from test_gpu_parity import run_case

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DIRECT_C = 16
DIRECT_D = 64


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K,cg", [(300, 200, 192, 1), (256, 264, 128, 1), (130, 41, 64, 1),
                                      (700, 600, 320, 2), (2048, 2056, 64, 2)])
def test_direct_c_exact(g, out, M, N, K, cg):
    in_fmt = "f16" if out == "f16" else "bf16"
    run_case(g, M, N, K, in_fmt=in_fmt, out=out, alpha=2.0, beta=-1.0, dist="int4", exact=True, seed=M + N,
             options=dict(cta_group=cg, flags=DIRECT_C))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_direct_c_padded_and_in_place(g, out):
    run_case(g, 320, 136, 128, out=out, beta=1.5, dist="int4", exact=True, seed=3, pad=24,
             options=dict(flags=DIRECT_C))
    run_case(g, 384, 264, 256, out=out, alpha=1.0, beta=1.0, dist="int4", exact=True, seed=4, inplace=True,
             options=dict(cta_group=1, tile_n=256, flags=DIRECT_C))


def test_direct_c_normal_inputs_within_tolerance(g):
    run_case(g, 1024, 1000, 512, a_major="K", b_major="MN", out="f32", alpha=0.75, beta=0.5, dist="normal",
             seed=5, options=dict(cta_group=2, tile_n=256, flags=DIRECT_C))


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("opts", [dict(cta_group=1, tile_n=128), dict(cta_group=1, tile_n=256, tile_m=128),
                                  dict(tile_m=256), dict(cta_group=2, tile_n=256)],
                         ids=["cg1n128", "cg1n256", "twohalf", "pairs"])
def test_direct_d_exact(g, out, opts):
    in_fmt = "f16" if out == "f16" else "bf16"
    run_case(g, 700, 517, 200, in_fmt=in_fmt, out=out, alpha=2.0, beta=-1.0, dist="int4", exact=True, seed=7,
             options=dict(opts, flags=DIRECT_D))
    run_case(g, 513, 1000, 776, in_fmt=in_fmt, out=out, dist="int4", exact=True, seed=8,
             options=dict(opts, flags=DIRECT_D))


def test_direct_d_in_place_padded_and_k_zero(g):
    run_case(g, 300, 520, 136, out="f32", beta=1.0, dist="int4", exact=True, inplace=True, pad=24,
             options=dict(tile_m=256, flags=DIRECT_D))
    run_case(g, 300, 300, 0, out="bf16", beta=0.5, dist="uniform", options=dict(flags=DIRECT_D))


@pytest.mark.parametrize("tile_m", [128, 256])
def test_direct_d_stream_k_heads(g, tile_m):
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device="cuda:0")
    run_case(g, 2048, 2304, 3000, dist="int4", exact=True, out="bf16",
             options=dict(cta_group=1, tile_m=tile_m, workspace=ws, stream_k=1, flags=DIRECT_D))
