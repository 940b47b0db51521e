"""GPU parity of the epilogue's direct C path (flags bit 4): C read from global
memory into registers instead of staged in shared memory by TMA.

Integer-valued inputs make every result exact, so the cases compare bit for
bit against the oracle. They cover the chunk at the N edge (partial 16-byte
units, 4- and 2-byte outputs), rows past M, padded leading dimensions, D
aliasing C, and single CTAs and pairs.
"""
import pytest

from test_gpu_parity import run_case

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DIRECT_C = 16


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
