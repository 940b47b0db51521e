"""GPU parity of the B-multicast clusters (options.multicast_b) against the oracle.

Two single-CTA (cta_group::1) 128 x 256 tiles that share a B panel run as a
cluster: each CTA loads half of every B stage and multicasts it into both
CTAs' shared memory, and each CTA's MMA completion releases the stage in
both. Integer-valued cases compare bit for bit; normal inputs are held to the
parity tolerance. Ragged shapes put the second CTA of a cluster past M (it
still loads its half of B for the first) and cut N inside a B half. The
256-row tiles that share B the same way are covered in test_gpu_two_half.py.
"""
import pytest

from test_gpu_parity import run_case, sample_entries

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MC = dict(cta_group=1, tile_n=256, tile_m=128, multicast_b=1)


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


def test_mcast_single_cluster_tile_exact(g):
    run_case(g, 256, 256, 256, dist="int4", exact=True, options=MC)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (100, 300, 200), (384, 520, 1000), (640, 384, 512),
                                   (257, 200, 136), (1000, 1000, 1000)])
def test_mcast_ragged_shapes_exact(g, M, N, K):
    run_case(g, M, N, K, dist="int4", exact=True, seed=M + N + K, options=MC)


@pytest.mark.parametrize("a_major,b_major", [("K", "MN"), ("MN", "K"), ("MN", "MN")])
def test_mcast_operand_majors_exact(g, a_major, b_major):
    run_case(g, 512, 512, 384, a_major=a_major, b_major=b_major, dist="int4", exact=True, options=MC)


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_mcast_outputs_alpha_beta_within_tolerance(g, out):
    run_case(g, 640, 600, 768, dist="normal", out=out, alpha=0.5, beta=-1.25, seed=13, options=MC)


def test_mcast_fp8_exact(g):
    run_case(g, 520, 600, 512, in_fmt="e4m3", b_fmt="e5m2", a_major="K", b_major="MN", dist="int4", exact=True,
             options=MC)


def test_mcast_with_stream_k(g):
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device="cuda:0")
    run_case(g, 1536, 1280, 1024, dist="int4", exact=True, options=dict(MC, workspace=ws, stream_k=2, max_ctas=10))
    run_case(g, 2048, 2048, 1024, dist="normal", out="bf16", seed=5, options=dict(MC, workspace=ws))


def test_mcast_square_4096_sampled(g):
    M = N = K = 4096
    run_case(g, M, N, K, dist="normal", scale=0.1, out="bf16", seed=10, options=MC,
             sample=sample_entries(M, N, 2048, seed=4))
