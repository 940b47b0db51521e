"""GPU parity of split loads (``flags`` bit 5): two producer warps, one issuing
the A boxes and A scale atoms, the other the B boxes and B scale atoms, each
arming the stage's full barrier with the bytes it loads ("Tensor Cores,
layouts, and swizzling", TMA section: a stage is complete once every byte it
expects has landed, whoever issued the copies). Every kernel kind that has the
second producer warp is compared with the oracle, bit for bit on integer data;
NVFP4 kernels have no second warp and run their usual path under the bit.
"""
import pytest

from test_gpu_parity import DEV, _grouped, run_case
from test_gpu_fp4 import run_fp4
from test_gpu_mx import run_mx

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SPLIT = 32


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


@pytest.mark.parametrize("opts", [dict(cta_group=1, tile_n=256), dict(cta_group=2, tile_n=256), dict(cta_group=1, tile_n=128),
                                  dict(cta_group=2, tile_n=128), dict(cta_group=1, tile_n=256, multicast_b=1),
                                  dict(tile_m=32), dict(tile_m=64, mma_ws=1), dict(tile_m=64),
                                  dict(cta_group=2, tile_n=256, block_k=128)],
                         ids=["cg1n256", "cg2n256", "cg1n128", "cg2n128", "mcastB", "ws32", "ws64", "m64", "cg2bk128"])
@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("MN", "MN"), ("K", "MN")])
def test_split_load_16bit_exact(g, opts, a_major, b_major):
    run_case(g, 700, 1000, 776, dist="int4", exact=True, a_major=a_major, b_major=b_major,
             options=dict(opts, flags=SPLIT))


def test_split_load_normal_inputs_alpha_beta(g):
    run_case(g, 1000, 520, 1000, dist="normal", out="bf16", alpha=0.5, beta=-1.0, options=dict(cta_group=2, flags=SPLIT))


def test_split_load_with_stream_k(g):
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_case(g, 2048, 2048, 2048, dist="int4", exact=True, options=dict(cta_group=1, tile_n=256, flags=SPLIT, workspace=ws))


@pytest.mark.parametrize("fmt", ["e4m3", "tf32"])
@pytest.mark.parametrize("cg", [1, 2])
def test_split_load_fp8_and_tf32(g, fmt, cg):
    run_case(g, 600, 800, 1024, in_fmt=fmt, dist="int4", exact=True, options=dict(cta_group=cg, flags=SPLIT))


def test_split_load_mxfp8(g):
    run_mx(g, 700, 900, 1024, exact=True, options=dict(flags=SPLIT))
    run_mx(g, 700, 900, 1024, exact=True, options=dict(cta_group=2, tile_n=256, flags=SPLIT))


@pytest.mark.parametrize("kind", ["mxfp4", "nvfp4"])
def test_split_load_fp4(g, kind):
    run_fp4(g, 600, 700, 1024, kind, options=dict(flags=SPLIT))
    run_fp4(g, 600, 700, 1024, kind, options=dict(cta_group=2, tile_n=256, flags=SPLIT))


@pytest.mark.parametrize("cg", [1, 2])
def test_split_load_grouped(g, cg):
    _grouped(g, [128, 384, 0, 700, 256], 1000, 520, options=dict(cta_group=cg, flags=SPLIT))


@pytest.mark.parametrize("cta_group", [1, 2])
def test_split_load_injected_producer_timeout(g, cta_group):
    # the A producer waits on a barrier nothing arrives at and the B producer
    # stays idle: the status names the producer, and the next calls are exact
    g.gemm_debug_inject_timeout(20, role=1)
    M = N = K = 512
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(N, K, dtype=torch.bfloat16, device=DEV)
    D = torch.zeros(M, N, dtype=torch.float32, device=DEV)
    g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0, options=dict(cta_group=cta_group, flags=SPLIT))
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and (word & 0xFF, (word >> 8) & 0xFF) == (1, 6), hex(word)
    run_case(g, 512, 384, 256, dist="int4", exact=True, options=dict(cta_group=cta_group, flags=SPLIT))
