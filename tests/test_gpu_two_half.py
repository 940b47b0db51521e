"""GPU parity of the two-half single-CTA tiles (tile_m 256) against the oracle.

"06 Blackwell Tensor Core - tcgen05 MMA": a cta_group::1 MMA covers at most
128 rows, each issue reading its A rows and one B slice from shared memory
and accumulating into its own Tensor Memory columns. A 256-row tile on one CTA
issues two such MMAs per K slice on the same B slice, rows 128..255 of A
starting 128 rows further into the stage ("LBO, SBO and SWZ for a tcgen05
tile": 8-row groups SBO apart for K-major tiles, MN atoms LBO apart for
MN-major ones), into accumulators at TMEM columns 0 and 256. A wrong half offset or
column base would mix up the two halves, so the integer cases compare bit for
bit; normal inputs are held to the parity tolerance. By default two such CTAs
form a cluster that shares B by TMA multicast (each loads half of the B
panel into both); every case runs with and without that sharing.
"""
import pytest

from test_gpu_parity import DEV, run_case, sample_entries

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SHARING = [dict(tile_m=256), dict(tile_m=256, multicast_b=-1)]
IDS = ["sharedB", "ownB"]


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
def test_two_half_single_tile_exact(g, opts):
    run_case(g, 256, 256, 64, dist="int4", exact=True, options=opts)
    run_case(g, 512, 256, 64, dist="int4", exact=True, options=opts)  # one cluster tile when B is shared


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
@pytest.mark.parametrize("M,N,K", [(1000, 1000, 776), (130, 300, 72), (257, 513, 1000), (768, 256, 2048), (1, 256, 64),
                                   (1300, 520, 200)])
def test_two_half_ragged_shapes_exact(g, opts, M, N, K):
    # several row tiles, a second half (or a cluster's second CTA) partly or wholly
    # past M, ragged N and K tails
    run_case(g, M, N, K, dist="int4", exact=True, seed=M + N + K, options=opts)


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
@pytest.mark.parametrize("a_major,b_major", [("K", "MN"), ("MN", "K"), ("MN", "MN")])
def test_two_half_operand_majors_exact(g, opts, a_major, b_major):
    run_case(g, 700, 520, 200, a_major=a_major, b_major=b_major, dist="int4", exact=True, options=opts)


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
@pytest.mark.parametrize("swz", [1, 2, 3, 4], ids=["sw32", "sw64", "sw128", "none"])
@pytest.mark.parametrize("a_major", ["K", "MN"])
def test_two_half_swizzles_exact(g, opts, swz, a_major):
    run_case(g, 768, 512, 256, a_major=a_major, b_major=a_major, dist="int4", exact=True,
             options=dict(opts, swizzle_a=swz, swizzle_b=swz))


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_two_half_outputs_alpha_beta_within_tolerance(g, opts, out):
    run_case(g, 600, 700, 384, dist="normal", out=out, alpha=0.75, beta=-1.5, seed=11, options=opts)


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
def test_two_half_in_place_fp16_and_k_zero(g, opts):
    run_case(g, 300, 520, 136, in_fmt="f16", dist="uniform", out="f32", beta=1.0, inplace=True, options=opts)
    run_case(g, 300, 300, 0, dist="uniform", out="f32", beta=0.5, options=opts)


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_two_half_stream_k_exact(g, opts, mode):
    # split tiles: the head adds its contributors' 256-row partial sums chunk by chunk
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_case(g, 2048, 2304, 3000, dist="int4", exact=True, out="f32", beta=0.5, seed=mode,
             options=dict(opts, workspace=ws, stream_k=mode))


def test_two_half_is_the_default_for_large_single_cta_problems(g):
    # 4096^3 with cta_group 1 and the stream-K workspace (the bench launch):
    # two-half tiles 224 wide, unsplit; with tile_n 256, 256 wide in B-sharing
    # pairs; sampled entries of the full product
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    M = N = K = 4096
    for opts in (dict(cta_group=1, workspace=ws), dict(cta_group=1, tile_n=256, workspace=ws)):
        run_case(g, M, N, K, dist="normal", scale=0.1, out="bf16", seed=10, options=opts,
                 sample=sample_entries(M, N, 2048, seed=5))


@pytest.mark.parametrize("opts", SHARING, ids=IDS)
@pytest.mark.parametrize("role", [1, 2], ids=["producer", "mma"])
def test_two_half_injected_timeout_and_the_context_survives(g, opts, role):
    g.gemm_debug_inject_timeout(20, role=role)
    M = N = K = 512
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(N, K, dtype=torch.bfloat16, device=DEV)
    D = torch.zeros(M, N, dtype=torch.float32, device=DEV)
    g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0, options=opts)
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and word != 0, hex(word)
    run_case(g, 512, 384, 256, dist="int4", exact=True, options=opts)


# 224-wide two-half tiles: the second accumulator still starts at TMEM column 256,
# and with 16-bit output the last 32 columns of a tile row form a half chunk that
# the epilogue writes from registers, cut at the tile's edge
W224 = [dict(tile_m=256, tile_n=224), dict(tile_m=256, tile_n=224, multicast_b=1)]
IDS224 = ["ownB", "sharedB"]


@pytest.mark.parametrize("opts", W224, ids=IDS224)
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(256, 224, 64), (1000, 1000, 776), (1300, 500, 200), (600, 230, 300)])
def test_224_wide_tiles_exact(g, opts, out, M, N, K):
    in_fmt = "f16" if out == "f16" else "bf16"
    run_case(g, M, N, K, in_fmt=in_fmt, out=out, alpha=2.0, beta=-1.0, dist="int4", exact=True, seed=M + N,
             options=opts)


@pytest.mark.parametrize("a_major,b_major", [("MN", "K"), ("K", "MN"), ("MN", "MN")])
def test_224_wide_operand_majors_exact(g, a_major, b_major):
    run_case(g, 700, 900, 200, a_major=a_major, b_major=b_major, out="bf16", dist="int4", exact=True,
             options=dict(tile_m=256, tile_n=224))


def test_224_wide_in_place_k_zero_and_normal_inputs(g):
    o = dict(tile_m=256, tile_n=224)
    run_case(g, 300, 520, 136, out="bf16", beta=1.0, dist="int4", exact=True, inplace=True, options=o)
    run_case(g, 300, 440, 0, out="bf16", beta=0.5, dist="uniform", options=o)
    run_case(g, 1000, 600, 1000, out="bf16", beta=1.0, dist="normal", options=o)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_224_wide_stream_k_exact(g, mode):
    # contributors write 224-column slots; the head's partial sums stop at the slot's edge
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_case(g, 2048, 2240, 3000, dist="int4", exact=True, out="bf16", beta=0.5, seed=mode,
             options=dict(tile_m=256, tile_n=224, workspace=ws, stream_k=mode))
