"""GPU parity of the stream-K schedule (options.stream_k with a workspace).

A split tile is summed by several clusters: its head adds the others' fp32
partial sums to its own accumulator, so only the order of the additions
differs from the unsplit schedule. Integer-valued inputs therefore stay
bit-exact against the oracle; random inputs are held to the parity tolerance
(1e-3 * sum_k |a_ik b_kj| (+ |beta c_ij|) + 1 ulp of the output type).

`max_ctas` shrinks the persistent grid so that small problems still get the
cases that matter: tiles cut in two and in many pieces, clusters whose share
lies inside one tile, data-parallel tiles before the split ones, ragged M, N
and K.
"""
import numpy as np
import pytest

from test_gpu_parity import run_case, sample_entries

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


@pytest.fixture(scope="module")
def ws(g):
    n = g.gemm_streamk_workspace_size()
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device=DEV)


def _opts(ws, **kw):
    o = dict(workspace=ws)
    o.update(kw)
    return o


# (M, N, K, cta_group, tile_n, max_ctas, stream_k): tiles T, clusters G
SPLITS = [
    (300, 200, 1000, 1, 128, 4, 1),     # T=6 < 2G: every tile split, two clusters per tile
    (300, 200, 1000, 1, 128, 4, 2),
    (1100, 260, 700, 1, 128, 5, 1),     # T=27, G=5: 20 data-parallel tiles, 7 split
    (1100, 260, 700, 1, 128, 5, 2),     # every tile split over a small grid
    (200, 130, 1000, 1, 128, 7, 2),     # T=4, G=7: tiles cut three ways, middle pieces
    (130, 100, 130, 1, 128, 6, 2),      # two K blocks per tile, six clusters: one block each
    (520, 300, 900, 1, 256, 6, 1),      # 256-wide single-CTA tiles
    (700, 600, 1500, 2, 256, 8, 1),     # pairs: T=9, G=4: 4 data-parallel tiles, 5 split
    (700, 600, 1500, 2, 256, 8, 2),
    (600, 300, 1100, 2, 128, 6, 2),     # pairs with 128-wide tiles
    (1100, 260, 700, 1, 128, 5, 3),     # T=27, G=5: only the 2 tiles of the ragged wave split
    (700, 600, 1500, 2, 256, 8, 3),     # pairs: T=9, G=4: one tile split four ways
]


@pytest.mark.parametrize("M,N,K,cg,bn,ctas,mode", SPLITS)
def test_streamk_integer_inputs_bit_exact(g, ws, M, N, K, cg, bn, ctas, mode):
    run_case(g, M, N, K, dist="int4", exact=True, seed=M + K,
             options=_opts(ws, cta_group=cg, tile_n=bn, max_ctas=ctas, stream_k=mode))


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K,cg,bn,ctas,mode", [SPLITS[2], SPLITS[4], SPLITS[7]])
def test_streamk_random_inputs_within_tolerance(g, ws, out, M, N, K, cg, bn, ctas, mode):
    in_fmt = "f16" if out == "f16" else "bf16"
    run_case(g, M, N, K, in_fmt=in_fmt, out=out, dist="normal", seed=7 * M + N, alpha=0.75, beta=-0.5,
             options=_opts(ws, cta_group=cg, tile_n=bn, max_ctas=ctas, stream_k=mode))


@pytest.mark.parametrize("a_major,b_major", [("MN", "K"), ("K", "MN"), ("MN", "MN")])
def test_streamk_operand_majors(g, ws, a_major, b_major):
    run_case(g, 384, 320, 1000, a_major=a_major, b_major=b_major, dist="int4", exact=True, seed=11,
             options=_opts(ws, cta_group=1, tile_n=128, max_ctas=5, stream_k=2))


def test_streamk_fp8(g, ws):
    run_case(g, 520, 400, 1536, in_fmt="e4m3", dist="int4", exact=True, seed=13,
             options=_opts(ws, cta_group=1, tile_n=128, max_ctas=6, stream_k=2))


def test_streamk_in_place_beta(g, ws):
    # D aliases C: every split tile's head reads C before its own store
    run_case(g, 1100, 260, 700, dist="int4", exact=True, alpha=2.0, beta=1.0, inplace=True, seed=17,
             options=_opts(ws, cta_group=1, tile_n=128, max_ctas=5, stream_k=1))


def test_streamk_workspace_reused_across_calls(g, ws):
    # one workspace for successive launches: each launch tags its flags anew,
    # so a head never takes a partial sum left by an earlier launch
    for i, (M, N, K) in enumerate([(300, 200, 1000), (700, 600, 1500), (300, 200, 1000), (200, 130, 1000)]):
        run_case(g, M, N, K, dist="int4", exact=True, seed=100 + i,
                 options=_opts(ws, cta_group=1 if i != 1 else 2, tile_n=128 if i != 1 else 256,
                               max_ctas=[4, 8, 4, 7][i], stream_k=2))


def test_streamk_same_result_as_unsplit_within_tolerance(g, ws):
    # the split only reorders additions: compare with the data-parallel run directly
    import seeded_inputs as si
    M, N, K = 1024, 768, 2048
    A = si.torch_from_bits(si.matrix_bits(21, M, K, "normal", "bf16"), "bf16").to(DEV)
    B = si.torch_from_bits(si.matrix_bits(22, K, N, "normal", "bf16", transpose=True), "bf16").to(DEV)
    D0 = torch.empty(M, N, dtype=torch.float32, device=DEV)
    D1 = torch.empty_like(D0)
    base = dict(cta_group=1, tile_n=128, max_ctas=10)
    g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D0, N, 0, 1.0, 0.0, options=dict(base, stream_k=-1))
    g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D1, N, 0, 1.0, 0.0,
              options=_opts(ws, stream_k=2, **base))
    st, word = g.gemm_last_device_status()
    assert st == g.OK, hex(word)
    S = (A.float().abs() @ B.float().abs().t()).double()
    assert (D1.double() - D0.double()).abs().le(2e-5 * S + 1e-30).all()


def test_streamk_auto_on_ragged_wave_full_grid(g, ws):
    # 4096^3 with CTA pairs: 256 tiles on the resident clusters leave a ragged
    # last wave, so the default (auto) splits it; sampled entries vs the oracle
    M = N = K = 4096
    rows, cols = sample_entries(M, N, n=1024, seed=3)
    run_case(g, M, N, K, dist="uniform", seed=31, sample=(rows, cols),
             options=_opts(ws, cta_group=2, tile_n=256))


def test_streamk_skinny_full_grid(g, ws):
    # fewer tiles than clusters: every tile split across the whole grid
    M, N, K = 16384, 128, 8192
    rows, cols = sample_entries(M, N, n=1024, seed=4)
    run_case(g, M, N, K, dist="uniform", seed=41, sample=(rows, cols), out="bf16",
             options=_opts(ws, stream_k=2))


def test_streamk_rejects_small_or_misaligned_workspace(g, ws):
    M, N, K = 300, 200, 1000
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(N, K, dtype=torch.bfloat16, device=DEV)
    D = torch.empty(M, N, dtype=torch.float32, device=DEV)
    small = dict(workspace=ws, workspace_bytes=4096, max_ctas=4, tile_n=128, stream_k=2)
    with pytest.raises(g.GemmError) as ei:
        g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0, options=small)
    assert ei.value.status == g.ERR_INVALID_ARG
    odd = dict(workspace=ws[16:], workspace_bytes=ws.numel() - 16, stream_k=2)
    with pytest.raises(g.GemmError) as ei:
        g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0, options=odd)
    assert ei.value.status == g.ERR_ALIGNMENT
    bad = dict(workspace=ws, stream_k=4)
    with pytest.raises(g.GemmError) as ei:
        g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0, options=bad)
    assert ei.value.status == g.ERR_INVALID_ARG
    # without a workspace the option is a no-op: the launch runs unsplit
    g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0, options=dict(stream_k=2))
    assert np.all(D.cpu().numpy() == 0.0)
