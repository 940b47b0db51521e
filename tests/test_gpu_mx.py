"""GPU parity of the block-scaled fp8 GEMM (gemm_mxfp8) against the oracle.

Integer-valued E4M3/E5M2 operands with power-of-two scales make every product
and every partial sum exact in fp32, so those cases are bit-exact; normal
inputs are held to the parity tolerance (1e-3 * the scaled sum of |products|
(+ |beta c|) + 1 ulp of the output type). Scales are seeded E8M0 codes in
[124, 130] unless a case says otherwise, arranged in the ABI's 512-byte atoms.
"""
import numpy as np
import pytest

import seeded_inputs as si
from oracle import gemm as og
from test_gpu_parity import sample_entries

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
FP8 = {"e4m3": 0, "e5m2": 1}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
OUT = {"f32": 0, "bf16": 1, "f16": 2}


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


def _ru(x, m):
    return max(m, (x + m - 1) // m * m)


def _dev_bytes(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1).copy()).to(DEV)


def _out_bits(t, fmt):
    a = t.cpu()
    if fmt == "f32":
        return a.view(torch.int32).numpy().view(np.uint32)
    return a.view(torch.int16).numpy().view(np.uint16)


def run_mx(g, M, N, K, *, a_fmt="e4m3", b_fmt=None, a_major="K", b_major="K", out="f32", alpha=1.0, beta=0.0,
           dist="int4", seed=0, exact=False, options=None, sample=None, lo=124, hi=130, b_lo=None, b_hi=None):
    """One MXFP8 GEMM through the C ABI against the oracle. A's E8M0 codes are drawn
    from [lo, hi], B's from [b_lo, b_hi] (default: the same range)."""
    b_fmt = b_fmt or a_fmt
    lda = _ru(K if a_major == "K" else M, 16)
    ldb = _ru(K if b_major == "K" else N, 16)
    ldd = _ru(N, 4 if out == "f32" else 8)
    A = si.matrix_bits(seed, M, K, dist, a_fmt, transpose=(a_major == "MN"), ld=lda)
    B = si.matrix_bits(seed + 1, K, N, dist, b_fmt, transpose=(b_major == "K"), ld=ldb)
    C = si.matrix_bits(seed + 2, M, N, dist, out, ld=ldd) if beta != 0.0 else None
    nb = max(1, (K + 31) // 32)
    sa = si.scale_codes(seed + 3, M, nb, lo, hi)
    sb = si.scale_codes(seed + 4, N, nb, lo if b_lo is None else b_lo, hi if b_hi is None else b_hi)
    SA = torch.from_numpy(si.mx_scale_atoms(sa, M, K)).to(DEV) if K > 0 else None
    SB = torch.from_numpy(si.mx_scale_atoms(sb, N, K)).to(DEV) if K > 0 else None
    if K > 0:
        assert SA.numel() == g.gemm_mx_scale_bytes(M, K) and SB.numel() == g.gemm_mx_scale_bytes(N, K)
    At, Bt = _dev_bytes(A), _dev_bytes(B)
    Ct = si.torch_from_bits(C, out).to(DEV) if C is not None else None
    Dt = torch.full((M, ldd), float("nan"), dtype=TDT[out], device=DEV)
    g.gemm_mxfp8(M, N, K, At, FP8[a_fmt], 0 if a_major == "K" else 1, lda, SA, Bt, FP8[b_fmt],
                 0 if b_major == "K" else 1, ldb, SB, Ct, ldd if C is not None else 0, Dt, ldd, OUT[out],
                 alpha, beta, options=options)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, f"device status word {word:#x}"
    got_bits = _out_bits(Dt, out)[:, :N]
    got = si.bits_to_float64(got_bits, out)
    kw = dict(in_fmt=a_fmt, b_fmt=b_fmt, a_major=a_major, b_major=b_major, lda=lda, ldb=ldb, C=C, c_fmt=out,
              ldc=ldd, alpha=alpha, beta=beta)
    if sample is None:
        ref, S = og.gemm_mx(M, N, K, A, B, sa, sb, **kw)
        gsel, bsel = got, got_bits
    else:
        rows, cols = sample
        ref, S = og.gemm_mx_entries(M, N, K, A, B, sa, sb, rows, cols, **kw)
        gsel, bsel = got[rows, cols], got_bits[rows, cols]
    if exact:
        assert np.array_equal(bsel, og.round_bits(ref, out)), "integer case must be bit-exact"
        return
    err = np.abs(gsel - ref)
    bad = err > og.tolerance(S, ref, out)
    assert not bad.any(), f"{int(bad.sum())} entries outside tolerance, first {np.argwhere(bad)[0]}"
    assert np.isfinite(gsel).all()


def test_mx_single_tile_exact(g):
    run_mx(g, 128, 128, 128, exact=True, seed=1)


@pytest.mark.parametrize("M,N,K", [(300, 200, 600), (128, 256, 1024), (77, 390, 256), (520, 136, 100),
                                   (1000, 1000, 1000)])
def test_mx_ragged_shapes_exact(g, M, N, K):
    run_mx(g, M, N, K, exact=True, seed=M + N + K)


@pytest.mark.parametrize("a_major,b_major", [("K", "MN"), ("MN", "K"), ("MN", "MN")])
def test_mx_operand_majors_exact(g, a_major, b_major):
    run_mx(g, 384, 256, 512, a_major=a_major, b_major=b_major, exact=True, seed=7)


@pytest.mark.parametrize("fa,fb", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_mx_formats_exact(g, fa, fb):
    run_mx(g, 256, 384, 640, a_fmt=fa, b_fmt=fb, exact=True, seed=11)


def test_mx_wide_scale_range_within_tolerance(g):
    # scales from 2^-27 to 2^27: fp32 accumulation is no longer exact across
    # blocks, so the tolerance bound applies
    run_mx(g, 256, 256, 512, dist="normal", seed=13, lo=100, hi=154)


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_mx_normal_inputs_alpha_beta_within_tolerance(g, out):
    run_mx(g, 640, 520, 768, dist="normal", out=out, alpha=0.5, beta=-1.25, seed=17)


@pytest.mark.parametrize("M,N,K", [(300, 200, 600), (256, 128, 384), (520, 136, 100)])
def test_mx_block_k_128_exact(g, M, N, K):
    # the 128-element K stage variant (five stages) next to the default 256
    run_mx(g, M, N, K, exact=True, seed=M + K + 1, options=dict(block_k=128))


@pytest.mark.parametrize("M,N,K", [(256, 128, 256), (300, 200, 600), (700, 390, 1000), (2048, 2048, 512)])
def test_mx_cta_pairs_exact(g, M, N, K):
    # 256 x 128 pair tiles: each CTA's TMEM holds its own A rows' scales and a
    # copy of the tile's B scales (ragged M leaves the odd CTA past the last atom row)
    run_mx(g, M, N, K, exact=True, seed=3 * M + K, options=dict(cta_group=2))


@pytest.mark.parametrize("a_major,b_major", [("MN", "MN"), ("K", "MN")])
def test_mx_cta_pairs_majors_and_e5m2(g, a_major, b_major):
    run_mx(g, 512, 384, 768, a_major=a_major, b_major=b_major, a_fmt="e5m2", b_fmt="e4m3", exact=True, seed=29,
           options=dict(cta_group=2))


def test_mx_cta_pairs_stream_k_and_tolerance(g):
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_mx(g, 700, 300, 1500, exact=True, seed=31, options=dict(cta_group=2, workspace=ws, stream_k=2, max_ctas=6))
    run_mx(g, 1024, 640, 1024, dist="normal", out="bf16", alpha=1.5, beta=0.5, seed=37, options=dict(cta_group=2))


@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (700, 600, 1000), (2048, 2048, 768), (256, 200, 96)])
def test_mx_wide_pairs_exact(g, M, N, K):
    # 256 x 256 pair tiles with a single accumulator buffer; each CTA's TMEM
    # holds the scales of its A rows and both B atoms of the tile
    run_mx(g, M, N, K, exact=True, seed=5 * M + K, options=dict(cta_group=2, tile_n=256))


def test_mx_wide_pairs_majors_formats_and_tolerance(g):
    run_mx(g, 512, 768, 640, a_major="MN", b_major="MN", a_fmt="e5m2", b_fmt="e4m3", exact=True, seed=41,
           options=dict(cta_group=2, tile_n=256))
    run_mx(g, 1024, 768, 1024, dist="normal", out="bf16", alpha=0.5, beta=1.5, seed=43,
           options=dict(cta_group=2, tile_n=256))


@pytest.mark.parametrize("out", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(512, 520, 512), (700, 600, 1000), (2048, 2048, 256)])
def test_mx_wide_pairs_16bit_out_without_c(g, out, M, N, K):
    # one-accumulator pair tiles, 16-bit output, no C: the epilogue reads the whole
    # accumulator row before its stores (ragged N chunks, rows past M, several
    # tiles per cluster with the grid capped at four clusters)
    run_mx(g, M, N, K, out=out, alpha=0.75, exact=True, seed=11 * M + K,
           options=dict(cta_group=2, tile_n=256, max_ctas=8))


def test_mx_wide_pairs_ignore_stream_k(g):
    # no spare accumulator buffer: the split is not applied, the result is unchanged
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_mx(g, 700, 600, 1500, exact=True, seed=47, options=dict(cta_group=2, tile_n=256, workspace=ws, stream_k=2,
                                                                  max_ctas=6))


def test_mx_stream_k_exact(g):
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_mx(g, 700, 300, 1500, exact=True, seed=19, options=dict(workspace=ws, stream_k=2, max_ctas=5))


def test_mx_large_sampled(g):
    M = N = K = 4096
    rng = np.random.default_rng(5)
    rows = np.concatenate([rng.integers(0, M, 2048), [0, 127, 128, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 2048), [0, 127, 128, N - 1]])
    run_mx(g, M, N, K, dist="normal", out="bf16", seed=23, sample=(rows, cols))


def test_mx_full_size_bench_launch(g):
    # 8192^3 in the launch bench.py times (default options: 256 x 256 CTA pairs with
    # one accumulator, copier warp, early accumulator release) on its input recipe
    M = N = K = 8192
    rows, cols = sample_entries(M, N, n=1024, seed=50)
    run_mx(g, M, N, K, dist="uniform", out="bf16", seed=50, sample=(rows, cols))


def test_mx_injected_wait_times_out_and_the_context_survives(g):
    # the MXFP8 pair kernel with its scale copier warp: an injected wait runs out,
    # every role ends within its bound, and the next call computes correctly
    M = N = K = 512
    A = torch.zeros(M * K, dtype=torch.uint8, device=DEV)
    B = torch.zeros(N * K, dtype=torch.uint8, device=DEV)
    SA = torch.full((g.gemm_mx_scale_bytes(M, K),), 127, dtype=torch.uint8, device=DEV)
    SB = torch.full((g.gemm_mx_scale_bytes(N, K),), 127, dtype=torch.uint8, device=DEV)
    D = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    g.gemm_debug_inject_timeout(20)
    g.gemm_mxfp8(M, N, K, A, 0, 0, K, SA, B, 0, 0, K, SB, None, 0, D, N, 1, 1.0, 0.0,
                 options=dict(cta_group=2, tile_n=256))
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and word != 0
    run_mx(g, 512, 264, 512, exact=True, seed=73, options=dict(cta_group=2, tile_n=256))
    # the producer stuck instead: the copier warp ends on the abort flag and its
    # tcgen05.cp drain barrier is awaited before TMEM is freed
    g.gemm_debug_inject_timeout(20, role=1)
    g.gemm_mxfp8(M, N, K, A, 0, 0, K, SA, B, 0, 0, K, SB, None, 0, D, N, 1, 1.0, 0.0,
                 options=dict(cta_group=2, tile_n=256))
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and (word & 0xFF, (word >> 8) & 0xFF) == (1, 6), hex(word)
    run_mx(g, 512, 264, 512, exact=True, seed=74, options=dict(cta_group=2, tile_n=256))


def test_mx_argument_errors(g):
    M, N, K = 128, 128, 128
    A = torch.zeros(M * K, dtype=torch.uint8, device=DEV)
    B = torch.zeros(N * K, dtype=torch.uint8, device=DEV)
    S = torch.zeros(g.gemm_mx_scale_bytes(128, K) + 16, dtype=torch.uint8, device=DEV)
    D = torch.empty(M, N, dtype=torch.float32, device=DEV)

    def call(sa, sb, **opts):
        g.gemm_mxfp8(M, N, K, A, 0, 0, K, sa, B, 0, 0, K, sb, None, 0, D, N, 0, 1.0, 0.0, options=opts or None)

    with pytest.raises(g.GemmError) as ei:
        call(None, S)
    assert ei.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as ei:
        call(S[8:], S)
    assert ei.value.status == g.ERR_ALIGNMENT
    with pytest.raises(g.GemmError) as ei:
        call(S, S, tile_n=256)
    assert ei.value.status == g.ERR_UNSUPPORTED
    with pytest.raises(g.GemmError) as ei:
        call(S, S, cta_group=2, block_k=128)
    assert ei.value.status == g.ERR_UNSUPPORTED
    assert g.gemm_mx_scale_bytes(300, 260) == 3 * 3 * 512 and g.gemm_mx_scale_bytes(0, 5) == 0
