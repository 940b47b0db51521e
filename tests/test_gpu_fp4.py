"""GPU parity of the block-scaled fp4 GEMM (gemm_fp4: NVFP4 and MXFP4) against the oracle.

E2M1 values are multiples of 1/2 up to 6 and the scales used here are powers
of two (MXFP4) or powers of two times 1 or 1.5 (NVFP4), so every product and
partial sum of these sizes is exact in fp32: the cases compare bit for bit.
Operands use all sixteen E2M1 codes; scales are arranged in the ABI's
512-byte atoms (16-element blocks for NVFP4, 32 for MXFP4).
"""
import numpy as np
import pytest

import seeded_inputs as si
from oracle import gemm as og
from test_gpu_parity import sample_entries

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KINDS = {"nvfp4": (0, 16, "ue4m3"), "mxfp4": (1, 32, "e8m0")}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
OUT = {"f32": 0, "bf16": 1, "f16": 2}
UE4M3_POOL = np.array([(e << 3) | m for e in (5, 6, 7, 8, 9) for m in (0, 4)], np.uint8)  # 1/4 .. 6


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


def _out_bits(t, fmt):
    a = t.cpu()
    if fmt == "f32":
        return a.view(torch.int32).numpy().view(np.uint32)
    return a.view(torch.int16).numpy().view(np.uint16)


def run_fp4(g, M, N, K, kind, *, out="f32", alpha=1.0, beta=0.0, seed=0, options=None, pad=0, a_pool=None,
            b_pool=None):
    """One fp4 GEMM through the C ABI, bit for bit against the oracle. ``a_pool`` /
    ``b_pool`` (scale codes to draw from) replace the default scale distribution."""
    code, block, scale = KINDS[kind]
    lda = ldb = _ru(K, 32) + pad
    ca = np.zeros((M, lda), np.uint8)
    cb = np.zeros((N, ldb), np.uint8)
    ca[:, :K] = si.fp4_codes(seed, M, K)
    cb[:, :K] = si.fp4_codes(seed + 1, N, K)
    A, B = si.pack_fp4(ca), si.pack_fp4(cb)
    nb = (K + block - 1) // block
    if a_pool is not None or b_pool is not None:
        rng = np.random.default_rng(seed + 2)
        default = UE4M3_POOL if scale == "ue4m3" else np.arange(124, 131, dtype=np.uint8)
        sa = rng.choice(np.asarray(a_pool if a_pool is not None else default, np.uint8), (M, nb))
        sb = rng.choice(np.asarray(b_pool if b_pool is not None else default, np.uint8), (N, nb))
    elif scale == "ue4m3":
        rng = np.random.default_rng(seed + 2)
        sa, sb = rng.choice(UE4M3_POOL, (M, nb)), rng.choice(UE4M3_POOL, (N, nb))
    else:
        sa, sb = si.scale_codes(seed + 2, M, nb), si.scale_codes(seed + 3, N, nb)
    fill = 0x38 if scale == "ue4m3" else 127  # 1.0: padding scales multiply zeros and must be finite
    SA = torch.from_numpy(si.mx_scale_atoms(sa, M, K, block, fill)).to(DEV)
    SB = torch.from_numpy(si.mx_scale_atoms(sb, N, K, block, fill)).to(DEV)
    assert SA.numel() == g.gemm_fp4_scale_bytes(M, K, code) and SB.numel() == g.gemm_fp4_scale_bytes(N, K, code)
    ldd = _ru(N, 4 if out == "f32" else 8)
    C = si.matrix_bits(seed + 4, M, N, "int4", out, ld=ldd) if beta != 0.0 else None
    Ct = si.torch_from_bits(C, out).to(DEV) if C is not None else None
    At = torch.from_numpy(A.reshape(-1).copy()).to(DEV)
    Bt = torch.from_numpy(B.reshape(-1).copy()).to(DEV)
    Dt = torch.full((M, ldd), float("nan"), dtype=TDT[out], device=DEV)
    g.gemm_fp4(M, N, K, At, lda, SA, Bt, ldb, SB, code, Ct, ldd if C is not None else 0, Dt, ldd, OUT[out],
               alpha, beta, options=options)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, f"device status word {word:#x}"
    ref, _ = og.gemm_fp4(M, N, K, A, B, sa, sb, block=block, scale=scale, lda=lda, ldb=ldb, C=C, c_fmt=out,
                         ldc=ldd, alpha=alpha, beta=beta)
    got = _out_bits(Dt, out)[:, :N]
    assert np.array_equal(got, og.round_bits(ref, out)), "fp4 case must be bit-exact"


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
def test_fp4_single_tile(g, kind):
    run_fp4(g, 128, 128, 256, kind, seed=1)


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", [(300, 200, 600), (128, 384, 1024), (77, 140, 100), (520, 136, 64),
                                   (640, 512, 2048)])
def test_fp4_ragged_shapes(g, kind, M, N, K):
    run_fp4(g, M, N, K, kind, seed=M + N + K)


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_fp4_outputs_alpha_beta(g, kind, out):
    run_fp4(g, 384, 264, 512, kind, out=out, alpha=0.5, beta=-2.0, seed=9)


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
def test_fp4_padded_leading_dimensions(g, kind):
    run_fp4(g, 256, 200, 320, kind, seed=13, pad=64)


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
def test_fp4_stream_k(g, kind):
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_fp4(g, 700, 300, 1536, kind, seed=17, options=dict(workspace=ws, stream_k=2, max_ctas=5))


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (700, 600, 1000), (2048, 2048, 512), (300, 130, 96)])
def test_fp4_cta_pairs(g, kind, M, N, K):
    # 256 x 256 pair tiles (one accumulator buffer): each CTA holds its A rows' scales
    # and both B atoms of the tile
    run_fp4(g, M, N, K, kind, seed=2 * M + K, options=dict(cta_group=2))


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("out", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(512, 520, 512), (700, 600, 1000), (2048, 2048, 256)])
def test_fp4_pairs_16bit_out_without_c(g, kind, out, M, N, K):
    # one-accumulator pair tiles with 16-bit output and no C read the whole
    # accumulator row before storing: ragged N chunks, rows past M, and several
    # tiles per cluster (grid capped at four clusters)
    run_fp4(g, M, N, K, kind, out=out, alpha=0.75, seed=M + 7 * K, options=dict(cta_group=2, max_ctas=8))


@pytest.mark.parametrize("M,N,K", [(512, 512, 1024), (700, 600, 1000)])
def test_mxfp4_pairs_128_byte_stages(g, M, N, K):
    # MXFP4 pairs default to 256 bytes of K per stage; 128-byte stages stay available
    run_fp4(g, M, N, K, "mxfp4", seed=3 * M + K, options=dict(cta_group=2, block_k=128))


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
def test_fp4_cta_pairs_alpha_beta(g, kind):
    run_fp4(g, 512, 768, 640, kind, out="bf16", alpha=1.5, beta=-0.5, seed=19, options=dict(cta_group=2))


def test_fp4_argument_errors(g):
    M, N, K = 128, 128, 256
    A = torch.zeros(M * K // 2, dtype=torch.uint8, device=DEV)
    S = torch.zeros(g.gemm_fp4_scale_bytes(128, K, 0) + 16, dtype=torch.uint8, device=DEV)
    D = torch.empty(M, N, dtype=torch.float32, device=DEV)

    def call(k=K, lda=K, kind=0, **opts):
        g.gemm_fp4(M, N, k, A, lda, S, A, lda, S, kind, None, 0, D, N, 0, 1.0, 0.0, options=opts or None)

    for kw, status in [(dict(k=255), g.ERR_INVALID_ARG), (dict(kind=2), g.ERR_INVALID_ARG),
                       (dict(lda=272), g.ERR_ALIGNMENT), (dict(cta_group=2, tile_n=128), g.ERR_UNSUPPORTED),
                       (dict(block_k=64), g.ERR_UNSUPPORTED)]:
        with pytest.raises(g.GemmError) as ei:
            call(**kw)
        assert ei.value.status == status, kw
    assert g.gemm_fp4_scale_bytes(300, 600, 0) == 3 * 10 * 512 and g.gemm_fp4_scale_bytes(300, 600, 1) == 3 * 5 * 512


@pytest.fixture(scope="module")
def fp4_full_operands():
    # 8192 x 8192 packed E2M1 operands, all sixteen codes, shared by both kinds
    M = N = K = 8192
    return M, N, K, si.pack_fp4(si.fp4_codes(60, M, K)), si.pack_fp4(si.fp4_codes(61, N, K))


@pytest.mark.parametrize("kind", ["nvfp4", "mxfp4"])
def test_fp4_full_size_bench_launch(g, fp4_full_operands, kind):
    # 8192^3 in the launch bench.py times (default options: 256 x 256 CTA pairs, one
    # accumulator, copier warps, early accumulator release) on its input recipe;
    # sampled entries against the oracle within the fp32-accumulation tolerance
    M, N, K, A, B = fp4_full_operands
    code, block, scale = KINDS[kind]
    nb = K // block
    if scale == "ue4m3":
        z = si.scale_codes(62, M + N, nb, 0, len(UE4M3_POOL) - 1)
        sa, sb = UE4M3_POOL[z[:M]], UE4M3_POOL[z[M:]]
    else:
        sa, sb = si.scale_codes(62, M, nb), si.scale_codes(63, N, nb)
    fill = 0x38 if scale == "ue4m3" else 127
    SA = torch.from_numpy(si.mx_scale_atoms(sa, M, K, block, fill)).to(DEV)
    SB = torch.from_numpy(si.mx_scale_atoms(sb, N, K, block, fill)).to(DEV)
    At = torch.from_numpy(A.reshape(-1).copy()).to(DEV)
    Bt = torch.from_numpy(B.reshape(-1).copy()).to(DEV)
    Dt = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    g.gemm_fp4(M, N, K, At, K, SA, Bt, K, SB, code, None, 0, Dt, N, OUT["bf16"], 1.0, 0.0)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, f"device status word {word:#x}"
    rows, cols = sample_entries(M, N, n=1024, seed=60 + code)
    ref, S = og.gemm_fp4_entries(M, N, K, A, B, sa, sb, rows, cols, block=block, scale=scale)
    got = si.bits_to_float64(_out_bits(Dt, "bf16")[rows, cols], "bf16")
    err = np.abs(got - ref)
    bad = err > og.tolerance(S, ref, "bf16")
    assert not bad.any(), f"{int(bad.sum())} of {rows.size} sampled entries outside tolerance"


@pytest.mark.parametrize("kind,options", [("nvfp4", dict(cta_group=2, tile_n=256)), ("nvfp4", dict(cta_group=1)),
                                          ("mxfp4", dict(cta_group=2, tile_n=256))])
def test_fp4_injected_wait_times_out_and_the_context_survives(g, kind, options):
    # the block-scaled kernels add scale copier warps: a wait that nothing satisfies
    # must still end every role within its bound, report the status, and leave the
    # context usable
    code, block, scale = KINDS[kind]
    M = N = 512
    K = 512
    fill = 0x38 if scale == "ue4m3" else 127
    A = torch.zeros(M * K // 2, dtype=torch.uint8, device=DEV)
    B = torch.zeros(N * K // 2, dtype=torch.uint8, device=DEV)
    SA = torch.full((g.gemm_fp4_scale_bytes(M, K, code),), fill, dtype=torch.uint8, device=DEV)
    SB = torch.full((g.gemm_fp4_scale_bytes(N, K, code),), fill, dtype=torch.uint8, device=DEV)
    D = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    g.gemm_debug_inject_timeout(20)
    g.gemm_fp4(M, N, K, A, K, SA, B, K, SB, code, None, 0, D, N, OUT["bf16"], 1.0, 0.0, options=options)
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and word != 0
    run_fp4(g, 256, 264, 512, kind, out="bf16", seed=71, options=options)
    # the producer stuck instead (the copier warps then end on the abort flag)
    g.gemm_debug_inject_timeout(20, role=1)
    g.gemm_fp4(M, N, K, A, K, SA, B, K, SB, code, None, 0, D, N, OUT["bf16"], 1.0, 0.0, options=options)
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and (word & 0xFF, (word >> 8) & 0xFF) == (1, 6), hex(word)
    run_fp4(g, 256, 264, 512, kind, out="bf16", seed=72, options=options)
