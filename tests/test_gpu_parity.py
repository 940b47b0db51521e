"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by element.

Tolerance (floating point): |d - ref| <= 1e-3 * (|alpha| sum_k |a_ik b_kj| + |beta c_ij|)
                            + 1 ulp of the output type at ref.
Integer-valued inputs and the descriptor / shared-memory address tables are bit-exact.
"""
import os

import numpy as np
import pytest

import seeded_inputs as si
from oracle import gemm as og
from oracle import layouts as L

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


DEV = "cuda:0"
SWZ_PARAM = {"sw32": 1, "sw64": 2, "sw128": 3, "none": 4, "sw128_base32b": 5}  # gemm_swizzle_t
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _to_dev(bits, fmt):
    return si.torch_from_bits(bits, fmt).to(DEV)


def _out_bits(t, fmt):
    a = t.cpu()
    if fmt == "f32":
        return a.view(torch.int32).numpy().view(np.uint32)
    return a.view(torch.int16).numpy().view(np.uint16)


def _ru(x, m):
    return max(m, (x + m - 1) // m * m)


FP8 = {"e4m3": 0, "e5m2": 1}


def run_case(g, M, N, K, *, in_fmt="bf16", b_fmt=None, a_major="K", b_major="K", out="f32", alpha=1.0,
             beta=0.0, dist="uniform", scale=1.0, seed=0, pad=0, options=None, inplace=False, exact=False,
             sample=None):
    """Run one GEMM through the C ABI and compare with the oracle; returns max |err|."""
    if options and options.get("cta_group") == 2 and os.environ.get("GEMM_TEST_NO_PAIRS"):
        pytest.skip("CTA-pair cases disabled for this run")
    b_fmt = b_fmt or in_fmt
    fp8 = in_fmt in FP8
    # leading dimensions rounded up to the 16-byte TMA stride rule, plus optional padding
    lda = _ru(K if a_major == "K" else M, 16 if fp8 else 8) + pad
    ldb = _ru(K if b_major == "K" else N, 16 if fp8 else 8) + pad
    ldd = _ru(N, 4 if out == "f32" else 8) + pad
    A = si.matrix_bits(seed, M, K, dist, in_fmt, scale=scale, transpose=(a_major == "MN"), ld=lda)
    B = si.matrix_bits(seed + 1, K, N, dist, b_fmt, scale=scale, transpose=(b_major == "K"), ld=ldb)
    C = si.matrix_bits(seed + 2, M, N, dist, out, scale=scale, ld=ldd) if beta != 0.0 else None
    At, Bt = _to_dev(A, in_fmt), _to_dev(B, b_fmt)
    Ct = _to_dev(C, out) if C is not None else None
    Dt = Ct if inplace else torch.full((M, ldd), float("nan"), dtype=TDT[out], device=DEV)
    am, bm, dt = (0 if a_major == "K" else 1), (0 if b_major == "K" else 1), {"f32": 0, "bf16": 1, "f16": 2}[out]
    if fp8:
        g.gemm_fp8_ex(M, N, K, At, FP8[in_fmt], am, lda, Bt, FP8[b_fmt], bm, ldb, Ct, ldd if C is not None else 0,
                      Dt, ldd, dt, alpha, beta, options=options)
    else:
        in_type = {"f16": 0, "bf16": 1, "tf32": 2}[in_fmt]
        g.gemm_ex(in_type, M, N, K, At, am, lda, Bt, bm, ldb, Ct, ldd if C is not None else 0, Dt, ldd, dt,
                  alpha, beta, options=options)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, f"device status word {word:#x}"
    got_bits = _out_bits(Dt, out)[:, :N]
    got = si.bits_to_float64(got_bits, out)
    kw = dict(in_fmt=in_fmt, b_fmt=b_fmt, a_major=a_major, b_major=b_major, lda=lda, ldb=ldb, C=C, c_fmt=out,
              ldc=ldd, alpha=alpha, beta=beta)
    if sample is None:
        ref, S = og.gemm(M, N, K, A, B, **kw)
        rows, cols = slice(None), slice(None)
        gsel = got
        bsel = got_bits
    else:
        rows, cols = sample
        ref, S = og.gemm_entries(M, N, K, A, B, rows, cols, **kw)
        gsel = got[rows, cols]
        bsel = got_bits[rows, cols]
    if exact:
        assert np.array_equal(bsel, og.round_bits(ref, out)), "integer case must be bit-exact"
        return 0.0
    err = np.abs(gsel - ref)
    tol = og.tolerance(S, ref, out)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} entries outside tolerance; first at "
                           f"{np.argwhere(bad)[0]} got {gsel[bad][0]} ref {ref[bad][0]}")
    assert np.isfinite(gsel).all()
    return float(err.max()) if err.size else 0.0


def sample_entries(M, N, n=2048, seed=0):
    """Random entries plus every tile corner along the first and last rows/columns."""
    rng = np.random.default_rng(seed)
    r = list(rng.integers(0, M, n))
    c = list(rng.integers(0, N, n))
    edges_m = sorted({0, 127, 128, 255, 256, M - 129, M - 128, M - 1} & set(range(M)))
    edges_n = sorted({0, 31, 32, 63, 64, 127, 128, 255, 256, N - 1} & set(range(N)))
    for i in edges_m:
        for j in edges_n:
            r.append(i)
            c.append(j)
    return np.array(r, dtype=np.int64), np.array(c, dtype=np.int64)


# ---------------------------------------------------------------- address tables (bit-exact)

@pytest.mark.parametrize("major", ["K", "MN"])
@pytest.mark.parametrize("mode", ["sw32", "sw64", "sw128", "none", "sw128_base32b"])
@pytest.mark.parametrize("rows,bk", [(128, 64), (256, 64), (128, 32), (64, 64), (128, 128)])
def test_device_descriptor_words_match_oracle(g, major, mode, rows, bk):
    W = L.swizzle_width(mode)
    if major == "K" and W > 2 * bk:
        pytest.skip("swizzled K row wider than the K block")
    if major == "K" and mode == L.ATOM32:
        pytest.skip("the 32-byte-atom mode is read for MN-major operands only")
    if major == "MN" and rows % (W // 2):
        pytest.skip("MN atom wider than the tile")
    n = bk // 16
    out = torch.zeros(n + 1, dtype=torch.int64, device=DEV)
    base = 3 * 1024 * 16
    g.gemm_debug_descriptors(0 if major == "K" else 1, SWZ_PARAM[mode], rows, bk, base, n, 1, 128, 1,
                             0, 1, out)
    words = [int(x) & (2 ** 64 - 1) for x in out.cpu().tolist()]
    for j in range(n):
        want = L.encode_smem_desc(L.stage_slice_desc(major, mode, rows, bk, 2, j, base))
        assert words[j] == want, (j, hex(words[j]), hex(want))
    assert words[n] & 0xFFFFFFFF == L.encode_idesc(128, 128, L.FMT_BF16, L.DFMT_F32, 0, 1)


@pytest.mark.parametrize("cg,tile_n,in_type,am,bm", [(1, 256, 1, 0, 0), (2, 256, 0, 0, 1), (1, 64, 1, 1, 0),
                                                       (1, 8, 0, 1, 1)])
def test_device_instruction_descriptor(g, cg, tile_n, in_type, am, bm):
    out = torch.zeros(1, dtype=torch.int64, device=DEV)
    g.gemm_debug_descriptors(0, 3, 128, 64, 0, 0, cg, tile_n, in_type, am, bm, out)
    word = int(out.cpu()[0]) & 0xFFFFFFFF
    assert word == L.encode_idesc(128 * cg, tile_n, in_type, L.DFMT_F32, am, bm)


def _stage_image(g, major, mode, rows, bk, rows_total=None, k_total=None, mn0=0, k0=0):
    rows_total = rows_total or rows
    k_total = k_total or bk
    # element (mn, k) of the stage carries the code mn * bk + k + 1 (0 marks zero fill)
    codes = np.zeros((rows_total, k_total), dtype=np.uint16)
    for mn in range(rows_total):
        for k in range(k_total):
            lm, lk = mn - mn0, k - k0
            if 0 <= lm < rows and 0 <= lk < bk:
                codes[mn, k] = lm * bk + lk + 1
    stored = codes if major == "K" else np.ascontiguousarray(codes.T)
    ld = stored.shape[1]
    src = torch.from_numpy(stored.view(np.int16)).to(DEV)
    out = torch.zeros(rows * bk, dtype=torch.int16, device=DEV)
    g.gemm_debug_stage_image(src, 0 if major == "K" else 1, SWZ_PARAM[mode], rows_total, k_total, ld,
                             rows, bk, mn0, k0, out)
    torch.cuda.synchronize()
    st, word = g.gemm_last_device_status()
    assert st == g.OK, hex(word)
    return out.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("major", ["K", "MN"])
@pytest.mark.parametrize("mode", ["sw32", "sw64", "sw128", "none", "sw128_base32b"])
@pytest.mark.parametrize("rows,bk", [(128, 64), (128, 32), (256, 64), (128, 128)])
def test_tma_stage_image_matches_swizzle_map(g, major, mode, rows, bk):
    # sw128_base32b: TMA's 128B_ATOM_32B mode against the oracle's Swizzle(2, 5, 2)
    W = L.swizzle_width(mode)
    if (major == "K" and W > 2 * bk) or (major == "MN" and rows % (W // 2)):
        pytest.skip("box wider than the stage")
    img = _stage_image(g, major, mode, rows, bk)
    expect = np.zeros(rows * bk, dtype=np.uint16)
    for mn in range(rows):
        for k in range(bk):
            expect[L.stage_element_offset(major, mode, rows, bk, 2, mn, k) // 2] = mn * bk + k + 1
    assert np.array_equal(img, expect)


def test_page_a_tile_lands_where_the_closed_form_says(g):
    # "LBO, SBO and SWZ for a tcgen05 tile": A[128 x 32] fp16, K-major, SW64
    img = _stage_image(g, "K", "sw64", 128, 32)
    for m in range(128):
        for k in range(32):
            assert img[L.p1_a_element_addr(0, m, k) // 2] == m * 32 + k + 1


def test_stage_image_zero_fills_out_of_range(g):
    # the stage hangs over the matrix end in both dimensions: TMA fills zeros
    rows, bk = 128, 64
    img = _stage_image(g, "K", "sw128", rows, bk, rows_total=200, k_total=96, mn0=128, k0=64)
    for mn in range(rows):
        for k in range(bk):
            v = img[L.stage_element_offset("K", "sw128", rows, bk, 2, mn, k) // 2]
            inside = mn + 128 < 200 and k + 64 < 96
            assert v == (mn * bk + k + 1 if inside else 0)


# ---------------------------------------------------------------- the page's single tile

def test_single_tile_fp16_kmajor_a_mnmajor_b_exact(g):
    run_case(g, 128, 128, 32, in_fmt="f16", a_major="K", b_major="MN", dist="int4", exact=True)


def test_single_tile_fp16_uniform(g):
    run_case(g, 128, 128, 32, in_fmt="f16", a_major="K", b_major="MN", dist="uniform")


def test_single_k16_mma_exact(g):
    run_case(g, 128, 128, 16, in_fmt="f16", a_major="K", b_major="MN", dist="int4", exact=True)


def test_identity_a_gives_b(g):
    n = 256
    eye = si.to_storage(np.eye(n), "bf16")
    B = si.matrix_bits(5, n, n, "uniform", "bf16")
    D = torch.empty(n, n, dtype=torch.float32, device=DEV)
    g.gemm_bf16(n, n, n, _to_dev(eye, "bf16"), 0, n, _to_dev(B, "bf16"), 1, n, None, 0, D, n, 0, 1.0, 0.0)
    assert np.array_equal(D.cpu().numpy().astype(np.float64), si.bits_to_float64(B, "bf16"))


# ---------------------------------------------------------------- shapes, majors, outputs

@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("K", "MN"), ("MN", "K"), ("MN", "MN")])
@pytest.mark.parametrize("cg", [1, 2])
def test_majors_integer_exact(g, a_major, b_major, cg):
    run_case(g, 384, 320, 192, a_major=a_major, b_major=b_major, dist="int4", exact=True,
             options=dict(cta_group=cg))


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 200, 136), (129, 65, 72), (640, 384, 512),
                                   (1, 8, 8), (130, 520, 1000)])
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_ragged_shapes(g, M, N, K, out):
    run_case(g, M, N, K, out=out, dist="normal", a_major="K", b_major="MN")


@pytest.mark.parametrize("cg,tile_n,bk", [(1, 64, 64), (1, 64, 128), (1, 128, 64), (1, 128, 128), (1, 256, 64),
                                          (2, 256, 64), (2, 256, 128), (2, 128, 128)])
@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("MN", "MN"), ("K", "MN")])
def test_tile_configs(g, cg, tile_n, bk, a_major, b_major):
    run_case(g, 520, 600, 264, a_major=a_major, b_major=b_major, dist="normal",
             options=dict(cta_group=cg, tile_n=tile_n, block_k=bk))
    run_case(g, 384, 320, 200, a_major=a_major, b_major=b_major, dist="int4", exact=True,
             options=dict(cta_group=cg, tile_n=tile_n, block_k=bk))


@pytest.mark.parametrize("swz_a", [1, 2, 3, 4])
@pytest.mark.parametrize("swz_b", [1, 2, 3, 4])
@pytest.mark.parametrize("a_major,b_major", [("K", "MN"), ("MN", "K")])
@pytest.mark.parametrize("bk", [64, 128])
def test_swizzle_modes(g, swz_a, swz_b, a_major, b_major, bk):
    run_case(g, 256, 256, 320, a_major=a_major, b_major=b_major, dist="int4", exact=True,
             options=dict(swizzle_a=swz_a, swizzle_b=swz_b, tile_n=128, block_k=bk))


@pytest.mark.parametrize("cg", [1, 2])
def test_no_swizzle_operands_all_majors(g, cg):
    for am, bm in (("K", "K"), ("K", "MN"), ("MN", "K"), ("MN", "MN")):
        run_case(g, 300, 264, 200, a_major=am, b_major=bm, dist="int4", exact=True,
                 options=dict(cta_group=cg, swizzle_a=4, swizzle_b=4))


def test_unswizzled_epilogue_staging(g):
    run_case(g, 300, 260, 128, dist="normal", beta=0.5, options=dict(epilogue_swizzle=-1))
    run_case(g, 300, 260, 128, dist="normal", out="bf16", options=dict(epilogue_swizzle=-1))


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("cg", [1, 2])
def test_alpha_beta(g, out, cg):
    run_case(g, 264, 320, 160, out=out, alpha=-0.75, beta=1.25, dist="uniform", options=dict(cta_group=cg))


def test_in_place_c_equals_d(g):
    run_case(g, 256, 192, 96, out="f32", alpha=1.0, beta=1.0, inplace=True)


def test_fp16_inputs(g):
    run_case(g, 384, 256, 320, in_fmt="f16", out="f16", dist="normal", a_major="MN", b_major="K")
    run_case(g, 256, 256, 128, in_fmt="f16", out="f32", dist="int4", exact=True, options=dict(cta_group=2))


def test_padded_leading_dimensions(g):
    run_case(g, 200, 136, 104, pad=8, out="f32", beta=1.0, a_major="K", b_major="K")
    run_case(g, 200, 136, 104, pad=24, out="bf16", a_major="MN", b_major="MN")


def test_k_zero_gives_beta_c(g):
    run_case(g, 130, 70, 0, out="f32", alpha=2.0, beta=0.5)


@pytest.mark.parametrize("M,N,K,tn", [(1000, 136, 1000, 128), (128, 1000, 520, 64), (384, 512, 64, 256)])
def test_rotated_k_start(g, M, N, K, tn):
    run_case(g, M, N, K, dist="int4", exact=True, options=dict(tile_n=tn, flags=4))
    run_case(g, M, N, K, dist="normal", out="bf16", beta=1.0, options=dict(tile_n=tn, flags=4))


def test_k_tail_and_single_column(g):
    run_case(g, 128, 8, 40, dist="int4", exact=True)
    run_case(g, 64, 264, 8, dist="int4", exact=True)


# ---------------------------------------------------------------- full-size configurations (sampled)

def test_config2_square_4096_bf16_out(g):
    # single CTAs of 128 x 256 (the 128-row tile, split over the ragged fourth wave)
    M = N = K = 4096
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_case(g, M, N, K, a_major="K", b_major="K", out="bf16", dist="normal", scale=0.1, seed=10,
             options=dict(cta_group=1, tile_n=256, tile_m=128, workspace=ws), sample=sample_entries(M, N))


def test_config2_square_4096_bench_launch(g):
    # the launch bench.py times: cta_group 1 and a stream-K workspace, the library
    # choosing the tile (two-half 256 x 224: two full rounds on 152 SMs, unsplit)
    M = N = K = 4096
    ws = torch.zeros(g.gemm_streamk_workspace_size(), dtype=torch.uint8, device=DEV)
    run_case(g, M, N, K, a_major="K", b_major="K", out="bf16", dist="normal", scale=0.1, seed=10,
             options=dict(cta_group=1, workspace=ws), sample=sample_entries(M, N, n=1024, seed=7))


def test_config3_square_8192_pair_fp32_beta(g):
    M = N = K = 8192
    run_case(g, M, N, K, a_major="K", b_major="MN", out="f32", alpha=1.0, beta=1.0, dist="uniform", seed=20,
             options=dict(cta_group=2, tile_n=256), sample=sample_entries(M, N, n=1024))


@pytest.mark.parametrize("M,N,K", [(16384, 128, 8192), (128, 16384, 4096)])
@pytest.mark.parametrize("cg", [1, 2])
def test_config4_skinny(g, M, N, K, cg):
    run_case(g, M, N, K, a_major="K", b_major="K", out="bf16", dist="normal", seed=30,
             sample=sample_entries(M, N, n=1024), options=dict(cta_group=cg))


# ---------------------------------------------------------------- grouped

def _grouped(g, Ms, N, K, *, out="bf16", a_major="K", b_major="K", alpha=1.0, beta=0.0, seed=40,
             dist="uniform", sample=None, options=None):
    """Grouped GEMM through the C ABI (gemm_bf16_grouped, or gemm_grouped_ex with options)."""
    probs, host = [], []
    ldd = _ru(N, 4 if out == "f32" else 8)
    for i, M in enumerate(Ms):
        lda = _ru(K if a_major == "K" else M, 8)
        ldb = _ru(K if b_major == "K" else N, 8)
        A = si.matrix_bits(seed + 3 * i, M, K, dist, "bf16", transpose=(a_major == "MN"), ld=lda)
        B = si.matrix_bits(seed + 3 * i + 1, K, N, dist, "bf16", transpose=(b_major == "K"), ld=ldb)
        C = si.matrix_bits(seed + 3 * i + 2, M, N, dist, out, ld=ldd) if beta != 0.0 else None
        At, Bt = _to_dev(A, "bf16"), _to_dev(B, "bf16")
        Ct = _to_dev(C, out) if C is not None else None
        Dt = torch.full((max(M, 1), ldd), float("nan"), dtype=TDT[out], device=DEV)
        probs.append(dict(M=M, N=N, K=K, A=At, B=Bt, C=Ct, D=Dt, lda=lda, ldb=ldb,
                          ldc=ldd if C is not None else 0, ldd=ldd))
        host.append((A, B, C, Dt, lda, ldb))
    ws_bytes = g.gemm_grouped_workspace_size(len(Ms))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    am, bm, dt = (0 if a_major == "K" else 1), (0 if b_major == "K" else 1), {"f32": 0, "bf16": 1, "f16": 2}[out]
    if options:
        g.gemm_grouped_ex(1, probs, am, bm, dt, alpha, beta, ws, ws_bytes, options=options)
    else:
        g.gemm_bf16_grouped(probs, am, bm, dt, alpha, beta, ws, ws_bytes)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, hex(word)
    for i, (M, (A, B, C, Dt, lda, ldb)) in enumerate(zip(Ms, host)):
        if M == 0:
            continue
        got = si.bits_to_float64(_out_bits(Dt, out)[:, :N], out)
        kw = dict(in_fmt="bf16", a_major=a_major, b_major=b_major, lda=lda, ldb=ldb, C=C, c_fmt=out, ldc=ldd,
                  alpha=alpha, beta=beta)
        if sample:
            r, c = sample_entries(M, N, n=256, seed=i)
            ref, S = og.gemm_entries(M, N, K, A, B, r, c, **kw)
            got = got[r, c]
        else:
            ref, S = og.gemm(M, N, K, A, B, **kw)
        err = np.abs(got - ref)
        assert (err <= og.tolerance(S, ref, out)).all(), f"problem {i}: max err {err.max()}"


def test_grouped_small_varied(g):
    _grouped(g, [128, 256, 0, 384, 200, 130], 320, 136, out="bf16")
    _grouped(g, [64, 300, 128], 136, 72, out="f32", alpha=0.5, beta=-1.0, a_major="MN", b_major="MN")


def test_grouped_cta_pairs_with_odd_row_tiles(g):
    # pair tiles are 256 rows; 128-row and ragged problems leave the odd CTA partly idle
    _grouped(g, [128, 384, 200, 512, 0, 136], 264, 192, out="bf16", options=dict(cta_group=2))
    _grouped(g, [256, 130], 136, 320, out="f32", beta=1.0, a_major="MN", b_major="MN", options=dict(cta_group=2))


def test_grouped_k_zero_problem(g):
    _grouped(g, [128, 256], 128, 0, out="f32", beta=2.0)


@pytest.mark.parametrize("cg", [1, 2])
def test_config5_grouped_64_problems(g, cg):
    rng = np.random.default_rng(5)
    Ms = [int(x) for x in rng.integers(1, 33, 64) * 128]
    _grouped(g, Ms, 4096, 2048, out="bf16", dist="uniform", seed=100, sample=True, options=dict(cta_group=cg))


# ---------------------------------------------------------------- 64-row tiles (M = 64, TMEM Layout F)

@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("MN", "MN"), ("K", "MN")])
@pytest.mark.parametrize("max_ctas", [0, 1])
def test_m64_tiles_exact(g, tile_n, a_major, b_major, max_ctas):
    # max_ctas = 1: one CTA walks every tile, alternating the lane-0 and lane-16 accumulators
    run_case(g, 200, 520, 264, a_major=a_major, b_major=b_major, dist="int4", exact=True,
             options=dict(tile_m=64, tile_n=tile_n, max_ctas=max_ctas))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_m64_tiles_alpha_beta_ragged(g, out):
    run_case(g, 130, 264, 200, out=out, alpha=0.5, beta=-1.0, dist="normal",
             options=dict(tile_m=64, max_ctas=2))


def test_small_m_defaults_to_64_row_tiles(g):
    run_case(g, 48, 1000, 520, dist="normal", out="bf16")
    run_case(g, 64, 16384, 512, dist="int4", exact=True)


# ---------------------------------------------------------------- fp8 operands (kind::f8f6f4)

@pytest.mark.parametrize("major", ["K", "MN"])
@pytest.mark.parametrize("mode", ["sw64", "sw128", "none", "sw128_base32b"])
@pytest.mark.parametrize("rows,bk", [(128, 128), (128, 256), (256, 128)])
def test_fp8_descriptor_words_match_oracle(g, major, mode, rows, bk):
    W = L.swizzle_width(mode)
    if (major == "K" and W > bk) or (major == "MN" and rows % W):
        pytest.skip("box wider than the stage")
    if major == "K" and mode == L.ATOM32:
        pytest.skip("the 32-byte-atom mode is read for MN-major operands only")
    n = bk // 32
    out = torch.zeros(n + 1, dtype=torch.int64, device=DEV)
    g.gemm_debug_descriptors(0 if major == "K" else 1, SWZ_PARAM[mode], rows, bk, 8192, n, 1, 256, 2, 0, 1, out)
    words = [int(x) & (2 ** 64 - 1) for x in out.cpu().tolist()]
    for j in range(n):
        assert words[j] == L.encode_smem_desc(L.stage_slice_desc(major, mode, rows, bk, 1, j, 8192)), j
    assert words[n] & 0xFFFFFFFF == L.encode_idesc(128, 256, L.FMT_E4M3, L.DFMT_F32, 0, 1)


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e5m2", "e5m2")])
@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("K", "MN"), ("MN", "K"), ("MN", "MN")])
def test_fp8_integer_exact(g, fa, fb, a_major, b_major):
    run_case(g, 384, 320, 512, in_fmt=fa, b_fmt=fb, a_major=a_major, b_major=b_major, dist="int4", exact=True)


@pytest.mark.parametrize("cg,tile_n", [(1, 128), (1, 256), (2, 256)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fp8_tiles_ragged(g, cg, tile_n, out):
    run_case(g, 520, 600, 272, in_fmt="e4m3", b_fmt="e4m3", a_major="K", b_major="MN", out=out, dist="uniform",
             options=dict(cta_group=cg, tile_n=tile_n))
    run_case(g, 300, 264, 160, in_fmt="e5m2", b_fmt="e4m3", out=out, dist="int4", exact=True,
             beta=0.5 if out == "f32" else 0.0, options=dict(cta_group=cg, tile_n=tile_n))


@pytest.mark.parametrize("swz", [1, 2, 4])
def test_fp8_swizzle_modes(g, swz):
    run_case(g, 256, 256, 256, in_fmt="e4m3", a_major="K", b_major="MN", dist="int4", exact=True,
             options=dict(swizzle_a=swz, swizzle_b=swz, tile_n=128))


def test_fp8_square_8192_pair_sampled(g):
    M = N = K = 8192
    run_case(g, M, N, K, in_fmt="e4m3", a_major="K", b_major="K", out="bf16", dist="uniform", seed=40,
             options=dict(cta_group=2), sample=sample_entries(M, N, n=1024))


@pytest.mark.parametrize("flags", [0, 1, 2, 3, 4, 5])
def test_pair_signalling_modes(g, flags):
    # multicast commits (0), forwarded releases (1), cluster-scope waits (2), both (3), rotated K (4, 5)
    run_case(g, 640, 768, 320, a_major="K", b_major="MN", dist="int4", exact=True,
             options=dict(cta_group=2, flags=flags))
    run_case(g, 512, 512, 256, out="bf16", beta=0.5, dist="normal", options=dict(cta_group=2, flags=flags))


# ---------------------------------------------------------------- bounded waits

def test_injected_wait_times_out_and_the_context_survives(g):
    g.gemm_debug_inject_timeout(20)
    M = N = K = 256
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(N, K, dtype=torch.bfloat16, device=DEV)
    D = torch.zeros(M, N, dtype=torch.float32, device=DEV)
    g.gemm_bf16(M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0)
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and word != 0
    # the library and the context still work afterwards
    run_case(g, 256, 128, 64, dist="int4", exact=True)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_injected_producer_wait_times_out_and_the_context_survives(g, cta_group):
    # the producer (of both CTAs of a pair) waits on a barrier nothing arrives at before
    # its first load: every other role gives up on the abort flag, the status names the
    # producer and the injected wait, and the next calls compute correctly
    g.gemm_debug_inject_timeout(20, role=1)
    M = N = K = 512
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(N, K, dtype=torch.bfloat16, device=DEV)
    D = torch.zeros(M, N, dtype=torch.float32, device=DEV)
    g.gemm_ex(1, M, N, K, A, 0, K, B, 0, K, None, 0, D, N, 0, 1.0, 0.0, options=dict(cta_group=cta_group))
    st, word = g.gemm_last_device_status()
    assert st == g.ERR_TIMEOUT and (word & 0xFF, (word >> 8) & 0xFF) == (1, 6), hex(word)
    run_case(g, 512, 384, 256, dist="int4", exact=True, options=dict(cta_group=cta_group))
    run_case(g, 300, 200, 192, dist="int4", exact=True, options=dict(cta_group=cta_group))
