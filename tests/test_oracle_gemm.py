"""Pins of the fp64 GEMM oracle: exact integer products, identities, a hand case,
brute force in exact rationals, an independent library matmul, and the rounding."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import gemm as G


def _vals(bits, fmt):
    return si.bits_to_float64(bits, fmt)


# ---------------------------------------------------------------------------
# Exact cases.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("K", "MN"), ("MN", "K"), ("MN", "MN")])
@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_integer_inputs_give_the_exact_integer_product(a_major, b_major, fmt):
    M, N, K = 37, 29, 64
    A = si.matrix_bits(1, M, K, "int4", fmt, transpose=(a_major == "MN"))
    B = si.matrix_bits(2, K, N, "int4", fmt, transpose=(b_major == "K"))
    D, S = G.gemm(M, N, K, A, B, in_fmt=fmt, a_major=a_major, b_major=b_major)
    Ai = si.logical_values(1, M, K, "int4").astype(np.int64)
    Bi = si.logical_values(2, K, N, "int4").astype(np.int64)
    assert np.array_equal(D, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


def test_identity_gives_b_exactly():
    K = N = 48
    eye = si.to_storage(np.eye(K), "bf16")
    B = si.matrix_bits(7, K, N, "uniform", "bf16")
    D, _ = G.gemm(K, N, K, eye, B, in_fmt="bf16", a_major="K", b_major="MN")
    assert np.array_equal(D, _vals(B, "bf16"))


def test_single_k16_slice_integer():
    # the K = 16 extent of one kind::f16 MMA
    M, N, K = 128, 128, 16
    A = si.matrix_bits(3, M, K, "int4", "f16")
    B = si.matrix_bits(4, K, N, "int4", "f16", transpose=True)
    D, _ = G.gemm(M, N, K, A, B, in_fmt="f16", a_major="K", b_major="K")
    ref = si.logical_values(3, M, K, "int4") @ si.logical_values(4, K, N, "int4")
    assert np.array_equal(D, ref)


def test_hand_case_4x4():
    # A = [[1,2,0,-1],[0,1,3,0],[2,0,0,1],[-1,1,1,1]], B = [[1,0,2,0],[0,1,0,3],[4,0,1,0],[0,2,0,1]]
    A = np.array([[1, 2, 0, -1], [0, 1, 3, 0], [2, 0, 0, 1], [-1, 1, 1, 1]], dtype=np.float64)
    B = np.array([[1, 0, 2, 0], [0, 1, 0, 3], [4, 0, 1, 0], [0, 2, 0, 1]], dtype=np.float64)
    expect = np.array([[1, 0, 2, 5], [12, 1, 3, 3], [2, 2, 4, 1], [3, 3, -1, 4]], dtype=np.float64)
    C = np.full((4, 4), 0.5)
    D, S = G.gemm(4, 4, 4, si.to_storage(A, "f16"), si.to_storage(B, "f16"), in_fmt="f16",
                  a_major="K", b_major="MN", C=si.to_storage(C, "f32"), c_fmt="f32",
                  alpha=2.0, beta=-1.0)
    assert np.array_equal(D, 2.0 * expect - 0.5)
    assert S[0, 3] == 2.0 * (0 * 0 + 2 * 3 + 0 * 0 + 1 * 1) + 0.5


def test_beta_zero_never_reads_c():
    A = si.matrix_bits(1, 8, 8, "uniform", "bf16")
    B = si.matrix_bits(2, 8, 8, "uniform", "bf16")
    nan_c = np.full((8, 8), np.nan)
    D1, _ = G.gemm(8, 8, 8, A, B, C=si.to_storage(nan_c, "f32"), beta=0.0)
    D2, _ = G.gemm(8, 8, 8, A, B)
    assert np.array_equal(D1, D2) and np.isfinite(D1).all()


def test_k_zero_is_beta_c():
    C = si.matrix_bits(9, 5, 6, "uniform", "f32")
    empty = np.zeros(0, dtype=np.uint16)
    D, S = G.gemm(5, 6, 0, empty, empty, C=C, c_fmt="f32", alpha=3.0, beta=0.25)
    assert np.array_equal(D, 0.25 * _vals(C, "f32"))


# ---------------------------------------------------------------------------
# Brute force in exact rationals on tiny inputs; a plausible slip must fail.
# ---------------------------------------------------------------------------

def _exact(Av, Bv, Cv, alpha, beta):
    M, K = Av.shape
    N = Bv.shape[1]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(Av[i, k]) * Fraction(Bv[k, j]) for k in range(K))
            out[i, j] = float(Fraction(alpha) * s + Fraction(beta) * Fraction(Cv[i, j]))
    return out


@pytest.mark.parametrize("a_major,b_major", [("K", "MN"), ("MN", "K")])
def test_matches_exact_rationals(a_major, b_major):
    M, N, K = 5, 7, 9
    A = si.matrix_bits(11, M, K, "uniform", "bf16", transpose=(a_major == "MN"))
    B = si.matrix_bits(12, K, N, "normal", "bf16", transpose=(b_major == "K"))
    C = si.matrix_bits(13, M, N, "uniform", "f32")
    Av = _vals(si.matrix_bits(11, M, K, "uniform", "bf16"), "bf16")
    Bv = _vals(si.matrix_bits(12, K, N, "normal", "bf16"), "bf16")
    Cv = _vals(C, "f32")
    D, _ = G.gemm(M, N, K, A, B, a_major=a_major, b_major=b_major, C=C, alpha=0.75, beta=-1.5)
    ex = _exact(Av, Bv, Cv, 0.75, -1.5)
    assert np.allclose(D, ex, rtol=1e-14, atol=1e-15)
    Dt, _ = G.gemm(M, N, K, A, B, a_major=a_major, b_major=b_major, C=C, alpha=0.75, beta=1.5)
    assert not np.allclose(Dt, ex)                  # a sign slip on beta is caught


def test_square_transposed_operand_is_caught():
    n = 16
    A = si.matrix_bits(21, n, n, "uniform", "bf16")
    B = si.matrix_bits(22, n, n, "uniform", "bf16")
    D_k, _ = G.gemm(n, n, n, A, B, a_major="K", b_major="MN")
    D_t, _ = G.gemm(n, n, n, A, B, a_major="MN", b_major="MN")
    assert not np.allclose(D_k, D_t)
    ex = _vals(A, "bf16") @ _vals(B, "bf16")
    assert np.allclose(D_k, ex, rtol=1e-13)


def test_matches_torch_float64_matmul():
    M, N, K = 70, 90, 130
    A = si.matrix_bits(31, M, K, "normal", "bf16", scale=0.1)
    B = si.matrix_bits(32, K, N, "normal", "bf16", scale=0.1, transpose=True)
    C = si.matrix_bits(33, M, N, "uniform", "f32")
    D, S = G.gemm(M, N, K, A, B, a_major="K", b_major="K", C=C, alpha=1.25, beta=0.5)
    At = torch.from_numpy(_vals(A, "bf16"))
    Bt = torch.from_numpy(_vals(B, "bf16")).T
    ref = 1.25 * (At @ Bt) + 0.5 * torch.from_numpy(_vals(C, "f32"))
    assert np.allclose(D, ref.numpy(), rtol=1e-12, atol=1e-12)
    absref = 1.25 * (At.abs() @ Bt.abs()) + 0.5 * torch.from_numpy(_vals(C, "f32")).abs()
    assert np.allclose(S, absref.numpy(), rtol=1e-12)


def test_entries_match_full_product():
    M, N, K = 33, 41, 57
    A = si.matrix_bits(41, M, K, "uniform", "f16", transpose=True)
    B = si.matrix_bits(42, K, N, "uniform", "f16")
    C = si.matrix_bits(43, M, N, "uniform", "f16")
    D, S = G.gemm(M, N, K, A, B, in_fmt="f16", a_major="MN", b_major="MN", C=C, c_fmt="f16",
                  alpha=-0.5, beta=2.0)
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, M, 200), rng.integers(0, N, 200)
    De, Se = G.gemm_entries(M, N, K, A, B, rows, cols, in_fmt="f16", a_major="MN", b_major="MN",
                            C=C, c_fmt="f16", alpha=-0.5, beta=2.0)
    assert np.array_equal(De, D[rows, cols]) and np.array_equal(Se, S[rows, cols])
    with pytest.raises(ValueError):
        G.gemm_entries(M, N, K, A, B, [M], [0], in_fmt="f16", a_major="MN", b_major="MN")


def test_leading_dimensions():
    M, N, K = 9, 10, 11
    A = si.matrix_bits(51, M, K, "uniform", "bf16", ld=24)
    B = si.matrix_bits(52, K, N, "uniform", "bf16", ld=16)
    C = si.matrix_bits(53, M, N, "uniform", "f32", ld=12)
    D, _ = G.gemm(M, N, K, A, B, a_major="K", b_major="MN", lda=24, ldb=16, C=C, ldc=12, beta=1.0)
    ref = _vals(A, "bf16")[:, :K] @ _vals(B, "bf16")[:, :N] + _vals(C, "f32")[:, :N]
    assert np.allclose(D, ref, rtol=1e-13)


# ---------------------------------------------------------------------------
# Output rounding: round-to-nearest-even in one step.
# ---------------------------------------------------------------------------

def test_round_f16_and_f32_match_correctly_rounded_casts():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(size=3000) * 10.0 ** rng.integers(-9, 5, 3000),
                        [0.0, -0.0, 65504.0, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]])
    r16 = G.round_to(x, "f16")
    assert np.array_equal(r16, x.astype(np.float16).astype(np.float64))
    r32 = G.round_to(x, "f32")
    assert np.array_equal(r32, x.astype(np.float32).astype(np.float64))
    assert np.array_equal(G.round_bits(x, "f16"), x.astype(np.float16).view(np.uint16))
    assert np.array_equal(G.round_bits(x, "f32"), x.astype(np.float32).view(np.uint32))


def test_round_bf16_ties_and_no_double_rounding():
    one = 1.0
    cases = {
        one + 2.0 ** -8: one,                              # tie -> even (down)
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,              # tie -> even (up)
        one + 2.0 ** -8 + 2.0 ** -30: one + 2.0 ** -7,     # just above the tie; via f32 it would tie
        -(one + 2.0 ** -8 + 2.0 ** -30): -(one + 2.0 ** -7),
        2.0 ** 127 * (2 - 2.0 ** -8): float("inf"),        # rounds past the largest finite bf16
        2.0 ** -133: 2.0 ** -133,                          # subnormal, exact
        3 * 2.0 ** -134: 2.0 ** -132,                      # subnormal tie 1.5 steps -> even (2 steps)
    }
    for x, want in cases.items():
        assert G.round_to(np.array([x]), "bf16")[0] == want, x
    bits = G.round_bits(np.array([1.0, -2.0, 1.0 + 2.0 ** -7]), "bf16")
    assert list(bits) == [0x3F80, 0xC000, 0x3F81]


def test_ulp_and_tolerance():
    assert G.ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert G.ulp(np.array([1.0]), "f16")[0] == 2.0 ** -10
    assert G.ulp(np.array([1.5]), "f32")[0] == 2.0 ** -23
    assert G.ulp(np.array([0.0]), "f16")[0] == 2.0 ** -24
    assert G.tolerance(np.array([1000.0]), np.array([1.0]), "bf16")[0] == 1.0 + 2.0 ** -7


# ---------------------------------------------------------------------------
# fp8 operands (E4M3 / E5M2): decoding against format facts and an
# independent codec, and exact products.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,tdt", [("e4m3", "float8_e4m3fn"), ("e5m2", "float8_e5m2")])
def test_fp8_decode_matches_torch_for_every_code(fmt, tdt):
    codes = np.arange(256, dtype=np.uint8)
    ours = G.decode(codes, fmt)
    theirs = torch.from_numpy(codes).view(getattr(torch, tdt)).double().numpy()
    same = (ours == theirs) | (np.isnan(ours) & np.isnan(theirs))
    assert same.all()


def test_fp8_format_facts():
    # E4M3: 1.0 = 0x38, largest finite 0x7E = 448, smallest normal 0x08 = 2^-6,
    # smallest subnormal 0x01 = 2^-9, 0x7F is NaN, no infinity
    d = G.decode(np.array([0x38, 0xB8, 0x7E, 0x08, 0x01, 0x7F, 0x78], dtype=np.uint8), "e4m3")
    assert list(d[:5]) == [1.0, -1.0, 448.0, 2.0 ** -6, 2.0 ** -9] and np.isnan(d[5]) and d[6] == 256.0
    # E5M2: 1.0 = 0x3C, largest finite 0x7B = 57344, 0x7C = inf, smallest subnormal 2^-16
    d = G.decode(np.array([0x3C, 0x7B, 0x7C, 0x01, 0x04, 0x7D], dtype=np.uint8), "e5m2")
    assert list(d[:5]) == [1.0, 57344.0, np.inf, 2.0 ** -16, 2.0 ** -14] and np.isnan(d[5])


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e5m2")])
def test_fp8_integer_products_are_exact(fa, fb):
    M, N, K = 24, 40, 96
    A = si.matrix_bits(61, M, K, "int4", fa)
    B = si.matrix_bits(62, K, N, "int4", fb, transpose=True)
    D, _ = G.gemm(M, N, K, A, B, in_fmt=fa, b_fmt=fb, a_major="K", b_major="K")
    ref = si.logical_values(61, M, K, "int4").astype(np.int64) @ si.logical_values(62, K, N, "int4").astype(np.int64)
    assert np.array_equal(D, ref.astype(np.float64))


def test_fp8_mixed_formats_match_float64_matmul():
    M, N, K = 17, 33, 64
    A = si.matrix_bits(71, M, K, "normal", "e4m3")
    B = si.matrix_bits(72, K, N, "normal", "e5m2")
    D, _ = G.gemm(M, N, K, A, B, in_fmt="e4m3", b_fmt="e5m2", a_major="K", b_major="MN")
    ref = si.bits_to_float64(A, "e4m3") @ si.bits_to_float64(B, "e5m2")
    assert np.allclose(D, ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# Block-scaled (MXFP8) product: one E8M0 scale per 32 elements of K.
# ---------------------------------------------------------------------------

def test_e8m0_decode_is_a_power_of_two_and_255_is_nan():
    d = G.decode_e8m0(np.array([0, 1, 126, 127, 128, 254, 255], dtype=np.uint8))
    assert list(d[:6]) == [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127]
    assert np.isnan(d[6])


def test_mx_unit_scales_reduce_to_the_fp8_product():
    M, N, K = 9, 13, 100
    A = si.matrix_bits(81, M, K, "normal", "e4m3")
    B = si.matrix_bits(82, K, N, "normal", "e5m2", transpose=True)
    ones_a = np.full((M, 4), 127, np.uint8)
    ones_b = np.full((N, 4), 127, np.uint8)
    D, S = G.gemm_mx(M, N, K, A, B, ones_a, ones_b, in_fmt="e4m3", b_fmt="e5m2")
    D0, S0 = G.gemm(M, N, K, A, B, in_fmt="e4m3", b_fmt="e5m2")
    assert np.array_equal(D, D0) and np.array_equal(S, S0)


def test_mx_hand_case_in_exact_rationals():
    # one output, K = 70: blocks [0,32), [32,64) and the partial block [64,70)
    K = 70
    A = si.matrix_bits(83, 1, K, "normal", "e4m3")
    B = si.matrix_bits(84, K, 1, "normal", "e4m3", transpose=True)
    sa = np.array([[125, 130, 127]], np.uint8)
    sb = np.array([[129, 126, 131]], np.uint8)
    a = _vals(A, "e4m3").reshape(-1)
    b = _vals(B, "e4m3").reshape(-1)
    want = Fraction(0)
    for k in range(K):
        blk = k // 32
        want += (Fraction(2) ** (int(sa[0, blk]) - 127) * Fraction(a[k])) * \
                (Fraction(2) ** (int(sb[0, blk]) - 127) * Fraction(b[k]))
    D, _ = G.gemm_mx(1, 1, K, A, B, sa, sb, alpha=1.0)
    assert Fraction(D[0, 0]) == want


@pytest.mark.parametrize("a_major,b_major", [("K", "K"), ("MN", "K"), ("K", "MN")])
def test_mx_integer_inputs_with_power_of_two_scales_are_exact(a_major, b_major):
    M, N, K = 20, 36, 160
    A = si.matrix_bits(85, M, K, "int4", "e4m3", transpose=(a_major == "MN"))
    B = si.matrix_bits(86, K, N, "int4", "e4m3", transpose=(b_major == "K"))
    sa = si.scale_codes(87, M, K // 32)
    sb = si.scale_codes(88, N, K // 32)
    D, _ = G.gemm_mx(M, N, K, A, B, sa, sb, a_major=a_major, b_major=b_major)
    a = si.logical_values(85, M, K, "int4")
    b = si.logical_values(86, K, N, "int4")
    ref = np.zeros((M, N))
    for blk in range(K // 32):
        s = slice(32 * blk, 32 * blk + 32)
        ref += np.exp2(sa[:, blk:blk + 1] - 127.0) * (a[:, s] @ b[s, :]) * np.exp2(sb[:, blk][None, :] - 127.0)
    assert np.array_equal(D, ref)
    # swapping the roles of the two scale tables (a transposed reading) is caught
    D_bad, _ = G.gemm_mx(M, N, K, A, B, sa[:, ::-1], sb, a_major=a_major, b_major=b_major)
    assert not np.array_equal(D_bad, ref)


def test_mx_entries_match_full_product():
    M, N, K = 40, 24, 96
    A = si.matrix_bits(89, M, K, "normal", "e4m3")
    B = si.matrix_bits(90, K, N, "normal", "e4m3", transpose=True)
    sa = si.scale_codes(91, M, 3)
    sb = si.scale_codes(92, N, 3)
    C = si.matrix_bits(93, M, N, "normal", "f32")
    D, S = G.gemm_mx(M, N, K, A, B, sa, sb, C=C, alpha=0.5, beta=-2.0)
    rows = np.array([0, 39, 17, 5]); cols = np.array([0, 23, 11, 20])
    De, Se = G.gemm_mx_entries(M, N, K, A, B, sa, sb, rows, cols, C=C, alpha=0.5, beta=-2.0)
    assert np.array_equal(De, D[rows, cols]) and np.array_equal(Se, S[rows, cols])


def test_mx_scale_atom_layout_by_hand():
    # the atom arrangement the block-scaled ABI documents, checked at hand-picked positions
    rows, K = 300, 260                       # 3 row blocks, 9 scale blocks in 3 K groups
    codes = np.zeros((rows, 9), np.uint8)
    codes[33, 5] = 201                       # row block 0, K group 1, byte 16*1 + 4*1 + 1
    codes[130, 8] = 202                      # row block 1, K group 2, byte 16*2 + 4*0 + 0
    codes[299, 0] = 203                      # row block 2, K group 0, byte 16*11 + 4*1 + 0
    atoms = si.mx_scale_atoms(codes, rows, K)
    assert atoms.size == 3 * 3 * 512
    assert atoms[(0 * 3 + 1) * 512 + 21] == 201
    assert atoms[(1 * 3 + 2) * 512 + 32] == 202
    assert atoms[(2 * 3 + 0) * 512 + 180] == 203
    assert (atoms == 201).sum() == 1 and (atoms == 202).sum() == 1 and (atoms == 203).sum() == 1


# ---------------------------------------------------------------------------
# Block-scaled fp4 (NVFP4: UE4M3 per 16; MXFP4: E8M0 per 32), packed E2M1.
# ---------------------------------------------------------------------------

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # the eight E2M1 magnitudes (OCP Microscaling)


def test_e2m1_decode_matches_the_format_table():
    d = G.decode_e2m1(np.arange(16, dtype=np.uint8))
    assert list(d[:8]) == E2M1_TABLE
    assert list(-d[8:]) == E2M1_TABLE and all(np.signbit(d[8:]))


def test_ue4m3_decode_matches_torch_e4m3_for_every_unsigned_code():
    codes = np.arange(0x7F, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(G.decode_ue4m3(codes), want)
    assert np.isnan(G.decode_ue4m3(np.array([0x7F], np.uint8))[0])


def test_fp4_nibble_order_hand_case():
    # one output, K = 2: A = [1, 2], B = [3, 0.5]: 1*3 + 2*0.5 = 4 (the swapped order would give 6.5)
    A = np.array([[0x2 | (0x4 << 4)]], np.uint8)      # codes 2 (1.0) low, 4 (2.0) high
    B = np.array([[0x5 | (0x1 << 4)]], np.uint8)      # codes 5 (3.0) low, 1 (0.5) high
    one16 = np.array([[0x38]], np.uint8)              # UE4M3 1.0
    D, _ = G.gemm_fp4(1, 1, 2, A, B, one16, one16, block=16, scale="ue4m3")
    assert D[0, 0] == 4.0
    one32 = np.array([[127]], np.uint8)
    D, _ = G.gemm_fp4(1, 1, 2, A, B, one32, one32, block=32, scale="e8m0")
    assert D[0, 0] == 4.0


@pytest.mark.parametrize("block,scale", [(16, "ue4m3"), (32, "e8m0")])
def test_fp4_products_with_scales_are_exact(block, scale):
    M, N, K = 12, 20, 192
    ca, cb = si.fp4_codes(101, M, K), si.fp4_codes(102, N, K)
    nb = K // block
    rng = np.random.default_rng(103)
    if scale == "ue4m3":
        pool = np.array([(e << 3) | m for e in (5, 6, 7, 8, 9) for m in (0, 4)], np.uint8)
        sa, sb = rng.choice(pool, (M, nb)), rng.choice(pool, (N, nb))
        dec = lambda c: np.array([[2.0 ** (int(x) // 8 - 7) * (1 + (int(x) % 8) / 8) for x in r] for r in c])
    else:
        sa, sb = si.scale_codes(104, M, nb), si.scale_codes(105, N, nb)
        dec = lambda c: np.exp2(c.astype(np.float64) - 127.0)
    D, _ = G.gemm_fp4(M, N, K, si.pack_fp4(ca), si.pack_fp4(cb), sa, sb, block=block, scale=scale)
    table = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    a, b = table[ca], table[cb]
    ref = np.zeros((M, N))
    for blk in range(nb):
        s = slice(block * blk, block * blk + block)
        ref += dec(sa)[:, blk:blk + 1] * (a[:, s] @ b[:, s].T) * dec(sb)[:, blk][None, :]
    assert np.array_equal(D, ref)


def test_fp4_block_size_matters():
    # the same codes read with 16- and 32-element blocks differ once the scales differ per block
    M, N, K = 4, 4, 64
    ca, cb = si.fp4_codes(111, M, K), si.fp4_codes(112, N, K)
    s16 = np.tile(np.array([[0x38, 0x40, 0x38, 0x40]], np.uint8), (M, 1))   # 1, 2, 1, 2 per 16
    D16, _ = G.gemm_fp4(M, N, K, si.pack_fp4(ca), si.pack_fp4(cb), s16, np.tile(s16[:1], (N, 1)), block=16)
    D16u, _ = G.gemm_fp4(M, N, K, si.pack_fp4(ca), si.pack_fp4(cb), np.full((M, 4), 0x38, np.uint8),
                         np.full((N, 4), 0x38, np.uint8), block=16)
    assert not np.array_equal(D16, D16u)


@pytest.mark.parametrize("block,scale", [(16, "ue4m3"), (32, "e8m0")])
def test_fp4_entries_are_the_exact_scaled_product(block, scale):
    # the per-entry form (for sampled checks of large problems) against the exact
    # block-scaled sum written out with numpy, with a padded lda, a K that ends
    # inside a scale block, and beta * C; and equal to the whole-matrix form
    M, N, K, lda = 9, 14, 200, 224
    ca = np.zeros((M, lda), np.uint8)
    ca[:, :K] = si.fp4_codes(121, M, K)
    cb = si.fp4_codes(122, N, K)
    nb = (K + block - 1) // block
    rng = np.random.default_rng(123)
    if scale == "ue4m3":
        pool = np.array([(e << 3) | m for e in (5, 6, 7, 8, 9) for m in (0, 4)], np.uint8)
        sa, sb = rng.choice(pool, (M, nb)), rng.choice(pool, (N, nb))
        dec = lambda c: np.array([[2.0 ** (int(x) // 8 - 7) * (1 + (int(x) % 8) / 8) for x in r] for r in c])
    else:
        sa, sb = si.scale_codes(124, M, nb), si.scale_codes(125, N, nb)
        dec = lambda c: np.exp2(c.astype(np.float64) - 127.0)
    C = (rng.integers(-8, 9, (M, N)) * 0.25).astype(np.float32)
    rows = np.array([0, 8, 3, 5, 8, 0])
    cols = np.array([0, 13, 7, 2, 0, 13])
    A, B = si.pack_fp4(ca), si.pack_fp4(cb)
    D, S = G.gemm_fp4_entries(M, N, K, A, B, sa, sb, rows, cols, block=block, scale=scale, lda=lda, C=C,
                              c_fmt="f32", alpha=0.5, beta=-2.0)
    table = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    a, b = table[ca[:, :K]], table[cb]
    exact = np.zeros((M, N))
    for blk in range(nb):
        s = slice(block * blk, min(K, block * blk + block))
        exact += dec(sa)[:, blk:blk + 1] * (a[:, s] @ b[:, s].T) * dec(sb)[:, blk][None, :]
    ref = 0.5 * exact - 2.0 * C.astype(np.float64)
    assert np.array_equal(D, ref[rows, cols])
    Dfull, Sfull = G.gemm_fp4(M, N, K, A, B, sa, sb, block=block, scale=scale, lda=lda, C=C, c_fmt="f32",
                              alpha=0.5, beta=-2.0)
    assert np.array_equal(D, Dfull[rows, cols]) and np.array_equal(S, Sfull[rows, cols])
