"""Pins of the oracle's TF32 operand reading (fp32 words, low 13 fraction bits dropped).

TF32 keeps the sign, the 8 exponent bits and 10 fraction bits of an fp32
word. The oracle reads a kind::tf32 operand that way (truncation); the GPU
parity tests check the reading on the hardware with inputs whose truncated
and rounded values differ.
"""
import numpy as np

import seeded_inputs as si
from oracle import gemm as og


def _f32_bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def test_tf32_decode_drops_the_low_13_fraction_bits():
    one = 0x3F800000
    cases = {
        one: 1.0,
        one | 0x1FFF: 1.0,                         # every dropped bit set
        one | 0x2000: 1.0 + 2.0 ** -10,            # the lowest kept bit
        one | 0x2000 | 0x1000: 1.0 + 2.0 ** -10,   # above a half: still truncated
        0xBF800000 | 0x6000: -(1.0 + 2.0 ** -10 + 2.0 ** -9),
        0x00000001: 0.0,                           # an fp32 subnormal below the kept bits
    }
    for bits, want in cases.items():
        assert og.decode(np.array([bits], np.uint32), "tf32")[0] == want, hex(bits)


def test_tf32_inputs_from_the_generator_are_representable_and_round_to_nearest():
    bits = si.matrix_bits(3, 64, 64, "normal", "tf32")
    assert bits.dtype == np.uint32 and not (bits & 0x1FFF).any()
    v = si.bits_to_float64(bits, "tf32")
    x = si.logical_values(3, 64, 64, "normal").astype(np.float32).astype(np.float64)
    assert (np.abs(v - x) <= np.abs(x) * 2.0 ** -11 + 1e-45).all()   # half a TF32 unit
    assert np.array_equal(og.decode(bits.reshape(-1), "tf32").reshape(v.shape), v)


def test_tf32_integer_product_is_exact():
    rng = np.random.default_rng(1)
    A = rng.integers(-4, 5, (24, 40)).astype(np.float64)
    B = rng.integers(-4, 5, (40, 16)).astype(np.float64)
    D, _ = og.gemm(24, 16, 40, _f32_bits(A), _f32_bits(B.T), in_fmt="tf32", a_major="K", b_major="K")
    assert np.array_equal(D, A @ B)


def test_tf32_product_uses_the_truncated_operands():
    # A = 1 + 2^-11 + 2^-12 (truncates to 1, would round to 1 + 2^-10), B = 1
    a = np.zeros((1, 8), np.float32)
    b = np.zeros((1, 8), np.float32)
    a[0, 0] = 1.0 + 2.0 ** -11 + 2.0 ** -12
    b[0, 0] = 1.0
    D, _ = og.gemm(1, 1, 8, a.view(np.uint32), b.view(np.uint32), in_fmt="tf32", a_major="K", b_major="K")
    assert D[0, 0] == 1.0
    D32, _ = og.gemm(1, 1, 8, a.view(np.uint32), b.view(np.uint32), in_fmt="f32", a_major="K", b_major="K")
    assert D32[0, 0] == 1.0 + 2.0 ** -11 + 2.0 ** -12
