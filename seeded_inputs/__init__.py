"""Seeded synthetic inputs for the GEMM tests and the benchmark.

This module is shared by the oracle-side checks and the GPU path. It holds
no GEMM arithmetic: it only draws numbers and rounds them to the storage
type, so that both sides read the very same fp16/bf16/fp32 bit patterns.

Generator: counter-based splitmix64. Element ``i`` of stream ``seed`` is
``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)`` where ``mix`` is the splitmix64
finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014). Index ``i`` is the row-major position of the
element in the *logical* matrix (A is M x K, B is K x N, C is M x N), so
the same logical matrix comes out whatever its storage major-ness.

Distributions:

* ``"uniform"``: ``2u - 1`` with ``u = (z >> 40) / 2**24``, i.e. [-1, 1).
* ``"int4"``: ``((z >> 32) % 9) - 4``, integers in [-4, 4].
* ``"normal"``: Box-Muller on consecutive pairs ``(z_2j, z_2j+1)``, times
  ``scale``.

Rounding to the storage type is round-to-nearest-even: fp16 through
numpy's correctly rounded float64 -> float16 cast; bf16 from the float32
value by rounding its low 16 bits away (ties to even).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "splitmix64",
    "logical_values",
    "matrix_bits",
    "to_storage",
    "bits_to_float64",
    "torch_from_bits",
]

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Return ``count`` uint64 draws of stream ``seed`` from counter ``start``."""
    i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _draw(seed: int, dist: str, start: int, count: int, scale: float) -> np.ndarray:
    if dist == "uniform":
        z = splitmix64(seed, start, count)
        u = (z >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))
        return (2.0 * u - 1.0) * scale
    if dist == "int4":
        z = splitmix64(seed, start, count)
        return (((z >> np.uint64(32)) % np.uint64(9)).astype(np.int64) - 4).astype(np.float64) * scale
    if dist == "normal":
        # pairs (2j, 2j+1) share one Box-Muller transform
        first = start - (start & 1)
        n_pairs = (start + count - first + 1) // 2
        z = splitmix64(seed, first, 2 * n_pairs)
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / (1 << 53))
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))
        r = np.sqrt(-2.0 * np.log(u1))
        out = np.empty(2 * n_pairs, dtype=np.float64)
        out[0::2] = r * np.cos(2.0 * np.pi * u2)
        out[1::2] = r * np.sin(2.0 * np.pi * u2)
        off = start - first
        return out[off:off + count] * scale
    if dist == "zeros":
        return np.zeros(count, dtype=np.float64)
    raise ValueError(f"unknown distribution {dist!r}")


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to ``dtype`` ('f16', 'bf16', 'f32', 'tf32', 'e4m3', 'e5m2'); return the bits.

    fp8 rounding (ties to even, through float32) uses PyTorch's float8_e4m3fn and
    float8_e5m2 conversions; the inputs stay far inside both formats' ranges.
    """
    if dtype in ("e4m3", "e5m2"):
        import torch
        tdt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(tdt)
        return t.view(torch.uint8).numpy().copy()
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "f32":
        return x.astype(np.float32).view(np.uint32)
    if dtype == "tf32":
        # fp32 words holding values representable in TF32 (10 fraction bits): round the
        # fp32 value to nearest-even at fraction bit 10 and clear the 13 bits below it
        b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
        b = (b + np.uint64(0xFFF) + ((b >> np.uint64(13)) & np.uint64(1))) & np.uint64(0xFFFFE000)
        return b.astype(np.uint32)
    if dtype == "bf16":
        b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
        b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
        return b.astype(np.uint16)
    raise ValueError(f"unknown storage type {dtype!r}")


def logical_values(seed: int, rows: int, cols: int, dist: str, scale: float = 1.0) -> np.ndarray:
    """float64 values of the logical ``rows x cols`` matrix (before rounding)."""
    n = rows * cols
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = _draw(seed, dist, s, c, scale)
    return out.reshape(rows, cols)


def matrix_bits(seed: int, rows: int, cols: int, dist: str, dtype: str,
                scale: float = 1.0, transpose: bool = False, ld: int | None = None) -> np.ndarray:
    """Bit patterns of a seeded logical ``rows x cols`` matrix in storage type ``dtype``.

    ``transpose=False`` stores it row-major (``[r * ld + c]``); ``transpose=True``
    stores its transpose row-major (``[c * ld + r]``), i.e. column-major.
    ``ld`` (>= the stored row length) pads each stored row; pads are zero.
    The result is a 2-D array of the stored shape (with the padding columns).
    """
    n = rows * cols
    bits_dtype = np.uint32 if dtype in ("f32", "tf32") else (np.uint8 if dtype in ("e4m3", "e5m2") else np.uint16)
    flat = np.empty(n, dtype=bits_dtype)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        flat[s:s + c] = to_storage(_draw(seed, dist, s, c, scale), dtype)
    mat = flat.reshape(rows, cols)
    if transpose:
        mat = np.ascontiguousarray(mat.T)
    srows, scols = mat.shape
    if ld is None or ld == scols:
        return mat
    if ld < scols:
        raise ValueError("ld smaller than the stored row length")
    padded = np.zeros((srows, ld), dtype=bits_dtype)
    padded[:, :scols] = mat
    return padded


def bits_to_float64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored bit patterns (for building expected tables)."""
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype in ("f32", "tf32"):
        return bits.view(np.float32).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype in ("e4m3", "e5m2"):
        import torch
        tdt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).view(tdt).double().numpy()
    raise ValueError(dtype)


def torch_from_bits(bits: np.ndarray, dtype: str):
    """Wrap bit patterns as a CPU torch tensor of the matching dtype (no copy of values)."""
    import torch
    b = np.ascontiguousarray(bits)
    if dtype in ("f16", "bf16"):
        t = torch.from_numpy(b.view(np.int16))
        return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    if dtype in ("f32", "tf32"):
        return torch.from_numpy(b.view(np.int32)).view(torch.float32)
    if dtype in ("e4m3", "e5m2"):
        return torch.from_numpy(b.view(np.uint8))  # raw bytes; the library reads them as fp8
    raise ValueError(dtype)


def scale_codes(seed: int, rows: int, nblocks: int, lo: int = 124, hi: int = 130) -> np.ndarray:
    """Seeded E8M0 scale codes, ``rows x nblocks`` uint8, uniform in [lo, hi]."""
    z = splitmix64(seed, 0, rows * nblocks)
    span = np.uint64(hi - lo + 1)
    return ((z >> np.uint64(32)) % span + np.uint64(lo)).astype(np.uint8).reshape(rows, nblocks)


def fp4_codes(seed: int, rows: int, cols: int) -> np.ndarray:
    """Seeded 4-bit E2M1 codes, ``rows x cols`` uint8 in [0, 15] (all sixteen codes)."""
    z = splitmix64(seed, 0, rows * cols)
    return ((z >> np.uint64(32)) % np.uint64(16)).astype(np.uint8).reshape(rows, cols)


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes two to a byte along each row: element 2i in the low nibble of byte i."""
    codes = np.asarray(codes, dtype=np.uint8)
    if codes.shape[1] % 2:
        codes = np.concatenate([codes, np.zeros((codes.shape[0], 1), np.uint8)], axis=1)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def mx_scale_atoms(codes: np.ndarray, rows: int, K: int, block: int = 32, fill: int = 127) -> np.ndarray:
    """Arrange row-major scale codes (``rows x ceil(K/block)``) in the 512-byte atoms of the
    block-scaled GEMM's ABI: atom (r // 128) * ceil(K/(4 block)) + k // (4 block), byte
    16 * (r % 32) + 4 * ((r % 128) // 32) + (k // block) % 4. Unused entries hold ``fill``
    (127 is 1.0 as E8M0; UE4M3 needs 0x38 for 1.0, its 0x7F being NaN)."""
    nb = (K + block - 1) // block
    groups = (nb + 3) // 4
    blocks = (rows + 127) // 128
    out = np.full(blocks * groups * 512, fill, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    idx = ((r // 128) * groups + b // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4
    out[idx.reshape(-1)] = codes[:rows, :nb].reshape(-1)
    return out
