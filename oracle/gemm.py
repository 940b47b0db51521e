"""Python front of the fp64 GEMM oracle (``gemm_oracle.c``).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the CUDA path.

``build()`` compiles the C file with gcc and OpenMP into ``liboracle.so``
next to it; the first call builds it if it is missing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "tf32": 5}
MAJOR = {"K": 0, "MN": 1}


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` (plain -O2, no fast-math) into ``liboracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
                               "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            lib.oracle_gemm.argtypes = [i64, i64, i64, vp, ctypes.c_int, ctypes.c_int, i64,
                                        vp, ctypes.c_int, ctypes.c_int, i64, vp, ctypes.c_int, i64,
                                        ctypes.c_double, ctypes.c_double, dp, dp, ctypes.c_int]
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_gemm_entries.argtypes = [i64, i64, i64, vp, ctypes.c_int, ctypes.c_int, i64,
                                                vp, ctypes.c_int, ctypes.c_int, i64, vp, ctypes.c_int, i64,
                                                ctypes.c_double, ctypes.c_double, i64, vp, vp,
                                                dp, dp, ctypes.c_int]
            lib.oracle_gemm_entries.restype = ctypes.c_int
            lib.oracle_round.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.oracle_round.restype = ctypes.c_double
            lib.oracle_round_bits.argtypes = [dp, i64, ctypes.c_int, vp]
            lib.oracle_round_bits.restype = None
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
            lib.oracle_decode.restype = ctypes.c_double
            lib.oracle_decode_e8m0.argtypes = [ctypes.c_uint8]
            lib.oracle_decode_e8m0.restype = ctypes.c_double
            mx = [i64, i64, i64, vp, ctypes.c_int, ctypes.c_int, i64, vp, i64,
                  vp, ctypes.c_int, ctypes.c_int, i64, vp, i64, vp, ctypes.c_int, i64,
                  ctypes.c_double, ctypes.c_double]
            lib.oracle_gemm_mx.argtypes = mx + [dp, dp, ctypes.c_int]
            lib.oracle_gemm_mx.restype = ctypes.c_int
            lib.oracle_gemm_mx_entries.argtypes = mx + [i64, vp, vp, dp, dp, ctypes.c_int]
            lib.oracle_gemm_mx_entries.restype = ctypes.c_int
            lib.oracle_decode_e2m1.argtypes = [ctypes.c_uint8]
            lib.oracle_decode_e2m1.restype = ctypes.c_double
            lib.oracle_decode_ue4m3.argtypes = [ctypes.c_uint8]
            lib.oracle_decode_ue4m3.restype = ctypes.c_double
            lib.oracle_gemm_fp4.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                            ctypes.c_int, vp, ctypes.c_int, i64, ctypes.c_double, ctypes.c_double,
                                            dp, dp, ctypes.c_int]
            lib.oracle_gemm_fp4.restype = ctypes.c_int
            lib.oracle_gemm_fp4_entries.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                                    ctypes.c_int, vp, ctypes.c_int, i64, ctypes.c_double,
                                                    ctypes.c_double, i64, vp, vp, dp, dp, ctypes.c_int]
            lib.oracle_gemm_fp4_entries.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


def gemm(M, N, K, A, B, *, in_fmt="bf16", b_fmt=None, a_major="K", b_major="K", lda=None, ldb=None,
         C=None, c_fmt="f32", ldc=None, alpha=1.0, beta=0.0, threads=0):
    """Full fp64 product. ``A``, ``B``, ``C`` are bit-pattern arrays in storage layout.

    Returns (D, S): the exact float64 result and the tolerance scale
    |alpha| * sum_k |a_ik b_kj| + |beta c_ij|, both M x N.
    """
    lib = _load()
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    lda = lda if lda is not None else (K if a_major == "K" else M)
    ldb = ldb if ldb is not None else (K if b_major == "K" else N)
    if C is not None:
        C = np.ascontiguousarray(C)
        ldc = ldc if ldc is not None else N
    D = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    rc = lib.oracle_gemm(M, N, K, _ptr(A), FMT[in_fmt], MAJOR[a_major], lda, _ptr(B), FMT[b_fmt or in_fmt],
                         MAJOR[b_major], ldb,
                         _ptr(C), FMT[c_fmt], ldc or 0, float(alpha), float(beta),
                         _ptr(D), _ptr(S), int(threads))
    if rc:
        raise ValueError("oracle_gemm rejected its arguments")
    return D, S


def gemm_entries(M, N, K, A, B, rows, cols, *, in_fmt="bf16", b_fmt=None, a_major="K", b_major="K", lda=None,
                 ldb=None, C=None, c_fmt="f32", ldc=None, alpha=1.0, beta=0.0, threads=0):
    """fp64 result and tolerance scale at the listed (rows[e], cols[e]) entries only."""
    lib = _load()
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    lda = lda if lda is not None else (K if a_major == "K" else M)
    ldb = ldb if ldb is not None else (K if b_major == "K" else N)
    if C is not None:
        C = np.ascontiguousarray(C)
        ldc = ldc if ldc is not None else N
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    D = np.empty(n, dtype=np.float64)
    S = np.empty(n, dtype=np.float64)
    rc = lib.oracle_gemm_entries(M, N, K, _ptr(A), FMT[in_fmt], MAJOR[a_major], lda, _ptr(B),
                                 FMT[b_fmt or in_fmt], MAJOR[b_major], ldb, _ptr(C), FMT[c_fmt], ldc or 0,
                                 float(alpha), float(beta), n, _ptr(rows), _ptr(cols),
                                 _ptr(D), _ptr(S), int(threads))
    if rc:
        raise ValueError("oracle_gemm_entries: entry out of range")
    return D, S


def _mx_common(M, N, K, A, B, SA, SB, a_major, b_major, lda, ldb, C, ldc):
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    SA = np.ascontiguousarray(SA, dtype=np.uint8)
    SB = np.ascontiguousarray(SB, dtype=np.uint8)
    lda = lda if lda is not None else (K if a_major == "K" else M)
    ldb = ldb if ldb is not None else (K if b_major == "K" else N)
    if C is not None:
        C = np.ascontiguousarray(C)
        ldc = ldc if ldc is not None else N
    return A, B, SA, SB, lda, ldb, C, ldc


def gemm_mx(M, N, K, A, B, SA, SB, *, in_fmt="e4m3", b_fmt=None, a_major="K", b_major="K", lda=None, ldb=None,
            C=None, c_fmt="f32", ldc=None, alpha=1.0, beta=0.0, threads=0):
    """Block-scaled (MXFP8) fp64 product; ``SA`` is M x ceil(K/32) and ``SB`` N x ceil(K/32) E8M0 codes.

    Returns (D, S) as ``gemm`` does.
    """
    lib = _load()
    A, B, SA, SB, lda, ldb, C, ldc = _mx_common(M, N, K, A, B, SA, SB, a_major, b_major, lda, ldb, C, ldc)
    D = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    rc = lib.oracle_gemm_mx(M, N, K, _ptr(A), FMT[in_fmt], MAJOR[a_major], lda, _ptr(SA), SA.shape[1],
                            _ptr(B), FMT[b_fmt or in_fmt], MAJOR[b_major], ldb, _ptr(SB), SB.shape[1],
                            _ptr(C), FMT[c_fmt], ldc or 0, float(alpha), float(beta), _ptr(D), _ptr(S),
                            int(threads))
    if rc:
        raise ValueError("oracle_gemm_mx rejected its arguments")
    return D, S


def gemm_mx_entries(M, N, K, A, B, SA, SB, rows, cols, *, in_fmt="e4m3", b_fmt=None, a_major="K", b_major="K",
                    lda=None, ldb=None, C=None, c_fmt="f32", ldc=None, alpha=1.0, beta=0.0, threads=0):
    """The block-scaled product at the listed entries only."""
    lib = _load()
    A, B, SA, SB, lda, ldb, C, ldc = _mx_common(M, N, K, A, B, SA, SB, a_major, b_major, lda, ldb, C, ldc)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    D = np.empty(rows.size, dtype=np.float64)
    S = np.empty(rows.size, dtype=np.float64)
    rc = lib.oracle_gemm_mx_entries(M, N, K, _ptr(A), FMT[in_fmt], MAJOR[a_major], lda, _ptr(SA), SA.shape[1],
                                    _ptr(B), FMT[b_fmt or in_fmt], MAJOR[b_major], ldb, _ptr(SB), SB.shape[1],
                                    _ptr(C), FMT[c_fmt], ldc or 0, float(alpha), float(beta), rows.size,
                                    _ptr(rows), _ptr(cols), _ptr(D), _ptr(S), int(threads))
    if rc:
        raise ValueError("oracle_gemm_mx_entries: bad arguments")
    return D, S


def gemm_fp4(M, N, K, A, B, SA, SB, *, block, scale="ue4m3", lda=None, ldb=None, C=None, c_fmt="f32", ldc=None,
             alpha=1.0, beta=0.0, threads=0):
    """Block-scaled fp4 fp64 product. ``A`` (M x lda/2 bytes) and ``B`` (N x ldb/2 bytes) hold packed E2M1,
    K-major; ``SA`` is M x ceil(K/block) and ``SB`` N x ceil(K/block) scale codes (UE4M3 or E8M0).
    Returns (D, S) as ``gemm`` does."""
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    SA = np.ascontiguousarray(SA, dtype=np.uint8)
    SB = np.ascontiguousarray(SB, dtype=np.uint8)
    lda = lda if lda is not None else K
    ldb = ldb if ldb is not None else K
    if C is not None:
        C = np.ascontiguousarray(C)
        ldc = ldc if ldc is not None else N
    D = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    rc = lib.oracle_gemm_fp4(M, N, K, _ptr(A), lda, _ptr(SA), SA.shape[1], _ptr(B), ldb, _ptr(SB), SB.shape[1],
                             int(block), 1 if scale == "e8m0" else 0, _ptr(C), FMT[c_fmt], ldc or 0, float(alpha),
                             float(beta), _ptr(D), _ptr(S), int(threads))
    if rc:
        raise ValueError("oracle_gemm_fp4 rejected its arguments")
    return D, S


def gemm_fp4_entries(M, N, K, A, B, SA, SB, rows, cols, *, block, scale="ue4m3", lda=None, ldb=None, C=None,
                     c_fmt="f32", ldc=None, alpha=1.0, beta=0.0, threads=0):
    """The block-scaled fp4 product of ``gemm_fp4`` at the listed entries (rows[e], cols[e]) only."""
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    SA = np.ascontiguousarray(SA, dtype=np.uint8)
    SB = np.ascontiguousarray(SB, dtype=np.uint8)
    lda = lda if lda is not None else K
    ldb = ldb if ldb is not None else K
    if C is not None:
        C = np.ascontiguousarray(C)
        ldc = ldc if ldc is not None else N
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    D = np.empty(rows.size, dtype=np.float64)
    S = np.empty(rows.size, dtype=np.float64)
    rc = lib.oracle_gemm_fp4_entries(M, N, K, _ptr(A), lda, _ptr(SA), SA.shape[1], _ptr(B), ldb, _ptr(SB),
                                     SB.shape[1], int(block), 1 if scale == "e8m0" else 0, _ptr(C), FMT[c_fmt],
                                     ldc or 0, float(alpha), float(beta), rows.size, _ptr(rows), _ptr(cols),
                                     _ptr(D), _ptr(S), int(threads))
    if rc:
        raise ValueError("oracle_gemm_fp4_entries: bad arguments")
    return D, S


def decode_e2m1(codes) -> np.ndarray:
    """Values of 4-bit E2M1 codes."""
    lib = _load()
    c = np.asarray(codes).reshape(-1)
    return np.array([lib.oracle_decode_e2m1(int(x)) for x in c], dtype=np.float64).reshape(np.shape(codes))


def decode_ue4m3(codes) -> np.ndarray:
    """Values of UE4M3 scale codes (0x7F: NaN)."""
    lib = _load()
    c = np.asarray(codes).reshape(-1)
    return np.array([lib.oracle_decode_ue4m3(int(x)) for x in c], dtype=np.float64).reshape(np.shape(codes))


def decode_e8m0(codes) -> np.ndarray:
    """Values 2^(e - 127) of E8M0 scale codes (255: NaN)."""
    lib = _load()
    c = np.asarray(codes).reshape(-1)
    return np.array([lib.oracle_decode_e8m0(int(x)) for x in c], dtype=np.float64).reshape(np.shape(codes))


def decode(bits, fmt: str) -> np.ndarray:
    """Exact values of stored bit patterns in format ``fmt``."""
    lib = _load()
    b = np.asarray(bits).reshape(-1)
    return np.array([lib.oracle_decode(FMT[fmt], int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


def round_to(x, fmt: str) -> np.ndarray:
    """Round float64 values to ``fmt`` (ties to even); return float64 values."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    flat, o = x.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        o[i] = lib.oracle_round(float(flat[i]), FMT[fmt])
    return out


def round_bits(x, fmt: str) -> np.ndarray:
    """Round float64 values to ``fmt``; return the storage bit patterns."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint32 if fmt == "f32" else np.uint16)
    lib.oracle_round_bits(_ptr(x), x.size, FMT[fmt], _ptr(out))
    return out


def ulp(x, fmt: str) -> np.ndarray:
    """Spacing of ``fmt`` at |x| (the unit in the last place of the rounded value)."""
    p, emin = {"f16": (11, -14), "bf16": (8, -126), "f32": (24, -126)}[fmt]
    x = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.where(x > 0, np.floor(np.log2(np.where(x > 0, x, 1.0))), emin)
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - (p - 1)).astype(np.int64))


def tolerance(S, ref, out_fmt: str) -> np.ndarray:
    """Parity bound 1e-3 * S + 1 ulp of the output type at the reference value."""
    return 1e-3 * np.asarray(S) + ulp(ref, out_fmt)
