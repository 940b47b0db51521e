"""ctypes binding of ``libgemm_gb300.so`` (argument marshalling only).

The names mirror the C ABI in ``include/gemm_gb300.h``. Tensor arguments may
be torch tensors (their ``data_ptr()`` is passed) or plain integers
(addresses). ``stream`` may be a ``torch.cuda.Stream``, an integer handle or
None (torch's current stream). Every non-OK status raises ``GemmError``.
There is no fallback: if the library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgemm_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python smem_swizzle_layouts_gb300/build.py` "
        "(or __graft_entry__.build()); there is no CPU fallback")

_lib = ctypes.CDLL(LIB_PATH)

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(6)
K_MAJOR, MN_MAJOR = 0, 1
OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2
FP8_E4M3, FP8_E5M2 = 0, 1
FP4_NVFP4, FP4_MXFP4 = 0, 1
SWIZZLE_AUTO, SWIZZLE_32B, SWIZZLE_64B, SWIZZLE_128B, SWIZZLE_NONE, SWIZZLE_128B_ATOM32 = 0, 1, 2, 3, 4, 5

_i64, _vp, _f, _int, _u32, _u64 = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int,
                                   ctypes.c_uint32, ctypes.c_uint64)


class GemmOptions(ctypes.Structure):
    _fields_ = [("cta_group", _int), ("tile_m", _int), ("tile_n", _int), ("block_k", _int), ("swizzle_a", _int), ("swizzle_b", _int),
                ("epilogue_swizzle", _int), ("max_ctas", _int), ("group_m", _int),
                ("timeout_ms", _int), ("flags", _int), ("stats", _vp),
                ("stream_k", _int), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("mma_ws", _int),
                ("multicast_b", _int)]


class GemmProblem(ctypes.Structure):
    _fields_ = [("M", _i64), ("N", _i64), ("K", _i64), ("A", _vp), ("B", _vp), ("C", _vp),
                ("D", _vp), ("lda", _i64), ("ldb", _i64), ("ldc", _i64), ("ldd", _i64)]


_single = [_i64, _i64, _i64, _vp, _int, _i64, _vp, _int, _i64, _vp, _i64, _vp, _i64, _int, _f, _f, _vp]
_lib.gemm_bf16.argtypes = _single
_lib.gemm_f16.argtypes = _single
_lib.gemm_ex.argtypes = [_int] + _single[:-1] + [ctypes.POINTER(GemmOptions), _vp]
_fp8 = [_i64, _i64, _i64, _vp, _int, _int, _i64, _vp, _int, _int, _i64, _vp, _i64, _vp, _i64, _int, _f, _f]
_lib.gemm_fp8.argtypes = _fp8 + [_vp]
_lib.gemm_fp8_ex.argtypes = _fp8 + [ctypes.POINTER(GemmOptions), _vp]
_lib.gemm_mxfp8.argtypes = [_i64, _i64, _i64, _vp, _int, _int, _i64, _vp, _vp, _int, _int, _i64, _vp, _vp, _i64, _vp,
                            _i64, _int, _f, _f, ctypes.POINTER(GemmOptions), _vp]
_lib.gemm_fp4.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _vp, _int, _vp, _i64, _vp, _i64, _int, _f,
                          _f, ctypes.POINTER(GemmOptions), _vp]
_lib.gemm_fp4_scale_bytes.argtypes = [_i64, _i64, _int]
_lib.gemm_fp4_scale_bytes.restype = ctypes.c_size_t
_lib.gemm_mx_scale_bytes.argtypes = [_i64, _i64]
_lib.gemm_mx_scale_bytes.restype = ctypes.c_size_t
_grouped = [ctypes.POINTER(GemmProblem), _int, _int, _int, _int, _f, _f, _vp, ctypes.c_size_t, _vp]
_lib.gemm_bf16_grouped.argtypes = _grouped
_lib.gemm_f16_grouped.argtypes = _grouped
_lib.gemm_grouped_ex.argtypes = [_int] + _grouped[:-1] + [ctypes.POINTER(GemmOptions), _vp]
_lib.gemm_bf16_grouped_noalloc.argtypes = [ctypes.POINTER(GemmProblem), _int, _int, _int, _int, _f, _f, _vp]
_lib.gemm_grouped_workspace_size.argtypes = [_int]
_lib.gemm_grouped_workspace_size.restype = ctypes.c_size_t
_lib.gemm_streamk_workspace_size.argtypes = []
_lib.gemm_streamk_workspace_size.restype = ctypes.c_size_t
_lib.gemm_last_device_status.argtypes = [_vp, ctypes.POINTER(_u32)]
_lib.gemm_status_string.argtypes = [_int]
_lib.gemm_status_string.restype = ctypes.c_char_p
_lib.gemm_launch_count.restype = _u64
_lib.gemm_debug_descriptors.argtypes = [_int, _int, _int, _int, _u32, _int, _int, _int, _int, _int, _int,
                                        _vp, _vp]
_lib.gemm_debug_stage_image.argtypes = [_vp, _int, _int, _i64, _i64, _i64, _int, _int, _i64, _i64, _vp, _vp]
_lib.gemm_debug_plan.argtypes = [_i64, _i64, _i64, _int, _int, _int, _int, ctypes.POINTER(GemmOptions), _int,
                                 ctypes.POINTER(ctypes.c_int32)]
_lib.gemm_debug_plan.restype = _int
_lib.gemm_debug_streamk_units.argtypes = [_int, _i64, _int, _int, _int, ctypes.POINTER(ctypes.c_int32), _int]
_lib.gemm_debug_streamk_units.restype = _int
_lib.gemm_debug_inject_timeout.argtypes = [_int]
_lib.gemm_debug_inject_timeout.restype = None
_lib.gemm_debug_inject_timeout_at.argtypes = [_int, _int]
_lib.gemm_debug_inject_timeout_at.restype = None
for _name in ("gemm_bf16", "gemm_f16", "gemm_ex", "gemm_fp8", "gemm_fp8_ex", "gemm_mxfp8", "gemm_fp4", "gemm_bf16_grouped",
              "gemm_f16_grouped",
              "gemm_bf16_grouped_noalloc",
              "gemm_last_device_status", "gemm_debug_descriptors", "gemm_debug_stage_image"):
    getattr(_lib, _name).restype = _int

EXPORTED = ("gemm_bf16", "gemm_f16", "gemm_ex", "gemm_fp8", "gemm_fp8_ex", "gemm_mxfp8", "gemm_mx_scale_bytes",
            "gemm_fp4", "gemm_fp4_scale_bytes",
            "gemm_streamk_workspace_size",
            "gemm_grouped_workspace_size",
            "gemm_bf16_grouped", "gemm_grouped_ex",
            "gemm_f16_grouped", "gemm_bf16_grouped_noalloc", "gemm_last_device_status", "gemm_status_string", "gemm_launch_count",
            "gemm_debug_descriptors", "gemm_debug_stage_image", "gemm_debug_plan", "gemm_debug_streamk_units",
            "gemm_debug_inject_timeout", "gemm_debug_inject_timeout_at")


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_status_string(status)} (status {status})")


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> None:
    if status != OK:
        raise GemmError(status, where)


def _opts(options) -> ctypes.POINTER(GemmOptions) | None:
    if options is None:
        return None
    if isinstance(options, GemmOptions):
        return ctypes.pointer(options)
    opts = dict(options)
    if "stats" in opts:
        opts["stats"] = _addr(opts["stats"])
    if "workspace" in opts:
        ws = opts["workspace"]
        opts["workspace"] = _addr(ws)
        if "workspace_bytes" not in opts and ws is not None and not isinstance(ws, int):
            opts["workspace_bytes"] = ws.numel() * ws.element_size()
    return ctypes.pointer(GemmOptions(**opts))


def gemm_status_string(status: int) -> str:
    return _lib.gemm_status_string(status).decode()


def gemm_launch_count() -> int:
    return int(_lib.gemm_launch_count())


def gemm_bf16(M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd, d_type, alpha, beta, stream=None):
    _check(_lib.gemm_bf16(M, N, K, _addr(A), a_major, lda, _addr(B), b_major, ldb, _addr(C), ldc,
                          _addr(D), ldd, d_type, alpha, beta, _stream(stream)), "gemm_bf16")


def gemm_f16(M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd, d_type, alpha, beta, stream=None):
    _check(_lib.gemm_f16(M, N, K, _addr(A), a_major, lda, _addr(B), b_major, ldb, _addr(C), ldc,
                         _addr(D), ldd, d_type, alpha, beta, _stream(stream)), "gemm_f16")


def gemm_ex(in_type, M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd, d_type, alpha, beta,
            options=None, stream=None):
    _check(_lib.gemm_ex(in_type, M, N, K, _addr(A), a_major, lda, _addr(B), b_major, ldb, _addr(C), ldc,
                        _addr(D), ldd, d_type, alpha, beta, _opts(options), _stream(stream)), "gemm_ex")


class GemmCall:
    """gemm_ex with its arguments marshalled once, for repeated launches on the same buffers.

    Calling the object launches the GEMM again; it converts nothing per call.
    """

    def __init__(self, in_type, M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd, d_type, alpha, beta,
                 options=None, stream=None, fp8=None, scales=None, fp4=None):
        """``in_type`` 0 fp16 / 1 bf16; or ``fp8=(a_format, b_format)`` for gemm_fp8_ex, plus
        ``scales=(SFA, SFB)`` for the block-scaled gemm_mxfp8; or ``fp4=kind`` with ``scales``
        for gemm_fp4 (majors ignored: K-major)."""
        self._opts_ref = _opts(options)  # keeps the options struct alive
        tail = (_vp(_addr(C)), _i64(ldc), _vp(_addr(D)), _i64(ldd), _int(d_type), _f(alpha), _f(beta),
                self._opts_ref, _vp(_stream(stream)))
        if fp4 is not None:
            self._args = (_i64(M), _i64(N), _i64(K), _vp(_addr(A)), _i64(lda), _vp(_addr(scales[0])),
                          _vp(_addr(B)), _i64(ldb), _vp(_addr(scales[1])), _int(fp4)) + tail
            self._fn = _lib.gemm_fp4
        elif scales is not None:
            self._args = (_i64(M), _i64(N), _i64(K), _vp(_addr(A)), _int(fp8[0]), _int(a_major), _i64(lda),
                          _vp(_addr(scales[0])), _vp(_addr(B)), _int(fp8[1]), _int(b_major), _i64(ldb),
                          _vp(_addr(scales[1]))) + tail
            self._fn = _lib.gemm_mxfp8
        elif fp8 is not None:
            self._args = (_i64(M), _i64(N), _i64(K), _vp(_addr(A)), _int(fp8[0]), _int(a_major), _i64(lda),
                          _vp(_addr(B)), _int(fp8[1]), _int(b_major), _i64(ldb)) + tail
            self._fn = _lib.gemm_fp8_ex
        else:
            self._args = (_int(in_type), _i64(M), _i64(N), _i64(K), _vp(_addr(A)), _int(a_major), _i64(lda),
                          _vp(_addr(B)), _int(b_major), _i64(ldb)) + tail
            self._fn = _lib.gemm_ex

    def __call__(self):
        st = self._fn(*self._args)
        if st != OK:
            raise GemmError(st, self._fn.__name__)


def gemm_fp8(M, N, K, A, a_format, a_major, lda, B, b_format, b_major, ldb, C, ldc, D, ldd, d_type, alpha, beta,
             stream=None):
    _check(_lib.gemm_fp8(M, N, K, _addr(A), a_format, a_major, lda, _addr(B), b_format, b_major, ldb, _addr(C),
                         ldc, _addr(D), ldd, d_type, alpha, beta, _stream(stream)), "gemm_fp8")


def gemm_fp8_ex(M, N, K, A, a_format, a_major, lda, B, b_format, b_major, ldb, C, ldc, D, ldd, d_type, alpha,
                beta, options=None, stream=None):
    _check(_lib.gemm_fp8_ex(M, N, K, _addr(A), a_format, a_major, lda, _addr(B), b_format, b_major, ldb,
                            _addr(C), ldc, _addr(D), ldd, d_type, alpha, beta, _opts(options), _stream(stream)),
           "gemm_fp8_ex")


def gemm_mxfp8(M, N, K, A, a_format, a_major, lda, SFA, B, b_format, b_major, ldb, SFB, C, ldc, D, ldd, d_type,
               alpha, beta, options=None, stream=None):
    _check(_lib.gemm_mxfp8(M, N, K, _addr(A), a_format, a_major, lda, _addr(SFA), _addr(B), b_format, b_major, ldb,
                           _addr(SFB), _addr(C), ldc, _addr(D), ldd, d_type, alpha, beta, _opts(options),
                           _stream(stream)), "gemm_mxfp8")


def gemm_fp4(M, N, K, A, lda, SFA, B, ldb, SFB, kind, C, ldc, D, ldd, d_type, alpha, beta, options=None,
             stream=None):
    _check(_lib.gemm_fp4(M, N, K, _addr(A), lda, _addr(SFA), _addr(B), ldb, _addr(SFB), kind, _addr(C), ldc,
                         _addr(D), ldd, d_type, alpha, beta, _opts(options), _stream(stream)), "gemm_fp4")


def gemm_fp4_scale_bytes(rows: int, K: int, kind: int) -> int:
    return int(_lib.gemm_fp4_scale_bytes(rows, K, kind))


def gemm_mx_scale_bytes(rows: int, K: int) -> int:
    return int(_lib.gemm_mx_scale_bytes(rows, K))


PLAN_FIELDS = ("cta_group", "tile_n", "block_k", "tile_m", "swizzle_a", "swizzle_b", "epilogue_swizzle", "group_m",
               "mma_ws", "multicast_b")


def gemm_debug_plan(M, N, K, kind=0, a_major=0, b_major=0, grouped=False, options=None, sms=148):
    """The tile plan a call would launch (host only), as a dict; raises GemmError for rejected options."""
    out = (ctypes.c_int32 * 10)()
    _check(_lib.gemm_debug_plan(M, N, K, kind, a_major, b_major, int(grouped), _opts(options), sms, out),
           "gemm_debug_plan")
    return dict(zip(PLAN_FIELDS, list(out)))


def gemm_debug_streamk_units(mode, tiles, clusters, kb_per_tile, cluster):
    """The stream-K units of one cluster as (tile, kb0, kb1, kind, c_lo, c_hi) tuples, or None when unsplit."""
    n = _lib.gemm_debug_streamk_units(mode, tiles, clusters, kb_per_tile, cluster, None, 0)
    if n < 0:
        return None
    buf = (ctypes.c_int32 * (6 * max(n, 1)))()
    _lib.gemm_debug_streamk_units(mode, tiles, clusters, kb_per_tile, cluster, buf, n)
    return [tuple(buf[6 * i:6 * i + 6]) for i in range(n)]


def gemm_streamk_workspace_size() -> int:
    """Bytes of stream-K workspace for any single GEMM on the current device."""
    return int(_lib.gemm_streamk_workspace_size())


def gemm_grouped_workspace_size(num_problems: int) -> int:
    return int(_lib.gemm_grouped_workspace_size(num_problems))


def _problem_array(problems):
    arr = (GemmProblem * len(problems))()
    for i, q in enumerate(problems):
        arr[i] = GemmProblem(q["M"], q["N"], q["K"], _addr(q.get("A")), _addr(q.get("B")),
                             _addr(q.get("C")), _addr(q.get("D")), q["lda"], q["ldb"], q.get("ldc", 0),
                             q["ldd"])
    return arr


def gemm_bf16_grouped(problems, a_major, b_major, d_type, alpha, beta, workspace, workspace_bytes,
                      stream=None):
    arr = _problem_array(problems)
    _check(_lib.gemm_bf16_grouped(arr, len(problems), a_major, b_major, d_type, alpha, beta,
                                  _addr(workspace), workspace_bytes, _stream(stream)), "gemm_bf16_grouped")


def gemm_f16_grouped(problems, a_major, b_major, d_type, alpha, beta, workspace, workspace_bytes,
                     stream=None):
    arr = _problem_array(problems)
    _check(_lib.gemm_f16_grouped(arr, len(problems), a_major, b_major, d_type, alpha, beta,
                                 _addr(workspace), workspace_bytes, _stream(stream)), "gemm_f16_grouped")


def gemm_grouped_ex(in_type, problems, a_major, b_major, d_type, alpha, beta, workspace, workspace_bytes,
                    options=None, stream=None):
    arr = _problem_array(problems)
    _check(_lib.gemm_grouped_ex(in_type, arr, len(problems), a_major, b_major, d_type, alpha, beta,
                                _addr(workspace), workspace_bytes, _opts(options), _stream(stream)),
           "gemm_grouped_ex")


NOALLOC_MAX_PROBLEMS = 128


def gemm_bf16_grouped_noalloc(problems, a_major, b_major, d_type, alpha, beta, stream=None):
    """Grouped bf16 GEMM whose table lives in the library's fixed scratch (no allocation)."""
    arr = _problem_array(problems)
    _check(_lib.gemm_bf16_grouped_noalloc(arr, len(problems), a_major, b_major, d_type, alpha, beta,
                                          _stream(stream)), "gemm_bf16_grouped_noalloc")


def gemm_last_device_status(stream=None) -> tuple[int, int]:
    """(status, raw status word); clears the word."""
    detail = _u32(0)
    st = _lib.gemm_last_device_status(_stream(stream), ctypes.byref(detail))
    return st, int(detail.value)


def gemm_debug_descriptors(major, swizzle, rows, bk, stage_addr, n_slices, cta_group, tile_n, in_type,
                           a_major, b_major, out, stream=None):
    _check(_lib.gemm_debug_descriptors(major, swizzle, rows, bk, stage_addr, n_slices, cta_group, tile_n,
                                       in_type, a_major, b_major, _addr(out), _stream(stream)),
           "gemm_debug_descriptors")


def gemm_debug_stage_image(src, major, swizzle, rows_total, k_total, ld, rows, bk, mn0, k0, out, stream=None):
    _check(_lib.gemm_debug_stage_image(_addr(src), major, swizzle, rows_total, k_total, ld, rows, bk, mn0, k0,
                                       _addr(out), _stream(stream)), "gemm_debug_stage_image")


def gemm_debug_inject_timeout(timeout_ms: int, role: int = 2) -> None:
    """Make the next launch's MMA issuer (role 2) or producer (role 1) wait until `timeout_ms` runs out."""
    _lib.gemm_debug_inject_timeout_at(timeout_ms, role)
