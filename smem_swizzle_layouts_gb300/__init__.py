"""GB300 (sm_103a) tcgen05 GEMM: D = alpha * A * B + beta * C.

The compute path is the CUDA library ``libgemm_gb300.so`` (C ABI in
``include/gemm_gb300.h``); this package only marshals arguments to it.
PyTorch is used for device memory and streams. Importing the package fails
loudly if the library has not been built: there is no CPU fallback.
"""
from __future__ import annotations

from ._lib import (  # noqa: F401
    ERR_ALIGNMENT, ERR_CUDA, ERR_INVALID_ARG, FP4_MXFP4, FP4_NVFP4, FP8_E4M3, FP8_E5M2, ERR_TIMEOUT, ERR_UNSUPPORTED, EXPORTED, K_MAJOR, LIB_PATH,
    MN_MAJOR, NOALLOC_MAX_PROBLEMS, OK, OUT_BF16, OUT_F16, OUT_F32, SWIZZLE_128B, SWIZZLE_128B_ATOM32, SWIZZLE_32B, SWIZZLE_64B, SWIZZLE_AUTO, SWIZZLE_NONE,
    GemmCall, GemmError, GemmOptions, GemmProblem, gemm_bf16, gemm_bf16_grouped, gemm_bf16_grouped_noalloc, gemm_debug_descriptors,
    gemm_debug_inject_timeout, gemm_debug_stage_image, gemm_debug_streamk_units, gemm_ex, gemm_f16, gemm_f16_grouped, gemm_fp4, gemm_fp4_scale_bytes, gemm_fp8, gemm_fp8_ex,
    gemm_grouped_ex, gemm_grouped_workspace_size, gemm_mx_scale_bytes, gemm_mxfp8, gemm_streamk_workspace_size, gemm_last_device_status, gemm_launch_count, gemm_status_string,
)

_OUT = {"f32": OUT_F32, "bf16": OUT_BF16, "f16": OUT_F16}
_MAJ = {"K": K_MAJOR, "MN": MN_MAJOR}


def gemm(A, B, D, *, M, N, K, a_major="K", b_major="K", C=None, alpha=1.0, beta=0.0, out="f32",
         options=None, stream=None):
    """Run one GEMM on torch tensors already on the GPU.

    ``A``/``B`` are 2-D fp16 or bf16 tensors in storage layout (K-major A is
    M x lda with K contiguous, MN-major A is K x lda with M contiguous; B
    likewise with N). ``D`` (and ``C``) are row-major M x ldd tensors of the
    output type. Leading dimensions are the tensors' row strides.
    """
    import torch
    in_type = 1 if A.dtype == torch.bfloat16 else 0
    if A.dtype not in (torch.bfloat16, torch.float16) or B.dtype != A.dtype:
        raise TypeError("A and B must both be bf16 or both fp16")
    ldc = C.stride(0) if C is not None else 0
    gemm_ex(in_type, M, N, K, A, _MAJ[a_major], A.stride(0), B, _MAJ[b_major], B.stride(0), C, ldc,
            D, D.stride(0), _OUT[out], alpha, beta, options=options, stream=stream)
    return D
