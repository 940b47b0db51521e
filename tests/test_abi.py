"""Host-side checks of the C ABI: the library loads without a GPU, exports every
function the header declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gemm_gb300.h")


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(gemm_[a-z0-9_]+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = _declared_functions()
    for must in ("gemm_bf16", "gemm_f16", "gemm_bf16_grouped", "gemm_f16_grouped",
                 "gemm_grouped_workspace_size", "gemm_last_device_status", "gemm_status_string"):
        assert must in names


def test_library_exports_every_declared_function(g):
    lib = ctypes.CDLL(g.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(g.EXPORTED)


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "gemm_gb300.h"\nint main(void){return (int)GEMM_OK;}\n')
    import subprocess
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                           "-c", str(src), "-o", str(tmp_path / "t.o")])


def test_status_strings(g):
    for s in range(6):
        assert g.gemm_status_string(s)
    assert g.gemm_status_string(99) == "unknown status"


def test_workspace_size(g):
    assert g.gemm_grouped_workspace_size(0) == 0
    n = 64
    size = g.gemm_grouped_workspace_size(n)
    assert size >= n * 4 * 128 and size % 128 == 0


@pytest.mark.parametrize("case,expect", [
    (dict(M=-1), "ERR_INVALID_ARG"),
    (dict(K=-5), "ERR_INVALID_ARG"),
    (dict(A=0x1008), "ERR_ALIGNMENT"),          # 8-byte aligned only
    (dict(lda=36), "ERR_ALIGNMENT"),            # 72 B row stride: not a multiple of 16 B
    (dict(lda=16), "ERR_INVALID_ARG"),          # shorter than K
    (dict(ldd=66), "ERR_ALIGNMENT"),            # fp32 row of 264 B
    (dict(D=0), "ERR_INVALID_ARG"),
    (dict(beta=1.0, C=0), "ERR_INVALID_ARG"),
    (dict(a_major=7), "ERR_INVALID_ARG"),
    (dict(d_type=9), "ERR_INVALID_ARG"),
])
def test_validation_happens_before_any_cuda_call(g, case, expect):
    args = dict(M=64, N=64, K=32, A=0x1000, a_major=0, lda=32, B=0x2000, b_major=0, ldb=32,
                C=0, ldc=64, D=0x3000, ldd=64, d_type=0, alpha=1.0, beta=0.0)
    args.update(case)
    with pytest.raises(g.GemmError) as ei:
        g.gemm_bf16(**args, stream=0)
    assert ei.value.status == getattr(g, expect)


def test_empty_problem_is_a_no_op(g):
    g.gemm_bf16(0, 64, 32, 0x1000, 0, 32, 0x2000, 0, 32, 0, 64, 0x3000, 64, 0, 1.0, 0.0, stream=0)
    g.gemm_bf16(64, 0, 32, 0x1000, 0, 32, 0x2000, 0, 32, 0, 64, 0x3000, 64, 0, 1.0, 0.0, stream=0)


def test_bad_options_rejected(g):
    import smem_swizzle_layouts_gb300 as gg
    # option checks run after the device query; on a CPU-only host that query fails first,
    # so only the enum range checks that precede it are exercised here
    with pytest.raises(gg.GemmError) as ei:
        gg.gemm_ex(5, 64, 64, 32, 0x1000, 0, 32, 0x2000, 0, 32, 0, 64, 0x3000, 64, 0, 1.0, 0.0, stream=0)
    assert ei.value.status == gg.ERR_INVALID_ARG


def test_grouped_argument_checks(g):
    with pytest.raises(g.GemmError) as ei:
        g.gemm_bf16_grouped([dict(M=64, N=64, K=32, A=0x1000, B=0x2000, D=0x3000, lda=32, ldb=32, ldd=64)],
                            0, 0, 0, 1.0, 0.0, 0, 0, stream=0)
    assert ei.value.status == g.ERR_INVALID_ARG            # no workspace
    g.gemm_bf16_grouped([], 0, 0, 0, 1.0, 0.0, 0, 0, stream=0)   # nothing to do


def test_package_has_no_cpu_fallback():
    src = open(os.path.join(ROOT, "smem_swizzle_layouts_gb300", "_lib.py")).read()
    src += open(os.path.join(ROOT, "smem_swizzle_layouts_gb300", "__init__.py")).read()
    assert "oracle" not in src and "torch.matmul" not in src and "@" not in src.replace("@pytest", "")
