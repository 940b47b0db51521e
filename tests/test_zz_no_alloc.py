"""The grouped GEMM entry point that allocates nothing (gemm_bf16_grouped_noalloc).

It exists for callers that cannot allocate device memory when they launch a
GEMM: programs whose allocator has reserved the whole device, plug-ins that
a host runtime hands only their input and output buffers, and real-time
loops that may not block in the driver's allocator. Its problem table lives
in a fixed array inside the library instead of a caller workspace. This file
is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.

Both calls below go through the C ABI. Each result is checked element by
element against the fp64 oracle's D on the same inputs, and against the
workspace-taking entry point, within the parity tolerance
(1e-3 * sum_k |a_ik b_kj| (+ |beta c_ij|) + 1 ulp of the output type).
"""
import numpy as np
import pytest

import seeded_inputs as si
from oracle import gemm as og

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import smem_swizzle_layouts_gb300 as g
    return g


def _problems(Ms, N, K, seed, beta):
    host, dev = [], []
    ldd = (N + 7) // 8 * 8
    for i, M in enumerate(Ms):
        A = si.matrix_bits(seed + 3 * i, M, K, "uniform", "bf16")                   # K-major A
        B = si.matrix_bits(seed + 3 * i + 1, K, N, "uniform", "bf16", transpose=True)  # K-major B
        C = si.matrix_bits(seed + 3 * i + 2, M, N, "uniform", "bf16", ld=ldd) if beta else None
        At = si.torch_from_bits(A, "bf16").to(DEV)
        Bt = si.torch_from_bits(B, "bf16").to(DEV)
        Ct = si.torch_from_bits(C, "bf16").to(DEV) if C is not None else None
        host.append((M, A, B, C))
        dev.append(dict(M=M, N=N, K=K, A=At, B=Bt, C=Ct, lda=K, ldb=K, ldc=ldd if beta else 0, ldd=ldd))
    return host, dev


def _outputs(dev_probs, N):
    outs = []
    for q in dev_probs:
        D = torch.full((max(q["M"], 1), q["ldd"]), float("nan"), dtype=torch.bfloat16, device=DEV)
        outs.append(D)
    return [dict(q, D=D) for q, D in zip(dev_probs, outs)], outs


def _bits(D):
    return D.cpu().view(torch.int16).numpy().view(np.uint16)


def _one_round(g, Ms, N, K, seed, alpha, beta):
    host, dev = _problems(Ms, N, K, seed, beta)
    # the existing entry point, with a caller workspace
    ref_probs, ref_out = _outputs(dev, N)
    ws_bytes = g.gemm_grouped_workspace_size(len(Ms))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    g.gemm_bf16_grouped(ref_probs, g.K_MAJOR, g.K_MAJOR, g.OUT_BF16, alpha, beta, ws, ws_bytes)
    # the entry point without allocation
    new_probs, new_out = _outputs(dev, N)
    g.gemm_bf16_grouped_noalloc(new_probs, g.K_MAJOR, g.K_MAJOR, g.OUT_BF16, alpha, beta)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, hex(word)
    for (M, A, B, C), Dr, Dn in zip(host, ref_out, new_out):
        if M == 0:
            continue
        ref = si.bits_to_float64(_bits(Dr)[:, :N], "bf16")
        got = si.bits_to_float64(_bits(Dn)[:, :N], "bf16")
        D, S = og.gemm(M, N, K, A, B, in_fmt="bf16", a_major="K", b_major="K", C=C, c_fmt="bf16",
                       ldc=(N + 7) // 8 * 8, alpha=alpha, beta=beta)
        assert np.isfinite(got).all()
        # against the oracle: the parity bar of every GPU path
        assert (np.abs(got - D) <= og.tolerance(S, D, "bf16")).all()
        # against the workspace-taking entry point on the same inputs
        assert (np.abs(got - ref) <= og.tolerance(S, ref, "bf16")).all()


def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls_in_a_row(g):
    # first call: several ragged problems, one empty; second call: fewer, larger
    # problems with beta, reusing (and rewriting) the same fixed table
    _one_round(g, [128, 300, 0, 256, 72], 200, 136, seed=500, alpha=1.0, beta=0.0)
    _one_round(g, [384, 640], 264, 320, seed=600, alpha=0.5, beta=-1.5)


def test_noalloc_rejects_more_problems_than_the_table_holds(g):
    n = g.NOALLOC_MAX_PROBLEMS + 1
    probs = [dict(M=0, N=8, K=8, A=None, B=None, C=None, D=None, lda=8, ldb=8, ldc=0, ldd=8)] * n
    with pytest.raises(g.GemmError) as ei:
        g.gemm_bf16_grouped_noalloc(probs, g.K_MAJOR, g.K_MAJOR, g.OUT_BF16, 1.0, 0.0)
    assert ei.value.status == g.ERR_INVALID_ARG
