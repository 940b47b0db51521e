"""GPU parity at the size limits: outputs past 2^31 elements and very long K (2^19).

Entries are sampled (gathered on the GPU) and compared with the oracle's
entry-wise products within the parity tolerance; the samples include the
last row and column and the entries around linear offset 2^31 of D.
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


def _check_sampled(g, M, N, K, rows, cols, seed, options=None):
    A = si.matrix_bits(seed, M, K, "uniform", "bf16")                      # K-major A
    B = si.matrix_bits(seed + 1, K, N, "uniform", "bf16", transpose=True)  # K-major B
    At = si.torch_from_bits(A, "bf16").to(DEV)
    Bt = si.torch_from_bits(B, "bf16").to(DEV)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    g.gemm_ex(1, M, N, K, At, 0, K, Bt, 0, K, None, 0, D, N, 1, 1.0, 0.0, options=options)
    st, word = g.gemm_last_device_status()
    assert st == g.OK, hex(word)
    r = torch.from_numpy(rows).to(DEV)
    c = torch.from_numpy(cols).to(DEV)
    got = D[r, c].float().cpu().numpy().astype(np.float64)
    ref, S = og.gemm_entries(M, N, K, A, B, rows, cols, in_fmt="bf16")
    bad = np.abs(got - ref) > og.tolerance(S, ref, "bf16")
    assert not bad.any(), f"{int(bad.sum())} sampled entries outside tolerance"
    del D


def test_output_past_two_to_the_31_elements(g):
    M = N = 49152                      # 2.4e9 outputs (4.8 GB of bf16)
    K = 64
    rng = np.random.default_rng(11)
    edge = 2 ** 31
    lin = np.array([edge - 1, edge, edge + 1, edge + N, M * N - 1], dtype=np.int64)
    rows = np.concatenate([rng.integers(0, M, 512), lin // N, [0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 512), lin % N, [N - 1, 0]])
    _check_sampled(g, M, N, K, rows, cols, seed=71)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_very_long_k(g, cta_group):
    # one output tile (one pair tile for pairs) accumulating 2^19 products per entry
    M, N, K = 128 * cta_group, 256, 1 << 19
    rng = np.random.default_rng(12)
    rows = np.concatenate([rng.integers(0, M, 96), [0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 96), [N - 1, 0]])
    _check_sampled(g, M, N, K, rows, cols, seed=73, options=dict(cta_group=cta_group, tile_n=256))
