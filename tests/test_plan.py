"""Tile planning, on the host (gemm_debug_plan runs the library's own planner; no GPU).

Each case pins one rule of the planner: CTA pairs for large problems, the
64-row tiles for tiny M, the K depth per stage of each operand format, the
widest swizzle that fits a stage, the fixed tiles of the block-scaled
formats, and the options it must refuse.
"""
import pytest

SMS = 148
BF16, FP8, MXFP8, NVFP4, MXFP4, TF32 = 0, 1, 2, 3, 4, 5
K_MAJOR, MN_MAJOR = 0, 1


@pytest.fixture(scope="module")
def g():
    from smem_swizzle_layouts_gb300 import _lib
    return _lib


def plan(g, M, N, K, kind=BF16, a=K_MAJOR, b=K_MAJOR, sms=SMS, **opts):
    return g.gemm_debug_plan(M, N, K, kind, a, b, options=opts or None, sms=sms)


def test_large_bf16_uses_cta_pairs_with_256_wide_tiles_and_two_swizzle_rows_of_k(g):
    p = plan(g, 8192, 8192, 8192, b=MN_MAJOR)
    assert (p["cta_group"], p["tile_n"], p["block_k"], p["tile_m"]) == (2, 256, 128, 128)
    assert (p["swizzle_a"], p["swizzle_b"]) == (3, 3)


def test_pairs_only_from_2048_rows_and_columns(g):
    assert plan(g, 2048, 2048, 512)["cta_group"] == 2
    assert plan(g, 2047, 8192, 512)["cta_group"] == 1
    assert plan(g, 8192, 2047, 512)["cta_group"] == 1
    assert plan(g, 4096, 128, 4096, cta_group=2)["tile_n"] == 128  # narrow N: 128-wide pair tiles


def test_single_cta_256_wide_tiles_keep_four_stages_of_64(g):
    p = plan(g, 4096, 4096, 4096, cta_group=1, tile_n=256, tile_m=128)
    assert (p["tile_n"], p["block_k"], p["swizzle_a"]) == (256, 64, 3)


def test_single_cta_tile_width_follows_the_sm_count(g):
    # 256-wide tiles only when they still fill every SM
    assert plan(g, 8192, 8192, 1024, cta_group=1)["tile_n"] == 256
    assert plan(g, 4096, 512, 1024, cta_group=1)["tile_n"] == 128     # 32 x 2 tiles of 256 < 148 SMs
    assert plan(g, 4096, 64, 1024)["tile_n"] == 64


def test_tiny_m_uses_64_row_tiles(g):
    p = plan(g, 64, 4096, 4096)
    assert (p["tile_m"], p["cta_group"], p["tile_n"], p["block_k"]) == (64, 1, 128, 128)
    assert plan(g, 65, 4096, 4096)["tile_m"] == 128
    with pytest.raises(g.GemmError) as ei:
        plan(g, 64, 4096, 4096, tile_m=64, cta_group=2)
    assert ei.value.status == g.ERR_UNSUPPORTED


def test_short_k_rows_get_narrower_swizzles(g):
    # a K-major row of 64 bytes (32 bf16) cannot fill a 128-byte swizzle row
    p = plan(g, 512, 512, 32)
    assert (p["block_k"], p["swizzle_a"], p["swizzle_b"]) == (32, 2, 2)
    assert plan(g, 512, 512, 4096, swizzle_a=4, swizzle_b=1)["swizzle_a"] == 0   # explicit no-swizzle


def test_fp8_stage_depth_in_bytes_matches_bf16(g):
    assert plan(g, 8192, 8192, 8192, FP8)["block_k"] == 256
    assert plan(g, 8192, 8192, 8192, FP8, cta_group=1, tile_n=256)["block_k"] == 128


def test_mn_major_swizzle_fits_the_tile_extent(g):
    # fp8 pairs of 128-wide tiles: each CTA holds 64 columns of B, one 64-byte swizzle row
    p = plan(g, 4096, 4096, 4096, MXFP8, a=MN_MAJOR, b=MN_MAJOR, cta_group=2)
    assert (p["cta_group"], p["tile_n"], p["swizzle_a"], p["swizzle_b"]) == (2, 128, 3, 2)


def test_block_scaled_formats_have_fixed_tiles(g):
    # large MXFP8: 256 x 256 pair tiles; smaller problems and fp4: single CTAs of 128 x 128
    assert plan(g, 8192, 8192, 8192, MXFP8) == dict(cta_group=2, tile_n=256, block_k=256, tile_m=128, swizzle_a=3,
                                                    swizzle_b=3, epilogue_swizzle=1, group_m=8, mma_ws=0,
                                                    multicast_b=0)
    assert plan(g, 1024, 8192, 8192, MXFP8) == dict(cta_group=1, tile_n=128, block_k=256, tile_m=128, swizzle_a=3,
                                                    swizzle_b=3, epilogue_swizzle=1, group_m=8, mma_ws=0,
                                                    multicast_b=0)
    assert plan(g, 8192, 8192, 8192, MXFP8, cta_group=2)["tile_n"] == 128
    assert plan(g, 8192, 8192, 8192, MXFP8, cta_group=2, tile_n=256)["tile_n"] == 256
    # a stage depth only single CTAs are built for keeps large problems on single CTAs
    assert plan(g, 8192, 8192, 8192, MXFP8, block_k=128)["cta_group"] == 1
    # fp4 (K in bytes): 256 x 256 pairs by default for large problems, 128 bytes per
    # stage for NVFP4 and 256 for MXFP4 (a pair stage of four MMAs issues too slowly);
    # MXFP4 pairs also run 128-byte stages when asked
    for kind, bk in ((NVFP4, 128), (MXFP4, 256)):
        p = plan(g, 8192, 8192, 8192, kind)
        assert (p["cta_group"], p["tile_n"], p["block_k"]) == (2, 256, bk), kind
    assert plan(g, 8192, 8192, 8192, MXFP4, block_k=128)["block_k"] == 128
    assert plan(g, 1024, 8192, 8192, NVFP4)["block_k"] == 128    # single CTAs: 256 E2M1 per stage
    assert plan(g, 1024, 8192, 8192, MXFP4)["block_k"] == 256
    assert plan(g, 1024, 1024, 8192, NVFP4, cta_group=2)["tile_n"] == 256
    for kind, opts in [(MXFP8, dict(tile_n=256, cta_group=1)), (NVFP4, dict(cta_group=2, tile_n=128)),
                       (MXFP4, dict(cta_group=1, block_k=128)), (NVFP4, dict(tile_m=64))]:
        with pytest.raises(g.GemmError) as ei:
            plan(g, 4096, 4096, 4096, kind, **opts)
        assert ei.value.status == g.ERR_UNSUPPORTED, (kind, opts)


def test_invalid_options_are_rejected(g):
    for opts, status in [(dict(flags=128), g.ERR_INVALID_ARG), (dict(stream_k=4), g.ERR_INVALID_ARG),
                         (dict(swizzle_a=6), g.ERR_INVALID_ARG), (dict(tile_m=96), g.ERR_INVALID_ARG),
                         (dict(workspace=0x1010), g.ERR_ALIGNMENT), (dict(tile_n=96), g.ERR_UNSUPPORTED),
                         (dict(mma_ws=2), g.ERR_INVALID_ARG), (dict(tile_m=16), g.ERR_INVALID_ARG),
                         (dict(tile_m=512), g.ERR_INVALID_ARG)]:
        with pytest.raises(g.GemmError) as ei:
            plan(g, 1024, 1024, 1024, **opts)
        assert ei.value.status == status, opts


def test_32_byte_atom_swizzle_is_refused_for_gemm_operands(g):
    # GEMM_SWIZZLE_128B_ATOM32 (descriptor code 1) is read as zeros by the MMA kinds the
    # library issues, so the planner refuses it for either operand and major
    for kind in (BF16, FP8):
        for a, b, opts in ((MN_MAJOR, MN_MAJOR, dict(swizzle_a=5)), (MN_MAJOR, MN_MAJOR, dict(swizzle_b=5)),
                           (K_MAJOR, K_MAJOR, dict(swizzle_a=5))):
            with pytest.raises(g.GemmError) as ei:
                plan(g, 1024, 1024, 1024, kind, a=a, b=b, **opts)
            assert ei.value.status == g.ERR_UNSUPPORTED, (kind, opts)


def test_weight_stationary_tiles(g):
    # tile_m 32 exists only as tcgen05.mma.ws (256 wide, 64 K per stage); mma_ws 1 picks
    # .ws for 64-row tiles too; both are single-CTA, 16-bit, single-problem tiles
    p = plan(g, 20, 4096, 4096, tile_m=32)
    assert (p["tile_m"], p["mma_ws"], p["tile_n"], p["block_k"], p["cta_group"]) == (32, 1, 256, 64, 1)
    p = plan(g, 20, 4096, 4096, mma_ws=1)
    assert (p["tile_m"], p["mma_ws"], p["tile_n"]) == (64, 1, 128)
    p = plan(g, 64, 16384, 4096, mma_ws=1)
    assert (p["tile_m"], p["mma_ws"], p["tile_n"], p["block_k"]) == (64, 1, 128, 128)
    p = plan(g, 64, 16384, 4096, tile_m=64, tile_n=256, mma_ws=1)
    assert (p["tile_m"], p["mma_ws"], p["tile_n"], p["block_k"]) == (64, 1, 256, 64)
    # M <= 64 defaults to .ws 64 x 128 tiles; an explicit tile_m 64 (or mma_ws -1) keeps Layout F
    assert (plan(g, 64, 16384, 4096)["mma_ws"], plan(g, 20, 16384, 4096)["tile_m"]) == (1, 64)
    assert plan(g, 64, 16384, 4096, tile_m=64)["mma_ws"] == 0
    assert plan(g, 64, 16384, 4096, mma_ws=-1)["mma_ws"] == 0
    assert plan(g, 64, 65536, 4096)["mma_ws"] == 0        # 256-wide 64-row tiles stay in Layout F
    # M-major A of 32 rows: a 64-byte swizzle row (32 elements) fits the tile
    assert plan(g, 32, 4096, 4096, a=MN_MAJOR, tile_m=32)["swizzle_a"] == 2
    for kind, opts in [(BF16, dict(tile_m=32, cta_group=2)), (BF16, dict(tile_m=32, mma_ws=-1)),
                       (BF16, dict(tile_m=128, mma_ws=1)), (FP8, dict(tile_m=32)), (MXFP8, dict(mma_ws=1)),
                       (BF16, dict(tile_m=32, tile_n=128))]:
        with pytest.raises(g.GemmError) as ei:
            plan(g, 32, 4096, 4096, kind, **opts)
        assert ei.value.status == g.ERR_UNSUPPORTED, (kind, opts)
    with pytest.raises(g.GemmError) as ei:
        g.gemm_debug_plan(32, 4096, 4096, BF16, K_MAJOR, K_MAJOR, grouped=True, options=dict(mma_ws=1), sms=SMS)
    assert ei.value.status == g.ERR_UNSUPPORTED


def test_b_multicast_clusters(g):
    # two single-CTA 128 x 256 tiles share their B panel by multicast when asked
    p = plan(g, 4096, 4096, 4096, cta_group=1, tile_n=256, tile_m=128, multicast_b=1)
    assert (p["cta_group"], p["tile_n"], p["block_k"], p["tile_m"], p["multicast_b"]) == (1, 256, 64, 128, 1)
    p = plan(g, 4096, 4096, 2048, cta_group=1, tile_n=256, multicast_b=1)   # short K: 128-row tiles
    assert (p["tile_m"], p["multicast_b"]) == (128, 1)
    p = plan(g, 8192, 8192, 8192, FP8, cta_group=1, tile_n=256, multicast_b=1)
    assert (p["block_k"], p["multicast_b"]) == (128, 1)
    for kind, opts in [(BF16, dict(cta_group=2, multicast_b=1)), (BF16, dict(tile_m=64, multicast_b=1)),
                       (MXFP8, dict(multicast_b=1)), (BF16, dict(cta_group=1, tile_n=128, multicast_b=1))]:
        with pytest.raises(g.GemmError) as ei:
            plan(g, 4096, 4096, 4096, kind, **opts)
        assert ei.value.status == g.ERR_UNSUPPORTED, (kind, opts)
    with pytest.raises(g.GemmError) as ei:
        plan(g, 4096, 4096, 4096, multicast_b=2)
    assert ei.value.status == g.ERR_INVALID_ARG


def test_b_multicast_default_rule(g):
    # single-CTA 128 x 256 tiles share B by default when B is MN-major or A + B overflow L2
    one = dict(cta_group=1, tile_n=256, tile_m=128)
    assert plan(g, 4096, 4096, 4096, **one)["multicast_b"] == 0           # K/K, 64 MB
    assert plan(g, 4096, 4096, 4096, b=MN_MAJOR, **one)["multicast_b"] == 1
    assert plan(g, 8192, 8192, 8192, **one)["multicast_b"] == 1           # 256 MB
    assert plan(g, 8192, 8192, 2048, **one)["multicast_b"] == 0           # 64 MB
    assert plan(g, 8192, 8192, 8192, multicast_b=-1, **one)["multicast_b"] == 0
    assert plan(g, 128, 8192, 8192, **one)["multicast_b"] == 0            # one row tile
    assert plan(g, 8192, 8192, 2048, b=MN_MAJOR, cta_group=1, tile_n=256)["multicast_b"] == 1  # short K: 128 rows
    assert plan(g, 8192, 8192, 8192)["cta_group"] == 2                   # pairs stay the default


def test_two_half_tiles_for_large_single_cta_problems_with_long_k(g):
    # 256 rows on one CTA (two M = 128 MMAs per B slice, both accumulators in TMEM)
    p = plan(g, 4096, 4096, 4096, cta_group=1, tile_n=256)
    assert (p["tile_m"], p["tile_n"], p["block_k"], p["cta_group"], p["multicast_b"]) == (256, 256, 64, 1, 1)
    # 224 wide where that takes fewer rounds of the grid: 4096^2 on 152 SMs is two
    # full rounds of 256 x 224 tiles against two of 256-wide clusters for 1.68 waves
    p = plan(g, 4096, 4096, 4096, cta_group=1, sms=152)
    assert (p["tile_m"], p["tile_n"], p["block_k"], p["multicast_b"]) == (256, 224, 64, 0)
    assert plan(g, 8192, 8192, 8192, cta_group=1, sms=152)["tile_n"] == 256        # 7 rounds either way
    assert plan(g, 4096, 4096, 4096, b=MN_MAJOR, cta_group=1, sms=152)["tile_n"] == 256  # K-major A and B only
    assert plan(g, 4096, 4096, 4096, a=MN_MAJOR, cta_group=1, sms=152)["tile_n"] == 256
    p = plan(g, 700, 900, 200, tile_m=256, tile_n=224)
    assert (p["tile_n"], p["block_k"], p["multicast_b"]) == (224, 64, 0)   # 224 wide keeps its own B
    assert plan(g, 700, 900, 200, tile_m=256, tile_n=224, multicast_b=1)["multicast_b"] == 1
    with pytest.raises(g.GemmError) as ei:
        plan(g, 700, 900, 200, b=MN_MAJOR, tile_m=256, tile_n=224, multicast_b=1)  # halves of 112: not whole atoms
    assert ei.value.status == g.ERR_UNSUPPORTED
    assert plan(g, 4096, 4096, 4096, cta_group=1, multicast_b=-1)["multicast_b"] == 0   # pairs of CTAs share B unless refused
    assert plan(g, 256, 4096, 4096, tile_m=256)["multicast_b"] == 0                        # one row tile: nothing to share
    p = plan(g, 8192, 8192, 8192, cta_group=1, multicast_b=1)                              # asked for: two-half tiles share B
    assert (p["tile_m"], p["multicast_b"]) == (256, 1)
    assert plan(g, 8192, 8192, 8192, a=MN_MAJOR, b=MN_MAJOR, cta_group=1)["tile_m"] == 256
    assert plan(g, 8192, 8192, 2048, cta_group=1)["tile_m"] == 128       # short K: the epilogue would weigh more
    assert plan(g, 2047, 8192, 8192, cta_group=1)["tile_m"] == 128       # fewer than 2048 rows
    assert plan(g, 8192, 8192, 8192, cta_group=1, tile_m=128)["tile_m"] == 128
    assert plan(g, 8192, 8192, 8192, cta_group=1, tile_n=128)["tile_m"] == 128
    assert plan(g, 8192, 8192, 8192, FP8, cta_group=1)["tile_m"] == 128  # 16-bit operands only
    assert plan(g, 8192, 8192, 8192)["cta_group"] == 2                   # pairs stay the default
    p = plan(g, 512, 512, 256, tile_m=256)
    assert (p["tile_m"], p["tile_n"], p["cta_group"], p["block_k"], p["multicast_b"]) == (256, 256, 1, 64, 1)
    for opts in (dict(tile_m=256, cta_group=2), dict(tile_m=256, tile_n=128), dict(tile_m=256, mma_ws=1)):
        with pytest.raises(g.GemmError) as ei:
            plan(g, 4096, 4096, 4096, **opts)
        assert ei.value.status == g.ERR_UNSUPPORTED, opts
    with pytest.raises(g.GemmError) as ei:
        plan(g, 4096, 4096, 4096, FP8, tile_m=256)
    assert ei.value.status == g.ERR_UNSUPPORTED


def test_tf32_tiles_and_swizzles(g):
    # TF32 stages hold the bytes of the 16-bit ones; MN-major TF32 operands take the
    # 32-byte-atom swizzle (bits 4) and nothing else, K-major ones SW128
    p = plan(g, 4096, 4096, 4096, TF32, b=MN_MAJOR, cta_group=1, tile_n=256)
    assert (p["block_k"], p["swizzle_a"], p["swizzle_b"]) == (32, 3, 4)
    p = plan(g, 8192, 8192, 8192, TF32, a=MN_MAJOR, b=MN_MAJOR)
    assert (p["cta_group"], p["block_k"], p["swizzle_a"], p["swizzle_b"]) == (2, 64, 4, 4)
    for opts in (dict(swizzle_b=3), dict(swizzle_b=4), dict(swizzle_b=2)):
        with pytest.raises(g.GemmError) as ei:
            plan(g, 4096, 4096, 4096, TF32, b=MN_MAJOR, **opts)
        assert ei.value.status == g.ERR_UNSUPPORTED, opts
    with pytest.raises(g.GemmError):
        plan(g, 4096, 4096, 4096, TF32, swizzle_a=5)      # K-major TF32: not the 32-byte-atom mode
