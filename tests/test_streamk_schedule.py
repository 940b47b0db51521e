"""The stream-K schedule, listed on the host by the library's own unit iterator.

`gemm_debug_streamk_units` runs, on the CPU, the same split rule and unit
iterator that the kernel's producer, MMA issuer and epilogue walk. These
tests check what makes the split correct and deadlock-free, for many tile
counts, grid sizes, K-block counts and modes:
  - every (tile, K block) is accumulated by exactly one cluster;
  - a cluster contributes a partial sum at most once per launch (one slot
    per CTA suffices), and only in its first split unit;
  - a head is its cluster's last unit (so the other TMEM buffer is free
    while it runs), and it waits for exactly the clusters that contributed
    to its tile, all of them later clusters (the waits form no cycle);
  - data-parallel tiles come before split ones and are dealt round-robin.
"""
import itertools

import pytest

WHOLE, CONTRIB, HEAD = 0, 1, 2


@pytest.fixture(scope="module")
def g():
    from smem_swizzle_layouts_gb300 import _lib
    return _lib


def _schedule(g, mode, T, G, kbt):
    per = [g.gemm_debug_streamk_units(mode, T, G, kbt, c) for c in range(G)]
    if per[0] is None:
        assert all(p is None for p in per)
        return None
    return per


def _check(per, T, G, kbt):
    cover = {}
    contributors = {}
    heads = {}
    for c, units in enumerate(per):
        split_units = [u for u in units if u[2] >= 0]
        whole_dp = [u for u in units if u[2] < 0]
        # data-parallel tiles first, dealt c, c+G, ...
        assert units[:len(whole_dp)] == whole_dp
        assert [u[0] for u in whole_dp] == list(range(c, c + G * len(whole_dp), G))
        n_contrib = 0
        for i, (tile, k0, k1, kind, lo, hi) in enumerate(units):
            ks = range(kbt) if k1 < 0 else range(k0, k1)
            assert len(ks) > 0
            for k in ks:
                cover[(tile, k)] = cover.get((tile, k), 0) + 1
            if kind == CONTRIB:
                n_contrib += 1
                assert k0 > 0 and split_units.index(units[i]) == 0
                contributors.setdefault(tile, set()).add(c)
            elif kind == HEAD:
                assert k0 == 0 and k1 < kbt and i == len(units) - 1
                assert c < lo <= hi < G
                heads[tile] = (c, lo, hi)
            else:
                assert k1 < 0 or (k0 == 0 and k1 == kbt)
        assert n_contrib <= 1
    assert len(cover) == T * kbt and set(cover.values()) == {1}
    assert set(heads) == set(contributors)
    for tile, (c, lo, hi) in heads.items():
        assert contributors[tile] == set(range(lo, hi + 1)), (tile, c, lo, hi, contributors[tile])


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_schedule_invariants_over_many_shapes(g, mode):
    n_split = 0
    for T, G, kbt in itertools.product([1, 2, 3, 5, 7, 11, 16, 27, 40, 64, 100, 257],
                                       [2, 3, 4, 5, 7, 13, 74, 76],
                                       [1, 2, 3, 8, 32, 64]):
        per = _schedule(g, mode, T, G, kbt)
        if per is None:
            continue
        n_split += 1
        _check(per, T, G, kbt)
    assert n_split > 0


def test_auto_splits_only_a_ragged_wave_after_two_to_seven_full_ones(g):
    # 4096^3 CTA pairs on 76 clusters: 256 tiles = 3 waves + 28
    per = _schedule(g, 0, 256, 76, 32)
    assert per is not None
    dp = sum(1 for u in per[0] if u[2] < 0)
    assert dp == 2  # 76 + 28 tiles are split, 152 stay whole: two per cluster
    assert _schedule(g, 0, 228, 76, 32) is None     # whole waves
    assert _schedule(g, 0, 128, 152, 64) is None    # fewer tiles than two waves
    assert _schedule(g, 0, 1024, 76, 64) is None    # thirteen waves and more
    assert _schedule(g, -1, 256, 76, 32) is None    # off


def test_forced_modes(g):
    # mode 1 with fewer tiles than two waves splits every tile
    per = _schedule(g, 1, 6, 4, 8)
    assert all(u[2] >= 0 for units in per for u in units)
    # mode 3: only the ragged wave (27 = 5 * 5 + 2)
    per = _schedule(g, 3, 27, 5, 7)
    assert sum(1 for units in per for u in units if u[2] < 0) == 25
    # fewer K blocks in the split tiles than clusters: stays data-parallel
    assert _schedule(g, 2, 1, 8, 4) is None


def test_invalid_arguments(g):
    assert g.gemm_debug_streamk_units(2, 10, 0, 4, 0) is None
    assert g.gemm_debug_streamk_units(2, 10, 4, 0, 0) is None
    assert g.gemm_debug_streamk_units(2, 10, 4, 4, 4) is None
