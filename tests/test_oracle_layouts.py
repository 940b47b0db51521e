"""Pins of the layout oracle against what the pages print and what the maths fixes."""
import itertools

import pytest

from conftest import golden_lines
from oracle import layouts as L


# ---------------------------------------------------------------------------
# XOR grid swizzle: bijection, row and column distinctness, brute force
# ("Swizzling explained properly", "Why does that work?").
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("a,b", [(a, b) for b in range(0, 6) for a in range(0, b + 1)])
def test_xor_grid_is_bijective_and_spreads_rows_and_columns(a, b):
    M, N = 1 << a, 1 << b
    image = set()
    for r in range(M):
        cols = set()
        for c in range(N):
            r2, c2 = L.xor_grid(r, c)
            assert r2 == r and 0 <= c2 < N
            image.add((r2, c2))
            cols.add(c2)
        assert len(cols) == N                     # same row -> distinct columns
    assert len(image) == M * N                    # bijection
    for c in range(N):
        assert len({L.xor_grid(r, c)[1] for r in range(M)}) == M   # same column -> distinct columns


def test_xor_grid_needs_rows_le_cols():
    # with more rows than columns the XOR leaves the grid (the a <= b premise matters)
    assert any(L.xor_grid(r, c)[1] >= 2 for r in range(4) for c in range(2))


# ---------------------------------------------------------------------------
# Swizzle functor ("CUTLASS swizzling notation", "What about base?").
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits,base,shift", [(b, m, s) for b in range(0, 4) for m in range(0, 5)
                                             for s in range(max(b, 1), 6)])
def test_functor_is_a_bijection_that_keeps_the_base_bits(bits, base, shift):
    sw = L.Swizzle(bits, base, shift)
    span = 1 << (base + bits + shift + 1)
    out = [sw(o) for o in range(span)]
    assert sorted(out) == list(range(span))
    for o in range(span):
        assert out[o] & ((1 << base) - 1) == o & ((1 << base) - 1)
        assert sw(sw(o)) == o                      # an XOR with bits it does not change: involution


@pytest.mark.parametrize("bits,shift", [(1, 3), (2, 3), (3, 3), (2, 4)])
def test_functor_is_the_xor_grid_on_raster_offsets(bits, shift):
    # YY = row bits, ZZZ = column bits: offset r * 2^shift + c -> r * 2^shift + (c ^ r)
    sw = L.Swizzle(bits, 0, shift)
    for r in range(1 << bits):
        for c in range(1 << shift):
            assert sw(r * (1 << shift) + c) == r * (1 << shift) + L.xor_grid(r, c)[1]


def test_functor_negative_shift_moves_yyy_left():
    sw = L.Swizzle(2, 0, -3)
    assert sw.yyy_mask == 0b11 and sw.zzz_mask == 0b11000
    assert sw(0b00001) == 0b01001


def test_functor_for_small_grid_repeats_columns_on_a_bigger_grid():
    # a 2x8 pattern (1 row bit) used on an 8x8 grid sends each column to only 2 columns
    sw = L.Swizzle(1, 0, 3)
    for c in range(8):
        landed = [sw(r * 8 + c) % 8 for r in range(8)]
        assert len(set(landed)) == 2 and all(landed.count(x) == 4 for x in set(landed))


def test_canonical_modes_match_page(golden):
    for row in golden("p3_swizzle.txt"):
        if row[0] == "mode":
            mode, bits, base, shift = row[1], *map(int, row[2:])
            assert L.SWIZZLE[mode] == L.Swizzle(bits, base, shift)


def test_sw32_row1_example(golden):
    rows = {r[0]: list(map(int, r[1:])) for r in golden("p3_swizzle.txt") if r[0].startswith("sw32_row1")}
    sw = L.SWIZZLE["sw32"]
    # 16 B cells, 8 per 128 B row: cell index = byte offset / 16
    after = [sw(cell * 16) // 16 for cell in rows["sw32_row1_before"]]
    # the page lists, slot by slot, which logical cell now sits in the slot
    inv = {sw(cell * 16) // 16: cell for cell in range(16)}
    assert [inv[slot] for slot in rows["sw32_row1_before"]] == rows["sw32_row1_after"]
    assert sorted(after) == rows["sw32_row1_before"]


def test_column_read_conflict_degrees(golden):
    for row in golden("p3_swizzle.txt"):
        if row[0] == "column_degree":
            for col in range(8):
                assert L.column_read_degree(row[1], col) == int(row[2])


def test_bank_model_wavefronts():
    # 32 threads x 4 B along a row: one wavefront; down a 128 B-stride column: 32-way
    assert L.conflict_degree([4 * t for t in range(32)], 4) == (1, 1)
    assert L.conflict_degree([128 * t for t in range(32)], 4) == (32, 32)
    # 32 threads x 8 B contiguous: two 128 B wavefronts, no conflict
    assert L.conflict_degree([8 * t for t in range(32)], 8) == (1, 2)
    # the same address from every thread is a broadcast, not a conflict
    assert L.conflict_degree([0] * 32, 4) == (1, 1)


# ---------------------------------------------------------------------------
# "LBO, SBO and SWZ for a tcgen05 tile": printed values.
# ---------------------------------------------------------------------------

def test_p1_unswizzled_rows_and_cell_banks(golden):
    rows = golden("p1_unswizzled_rows.txt")
    starts = list(map(int, rows[0][1:]))
    assert [L.p1_unswizzled_cell(m, 0) for m in range(8)] == starts
    for r in rows[1:]:
        q = int(r[1][1:-1])
        lo, hi = int(r[2]), int(r[3])
        b = L.banks_of_access(L.p1_unswizzled_cell(0, q), 16)
        assert (b[0], b[-1]) == (lo, hi)


def test_p1_sw64_bank_sequence(golden):
    for r, lo, hi in (map(int, row) for row in golden("p1_sw64_banks.txt")):
        b = L.banks_of_access(L.p1_sw64_cell_addr(0, 0, r, 0), 16)
        assert (b[0], b[-1]) == (lo, hi)
    # the whole q0 column of the 8-row core matrix covers 32 distinct banks
    banks = [x for r in range(8) for x in L.banks_of_access(L.p1_sw64_cell_addr(0, 0, r, 0), 16)]
    assert sorted(banks) == list(range(32))
    # and the MMA's read of one core-matrix column is conflict-free
    assert L.conflict_degree([L.p1_sw64_cell_addr(0, 0, r, 0) for r in range(8)], 16)[0] == 1


def test_p1_mbo_key_tables(golden):
    rows = golden("p1_mbo_keys.txt")
    for row in rows:
        if row[0] == "mbo_from_start":
            assert L.p1_mbo(int(row[1])) == int(row[2])
        else:
            mbo, keys = int(row[0]), list(map(int, row[1:]))
            assert [L.p1_sw64_key(r, mbo) for r in range(8)] == keys


def test_p1_mbo_table_equals_absolute_address_xor():
    # a pattern starting at byte 128 (MBO = 1): the page's shifted key is what the XOR
    # of the absolute address bits gives
    P = 128
    for band, r, q in itertools.product(range(4), range(8), range(4)):
        pre = P + band * 512 + r * 64 + q * 16
        assert L.p1_sw64_cell_addr(P, band, r, q, mbo=L.p1_mbo(P)) == L._xor_absolute(pre, 2)


def test_p1_descriptor_values_encode(golden):
    g = {}
    for row in golden("p1_descriptors.txt"):
        if row[0] == "SWZ_INVALID":
            assert sorted(L.SWZ_INVALID) == sorted(map(int, row[1:]))
            assert not set(L.SWZ_INVALID) & set(L.SWZ_CODE.values())
            continue
        g[(row[0], row[1])] = list(map(int, row[2:]))
    for name in ("none", "sw32", "sw64", "sw128", "sw128_base32b"):
        assert L.SWZ_CODE[name] == g[("SWZ", name)][0]
    a = L.SmemDesc(start=0, lbo=16, sbo=g[("A", "sbo_bytes")][0], base_offset=0, swz=g[("A", "swz")][0])
    w = L.encode_smem_desc(a)
    assert (w >> 32) & 0x3FFF == g[("A", "sbo_field")][0]
    assert (w >> 16) & 0x3FFF == g[("A", "lbo_field")][0]
    assert w >> 61 == 4 and L.desc_fixed_bits(w) == 1
    assert L.decode_smem_desc(w) == a
    # the page's a_desc1 = a_desc0 + 32 B on the start field only
    a1 = L.SmemDesc(start=32, lbo=16, sbo=512, base_offset=0, swz=4)
    assert L.encode_smem_desc(a1) - w == 32 >> 4
    bn = g[("B", "bn")][0]
    b = L.SmemDesc(start=1024, lbo=g[("B", "lbo_bytes")][0], sbo=(bn // 64) * 1024, base_offset=0,
                   swz=g[("B", "swz")][0])
    assert b.sbo == g[("B", "sbo_bytes")][0]
    wb = L.encode_smem_desc(b)
    assert L.decode_smem_desc(wb) == b and (wb >> 16) & 0x3FFF == 64 and (wb >> 32) & 0x3FFF == 128
    # BK=64 K-major: SBO 1024 whether packed as SW128 or as two SW64 atoms per band
    assert L.stage_slice_desc("K", "sw128", 128, 64, 2, 0, 0).sbo == g[("BK64", "sbo_bytes")][0]


def test_desc_field_round_trip_random():
    import random
    rnd = random.Random(5)
    for _ in range(2000):
        d = L.SmemDesc(start=rnd.randrange(0, 1 << 18, 16), lbo=rnd.randrange(0, 1 << 18, 16),
                       sbo=rnd.randrange(0, 1 << 18, 16), base_offset=rnd.randrange(8),
                       swz=rnd.choice([0, 1, 2, 4, 6]), lbo_mode=rnd.randrange(2))
        assert L.decode_smem_desc(L.encode_smem_desc(d)) == d


# ---------------------------------------------------------------------------
# Three independent routes agree on the page's 128x128x32 fp16 tile.
# ---------------------------------------------------------------------------

P_BASE = 4096  # a 1024-aligned stage base: MBO = 0


def test_a_tile_closed_form_functor_and_descriptor_agree():
    a0 = L.SmemDesc(start=P_BASE, lbo=16, sbo=512, base_offset=0, swz=L.SWZ_CODE["sw64"])
    a1 = L.SmemDesc(start=P_BASE + 32, lbo=16, sbo=512, base_offset=0, swz=L.SWZ_CODE["sw64"])
    seen = set()
    for m in range(128):
        for k in range(32):
            closed = L.p1_a_element_addr(P_BASE, m, k)
            functor = P_BASE + L.SWIZZLE["sw64"](m * 64 + k * 2)
            d = a0 if k < 16 else a1
            interp = L.desc_element_addr(d, "K", 2, m, k % 16)
            rel = L.desc_element_addr_relative(d, "K", 2, m, k % 16, pattern_start=P_BASE)
            stage = P_BASE + L.stage_element_offset("K", "sw64", 128, 32, 2, m, k)
            assert closed == functor == interp == rel == stage, (m, k)
            seen.add(closed)
    assert len(seen) == 128 * 32 and max(seen) - min(seen) == 128 * 64 - 2


@pytest.mark.parametrize("packing", ["page", "tma"])
def test_b_tile_mn_major_sw128_packings(packing):
    # B[32 x 128] fp16, N-major, SW128 atoms of 64 N x 8 K rows
    BK, BN = 32, 128
    if packing == "page":   # K band holds both N atoms: LBO 1024, SBO 2048
        lbo, sbo = 1024, (BN // 64) * 1024
        lin = lambda n, k: (k // 8) * 2048 + (n // 64) * 1024 + (k % 8) * 128 + (n % 64) * 2
    else:                   # one TMA box per N atom (64 N x BK K): LBO BK*128, SBO 1024
        lbo, sbo = BK * 128, 1024
        lin = lambda n, k: (n // 64) * BK * 128 + (k % BK) * 128 + (n % 64) * 2
    seen = set()
    for n in range(BN):
        for k in range(BK):
            j, kk = divmod(k, 16)
            d = L.SmemDesc(start=P_BASE + j * 2 * sbo, lbo=lbo, sbo=sbo, base_offset=0, swz=2)
            interp = L.desc_element_addr(d, "MN", 2, n, kk)
            direct = P_BASE + L.SWIZZLE["sw128"](lin(n, k)) if packing == "tma" else \
                P_BASE + (lin(n, k) & ~1023) + L.SWIZZLE["sw128"](lin(n, k) & 1023)
            assert interp == direct, (n, k)
            if packing == "tma":
                assert interp == P_BASE + L.stage_element_offset("MN", "sw128", BN, BK, 2, n, k)
                assert L.stage_slice_desc("MN", "sw128", BN, BK, 2, j, P_BASE) == d
            seen.add(interp)
    assert len(seen) == BN * BK


@pytest.mark.parametrize("major", ["K", "MN"])
@pytest.mark.parametrize("mode", ["none", "sw32", "sw64", "sw128"])
@pytest.mark.parametrize("rows,bk", [(128, 64), (256, 64), (128, 32)])
def test_stage_packing_matches_descriptor_for_every_slice(major, mode, rows, bk):
    if major == "K" and L.swizzle_width(mode) > bk * 2:
        pytest.skip("K-major swizzle row wider than the K block")
    seen = set()
    for j in range(bk // 16):
        d = L.stage_slice_desc(major, mode, rows, bk, 2, j, P_BASE)
        for mn in range(rows):
            for kk in range(16):
                addr = L.desc_element_addr(d, major, 2, mn, kk)
                assert addr == P_BASE + L.stage_element_offset(major, mode, rows, bk, 2, mn, 16 * j + kk)
                seen.add(addr)
    assert len(seen) == rows * bk and min(seen) == P_BASE and max(seen) < P_BASE + rows * bk * 2


@pytest.mark.parametrize("major", ["K", "MN"])
@pytest.mark.parametrize("mode", ["none", "sw32", "sw64", "sw128"])
def test_second_half_of_a_256_row_stage_is_a_shifted_start(major, mode):
    # A 256-row A stage read by two M = 128 MMAs ("06 Blackwell Tensor Core -
    # tcgen05 MMA": cta_group::1 MMAs have at most 128 rows): the descriptor
    # of rows 128..255 is the stage's own slice descriptor with its start moved
    # by 128 rows' worth of the packing ("LBO, SBO and SWZ for a tcgen05 tile":
    # 8-row groups SBO = 8 W apart for K-major stages, so 16 groups = 128 W;
    # MN-major atoms of W / esize elements LBO = BK W apart, so 128 esize / W
    # atoms = 128 esize BK). Every element of every slice lands where the
    # stage packing puts row 128 + m.
    rows, bk, esize = 256, 64, 2
    W = L.swizzle_width(mode)
    shift = 128 * W if major == "K" else 128 * esize * bk
    for j in range(bk // 16):
        d = L.stage_slice_desc(major, mode, rows, bk, esize, j, P_BASE)
        d2 = L.SmemDesc(start=d.start + shift, lbo=d.lbo, sbo=d.sbo, base_offset=d.base_offset, swz=d.swz)
        for m in range(128):
            for kk in range(16):
                assert L.desc_element_addr(d2, major, esize, m, kk) == \
                    P_BASE + L.stage_element_offset(major, mode, rows, bk, esize, 128 + m, 16 * j + kk)


def test_transposed_operand_reading_is_caught():
    # a plausible slip -- reading an MN-major stage with the K-major formula -- changes addresses
    d = L.stage_slice_desc("MN", "sw128", 128, 64, 2, 0, P_BASE)
    diff = sum(L.desc_element_addr(d, "MN", 2, mn, k) != L.desc_element_addr(d, "K", 2, mn, k)
               for mn in range(128) for k in range(16))
    assert diff > 0


def test_tma_box_rules():
    # SW128 caps the inner box at 128 B: 64 bf16 is fine, 128 bf16 needs two boxes
    assert L.tma_box_ok("sw128", 64, 2) and not L.tma_box_ok("sw128", 128, 2)
    assert L.tma_box_ok("sw64", 32, 2) and not L.tma_box_ok("sw64", 64, 2)
    assert L.tma_stride_ok(8192 * 2) and not L.tma_stride_ok(8190) and not L.tma_stride_ok(1 << 40)


# ---------------------------------------------------------------------------
# Instruction descriptor and legal N.
# ---------------------------------------------------------------------------

def test_legal_n(golden):
    for row in golden("p4_tmem.txt"):
        if row[0] == "N":
            g, lo, hi, step = map(int, row[1:])
            legal = [n for n in range(0, 300) if L.legal_mma_n(g, n)]
            assert legal == list(range(lo, hi + 1, step))


def test_idesc_fields_do_not_overlap():
    w = L.encode_idesc(256, 256, L.FMT_BF16, L.DFMT_F32, 1, 1)
    assert (w >> 24) & 0x1F == 16 and (w >> 17) & 0x3F == 32
    assert (w >> 15) & 1 == 1 and (w >> 16) & 1 == 1
    assert (w >> 4) & 3 == 1 and (w >> 7) & 7 == 1 and (w >> 10) & 7 == 1
    # M, N, formats and majors each move disjoint bits
    fields = [L.encode_idesc(16, 0, 0, 0, 0, 0), L.encode_idesc(0, 8 * 63, 0, 0, 0, 0),
              L.encode_idesc(0, 0, 7, 0, 0, 0), L.encode_idesc(0, 0, 0, 3, 0, 0),
              L.encode_idesc(0, 0, 0, 0, 1, 0), L.encode_idesc(0, 0, 0, 0, 0, 1)]
    for x, y in itertools.combinations(fields, 2):
        assert x & y == 0


# ---------------------------------------------------------------------------
# TMEM maps ("06 Blackwell Tensor Core - tcgen05 MMA").
# ---------------------------------------------------------------------------

def test_tmem_layout_f(golden):
    for row in golden("p4_tmem.txt"):
        if row[0] == "F":
            a, r0, r1, l0, l1 = map(int, row[1:])
            assert [L.tmem_layout_f(m, 0, a)[1] for m in range(r0, r1 + 1)] == list(range(l0, l1 + 1))
    used0 = {L.tmem_layout_f(m, 0, 0)[1] for m in range(64)}
    used16 = {L.tmem_layout_f(m, 0, 16)[1] for m in range(64)}
    assert not used0 & used16 and used0 | used16 == set(range(128))


def test_tmem_layout_b_and_m256(golden):
    for row in golden("p4_tmem.txt"):
        if row[0] == "B":
            N, m, n, cta, lane = map(int, row[1:])
            got = L.tmem_layout_b(m, n, N)
            assert got[:2] == (cta, lane)
        if row[0] == "M256":
            m, cta, lane = map(int, row[1:])
            assert L.tmem_cta2_m256(m, 5)[:2] == (cta, lane)
    for N in (16, 64, 256):
        cells = {L.tmem_layout_b(m, n, N) for m in range(128) for n in range(N)}
        assert len(cells) == 128 * N
        assert {c[1] for c in cells} == set(range(128)) and {c[2] for c in cells} == set(range(N // 2))
    cells = {L.tmem_cta2_m256(m, n) for m in range(256) for n in range(16)}
    assert len(cells) == 256 * 16
    assert {L.tmem_cta1_m128(m, 0)[1] for m in range(128)} == set(range(128))


def test_tmem_warp_quarters():
    for w in range(8):
        assert list(L.tmem_warp_lanes(w)) == list(range(32 * (w % 4), 32 * (w % 4) + 32))


# ---------------------------------------------------------------------------
# mbarrier ring parity, by simulating the barriers ("6.6.1").
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 3, 4, 6])
def test_ring_parity_by_simulation(S):
    completed = [0] * S           # completed phases of each stage's barrier
    for k in range(50):
        s = L.ring_stage(k, S)
        # the consumer of iteration k waits for the phase that is about to complete
        assert L.ring_parity(k, S) == completed[s] & 1
        completed[s] += 1


# ---------------------------------------------------------------------------
# Reload traffic model ("Output swizzle"): 17.18 GB at 8192^3 with 128 tiles.
# ---------------------------------------------------------------------------

def test_reload_traffic(golden):
    g = {r[0]: float(r[1]) for r in golden("p3_traffic.txt")}
    m, n, k, t, e = (int(g[x]) for x in ("m", "n", "k", "tile", "esize"))
    b = L.reload_traffic_bytes(m, n, k, t, t, e)
    assert round(b / 1e9, 2) == g["gmem_to_smem_gb"]
    assert b == int(g["reloads"]) * m * k * e * 2
    assert round(m * n * 4 / 1e6) == g["c_fp32_mb"]


@pytest.mark.parametrize("major", ["K", "MN"])
@pytest.mark.parametrize("mode", ["none", "sw32", "sw64", "sw128"])
@pytest.mark.parametrize("rows,bk", [(128, 128), (256, 128), (128, 256)])
def test_fp8_stage_packing_matches_descriptor_for_every_slice(major, mode, rows, bk):
    # one MMA slice of an 8-bit type is 32 elements of K (32 bytes per row)
    if major == "K" and L.swizzle_width(mode) > bk:
        pytest.skip("K-major swizzle row wider than the K block")
    seen = set()
    for j in range(bk // 32):
        d = L.stage_slice_desc(major, mode, rows, bk, 1, j, P_BASE)
        for mn in range(rows):
            for kk in range(32):
                addr = L.desc_element_addr(d, major, 1, mn, kk)
                assert addr == P_BASE + L.stage_element_offset(major, mode, rows, bk, 1, mn, 32 * j + kk)
                seen.add(addr)
    assert len(seen) == rows * bk


def test_idesc_mixed_ab_formats():
    w = L.encode_idesc(128, 128, L.FMT_E4M3, L.DFMT_F32, 0, 1, b_fmt=L.FMT_E5M2)
    assert (w >> 7) & 7 == 0 and (w >> 10) & 7 == 1 and (w >> 16) & 1 == 1


# ---------------------------------------------------------------------------
# The 128-byte swizzle with 32-byte atoms (raw SWZ value 1; "LBO, SBO and SWZ
# for a tcgen05 tile", section 4, read through "What about base?").
# ---------------------------------------------------------------------------

def test_atom32_functor_is_the_4x4_xor_grid_of_32_byte_atoms():
    sw = L.SWIZZLE[L.ATOM32]
    assert (sw.bits, sw.base, sw.shift) == (2, 5, 2)
    for r in range(4):
        for c in range(4):
            for b in range(32):           # every byte of the atom moves with it
                off = r * 128 + c * 32 + b
                assert sw(off) == r * 128 + L.xor_grid(r, c)[1] * 32 + b
    # a bijection on each 512-byte pattern, repeating every 512 bytes, 16-byte cells stay whole
    span = list(range(4096))
    out = [sw(o) for o in span]
    assert sorted(out) == span
    assert all(out[o + 512] == out[o] + 512 for o in range(4096 - 512))
    assert L.swizzle_repeat(L.ATOM32) == 512 and L.swizzle_width(L.ATOM32) == 128


def test_atom32_interpreter_xor_equals_the_functor_on_absolute_addresses():
    sw = L.SWIZZLE[L.ATOM32]
    for addr in range(0, 1 << 13, 16):
        assert L._xor_absolute(addr, 2, 5) == sw(addr)
        # pattern-relative form with MBO = the start's row phase gives the same address
        for start in (0, 128, 256, 384, 1024):
            if addr >= start:
                assert L._xor_relative(addr, start, (start >> 7) & 3, 2, 5) == sw(addr)


def test_atom32_column_reads_spread_over_four_32_byte_units():
    # reading one 32-byte unit of 4 consecutive 128-byte rows touches 4 distinct units
    sw = L.SWIZZLE[L.ATOM32]
    for c in range(4):
        assert len({sw(r * 128 + c * 32) % 128 for r in range(4)}) == 4


@pytest.mark.parametrize("esize", [2, 1])
@pytest.mark.parametrize("rows,bk", [(128, 64), (256, 64), (128, 128), (64, 256)])
def test_atom32_mn_major_stage_packing_matches_descriptor(esize, rows, bk):
    if esize == 2 and bk > 128:
        pytest.skip("16-bit stages of this width are not built")
    if rows % (128 // esize):
        pytest.skip("an MN atom (128 bytes of MN) wider than the tile")
    kper = 32 // esize
    seen = set()
    for j in range(bk // kper):
        d = L.stage_slice_desc("MN", L.ATOM32, rows, bk, esize, j, P_BASE)
        assert d.swz == 1 and d.sbo == L.ATOM32_K_BAND * 128 and d.lbo == bk * 128
        for mn in range(rows):
            for kk in range(kper):
                addr = L.desc_element_addr(d, "MN", esize, mn, kk)
                assert addr == P_BASE + L.stage_element_offset("MN", L.ATOM32, rows, bk, esize, mn, kper * j + kk)
                assert addr == L.desc_element_addr_relative(d, "MN", esize, mn, kk, pattern_start=P_BASE)
                seen.add(addr)
    assert len(seen) == rows * bk and min(seen) == P_BASE and max(seen) < P_BASE + rows * bk * esize


def test_atom32_is_not_offered_for_k_major_operands():
    with pytest.raises(ValueError):
        L.stage_slice_desc("K", L.ATOM32, 128, 64, 2, 0, P_BASE)
    d = L.SmemDesc(start=P_BASE, lbo=16, sbo=1024, base_offset=0, swz=1)
    with pytest.raises(ValueError):
        L.desc_element_addr(d, "K", 2, 0, 0)


# ---------------------------------------------------------------------------
# Weight-stationary (.ws) accumulator maps ("06 Blackwell Tensor Core -
# tcgen05 MMA", "How cta_group Sets the Operation Scope": .ws is one of the
# four choices that fix the layout; the map itself is a reading).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N", [(32, 64), (32, 128), (32, 256), (64, 64), (64, 128), (64, 256), (128, 128)])
def test_ws_map_is_a_bijection_onto_all_lanes(M, N):
    cells = {L.tmem_ws(m, n, M, N) for m in range(M) for n in range(N)}
    parts = 4 // (M // 32) if M < 128 else 1
    assert len(cells) == M * N
    assert {c[1] for c in cells} == set(range(128))               # every lane is used
    assert {c[2] for c in cells} == set(range(N // parts))        # N / parts columns
    assert all(c[0] == 0 for c in cells)                          # cta_group::1: this CTA's TMEM


@pytest.mark.parametrize("M,N", [(32, 256), (64, 128), (64, 256)])
def test_ws_lane_quarters_hold_whole_32_row_blocks_of_one_column_part(M, N):
    # what an epilogue warp reading its lane quarter (32q .. 32q+31) gets
    for q in range(4):
        lanes = L.tmem_warp_lanes(4 + q)
        held = [(m, n) for m in range(M) for n in range(N) if L.tmem_ws(m, n, M, N)[1] in lanes]
        rows = sorted({m for m, _ in held})
        cols = sorted({n for _, n in held})
        assert len(rows) == 32 and rows == list(range(rows[0], rows[0] + 32))
        assert cols == list(range(cols[0], cols[0] + len(cols))) and len(held) == 32 * len(cols)
        for m, n in held:   # lane = 32 q + row within the block, column = offset in the part
            assert L.tmem_ws(m, n, M, N)[1:] == (32 * q + m - rows[0], n - cols[0])


def test_ws_m128_is_the_ordinary_m128_map_and_m64_differs_from_layout_f():
    assert all(L.tmem_ws(m, n, 128, 128) == L.tmem_cta1_m128(m, n) for m in range(128) for n in range(128))
    # Layout F leaves half of each lane quarter empty; the .ws map uses every lane
    f_lanes = {L.tmem_layout_f(m, n)[1] for m in range(64) for n in range(128)}
    assert len(f_lanes) == 64
    assert any(L.tmem_ws(m, n, 64, 128) != L.tmem_layout_f(m, n) for m in range(64) for n in range(128))


@pytest.mark.parametrize("N", [224, 256, 128])
def test_two_half_map_is_two_m128_maps_side_by_side(N):
    # rows 0..127 are the M = 128 map; rows 128..255 the same map 256 columns on;
    # every cell distinct, inside 128 lanes x 512 columns, each half in the lane
    # quarter of its row (the epilogue warp that owns those lanes reads both halves)
    cells = {L.tmem_two_half(m, n, N) for m in range(256) for n in range(N)}
    assert len(cells) == 256 * N
    assert all(0 <= lane < L.TMEM_LANES and 0 <= col < L.TMEM_COLS for _, lane, col in cells)
    for m in range(128):
        for n in range(0, N, 7):
            assert L.tmem_two_half(m, n, N) == L.tmem_cta1_m128(m, n)
            _, lane, col = L.tmem_two_half(m + 128, n, N)
            assert (lane, col) == (m, 256 + n)
            assert lane in L.tmem_warp_lanes(m // 32)  # the warp of lane quarter m // 32
    # a 64-column chunk read at column 192 of a 224-wide first half stays clear of the second half
    assert max(col for _, _, col in cells if col < 256) == N - 1 < 256
    with pytest.raises(ValueError):
        L.tmem_two_half(0, 0, 320)
