"""Address-map oracle for swizzled shared-memory tiles and tcgen05 operands.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the CUDA path never does, and the
two share no code.

Everything here is a plain, slow restatement of what the pages define,
written as bit arithmetic on Python integers:

* the XOR swizzle of a 2^a x 2^b grid and the swizzle functor with its
  (bits, base, shift) parameters  -- "Swizzling explained properly",
  sections "What does swizzling do?", "Why does that work?",
  "CUTLASS swizzling notation", "What about base?", "32B, 64B and 128B
  swizzles";
* the shared-memory bank model (32 banks x 4 B, requests split into
  128 B wavefronts) -- same page, "Why swizzle?" and "Output swizzle";
* the SW64 K-major cell address, the matrix-base-offset key tables and the
  descriptor field values -- "LBO, SBO and SWZ for a tcgen05 tile",
  sections 2 and 3, and the parameter notes of section 4;
* the TMEM accumulator maps for cta_group::1/::2 -- "06 Blackwell Tensor
  Core - tcgen05 MMA", section "How cta_group Sets the Operation Scope";
* mbarrier ring parity and TMA box rules -- "Tensor Cores, layouts, and
  swizzling", TMA section and 6.6.1.

Readings where the pages are silent (each listed in the design notes):

* Descriptor bit positions (the field table on the LBO/SBO page did not
  survive): start [0,14), LBO [16,30), SBO [32,46), the fixed value 0b001
  in [46,49), base offset [49,52), LBO mode bit 52, swizzle code [61,64);
  start/LBO/SBO in 16-byte units, base offset and swizzle as raw 3-bit
  fields (the page states the units and the codes).
* Instruction-descriptor bit positions for kind::f16 (not on the pages):
  D format [4,6) (0 f16, 1 f32), A format [7,10) and B format [10,13)
  (0 f16, 1 bf16), A negate 13, B negate 14, A major 15, B major 16
  (0 K-major, 1 MN-major), N>>3 in [17,23), M>>4 in [24,29).
* Canonical operand layouts (element (mn, k) of one K=16 slice, before
  the XOR), W = swizzle width in bytes, e = element size, T = W / e:
    K-major,  swizzled : start + (mn//8)*SBO + (mn%8)*W + k*e
    K-major,  none     : start + (mn//8)*SBO + (mn%8)*16 + (k//8)*LBO + (k%8)*e
    MN-major, swizzled : start + (mn//T)*LBO + (k//8)*SBO + (k%8)*W + (mn%T)*e
    MN-major, none     : start + (mn//8)*SBO + (mn%8)*e + (k//8)*LBO + (k%8)*16
  The XOR then flips address bits [4, 4+B) with bits [7, 7+B) of the
  absolute shared-memory address (B = 1, 2, 3 for SW32/64/128).
* Layout B columns: the page gives only the lane; the column is read as
  ``n mod (N/2)``.
* The .ws accumulator (``tmem_ws``): the page names it without printing it;
  read as column parts spread over the lane quarters (see the function).
"""
from __future__ import annotations

from dataclasses import dataclass

# ---------------------------------------------------------------------------
# XOR swizzle on a grid ("Swizzling explained properly", "What does
# swizzling do?"): f(r, c) = (r, c XOR r).
# ---------------------------------------------------------------------------


def xor_grid(r: int, c: int) -> tuple[int, int]:
    """Send grid cell (r, c) to (r, c ^ r)."""
    return r, c ^ r


# ---------------------------------------------------------------------------
# The swizzle functor Swizzle(bits, base, shift) ("CUTLASS swizzling
# notation", "What about base?"), built from the XOR grid above.
#
# The page reads the functor's parameters as the shape of a grid laid out in
# raster order inside an offset: ``base`` is log2 of the atom (the bytes that
# move together, e.g. 16 for a ldmatrix row), ``shift`` is the number of
# column bits of a grid row, and ``bits`` the number of row bits. So an
# offset, from its least significant bit up, holds the position inside an
# atom (``base`` bits, never changed), the atom's column c, and above it the
# grid row r. Swizzling replaces c by c XOR r on the low ``bits`` bits of
# each: the grid map f(r, c) = (r, c XOR r). The row must not have more bits
# than the column ("Why does that work?", part 3), hence |shift| >= bits. A
# negative shift is the notation's mirror image: the row field sits at
# ``base`` and the column field |shift| bits above it.
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class Swizzle:
    bits: int
    base: int
    shift: int

    def __post_init__(self):
        if self.bits < 0 or self.base < 0 or abs(self.shift) < self.bits:
            raise ValueError("a grid needs bits >= 0, base >= 0 and no more row bits than column bits")

    @property
    def row_pos(self) -> int:
        """Lowest offset bit of the grid row."""
        return self.base + self.shift if self.shift >= 0 else self.base

    @property
    def col_pos(self) -> int:
        """Lowest offset bit of the atom's column."""
        return self.base if self.shift >= 0 else self.base - self.shift

    @property
    def yyy_mask(self) -> int:
        """Offset bits of the row that takes part (YYY in the notation)."""
        return ((1 << self.bits) - 1) << self.row_pos

    @property
    def zzz_mask(self) -> int:
        """Offset bits of the column that is rewritten (ZZZ)."""
        return ((1 << self.bits) - 1) << self.col_pos

    def __call__(self, offset: int) -> int:
        size = 1 << self.bits                   # rows (and columns) of the grid
        r = (offset >> self.row_pos) % size
        c = (offset >> self.col_pos) % size
        _, c_new = xor_grid(r, c)               # the cell's new column in the same row
        return offset + ((c_new - c) << self.col_pos)


# Canonical modes ("32B, 64B and 128B swizzles"): 16-byte atoms (base 4),
# 8 columns of 16 B per 128 B row (shift 3), 1/2/3 row bits.
MODE_BITS = {"none": 0, "sw32": 1, "sw64": 2, "sw128": 3}
SWIZZLE = {m: Swizzle(b, 4, 3) for m, b in MODE_BITS.items()}

# The 128-byte swizzle with 32-byte atoms (raw SWZ value 1, "LBO, SBO and SWZ
# for a tcgen05 tile", section 4, which names the mode and nothing more).
# Reading, through "What about base?" (base = log2 of the atom): 32-byte
# atoms (base 5), four of them to a 128-byte row (shift 2) and a square grid
# of four rows (bits 2), i.e. Swizzle(2, 5, 2): the pattern repeats every
# four 128-byte rows. As an MMA operand the mode is read for MN-major tiles
# with K rows in bands of ATOM32_K_BAND rows (SBO steps between bands).
ATOM32 = "sw128_base32b"
SWIZZLE[ATOM32] = Swizzle(2, 5, 2)
ATOM32_K_BAND = 4


def swizzle_width(mode: str) -> int:
    """Bytes per swizzled row: 16 (none), 32, 64 or 128 (both 128-byte modes)."""
    return 128 if mode == ATOM32 else 16 << MODE_BITS[mode]


def swizzle_repeat(mode: str) -> int:
    """Bytes after which the XOR pattern repeats (natural boundary): 8 rows, 4 for 32-byte atoms."""
    return (4 if mode == ATOM32 else 8) * swizzle_width(mode)


# Raw SWZ field values ("LBO, SBO and SWZ for a tcgen05 tile", section 4).
SWZ_CODE = {"none": 0, "sw128_base32b": 1, "sw128": 2, "sw64": 4, "sw32": 6}
SWZ_INVALID = (3, 5, 7)
SWZ_MODE = {v: k for k, v in SWZ_CODE.items()}


# ---------------------------------------------------------------------------
# Shared-memory bank model ("Swizzling explained properly", "Why swizzle?":
# 32 banks of 4 bytes, 128 B per cycle; "Output swizzle": a warp request is
# served in 128-byte wavefronts).
# ---------------------------------------------------------------------------

NUM_BANKS = 32
BANK_BYTES = 4


def bank_of(addr: int) -> int:
    return (addr // BANK_BYTES) % NUM_BANKS


def banks_of_access(addr: int, nbytes: int) -> list[int]:
    return [bank_of(a) for a in range(addr, addr + nbytes, BANK_BYTES)]


def conflict_degree(addrs: list[int], nbytes: int = 16) -> tuple[int, int]:
    """Bank-conflict degree of one warp request.

    ``addrs`` are the start addresses of the threads' accesses (thread
    order), each ``nbytes`` wide. The request is cut into groups of
    128 // nbytes consecutive threads (one 128 B wavefront's worth); in a
    group the cost is the largest number of *distinct* 4-byte words that
    fall into one bank. Returns (max degree over groups, total wavefronts).
    """
    per = max(1, 128 // nbytes)
    worst, total = 0, 0
    for g in range(0, len(addrs), per):
        words: dict[int, set[int]] = {}
        for a in addrs[g:g + per]:
            for w in range(a // BANK_BYTES, (a + nbytes) // BANK_BYTES):
                words.setdefault(w % NUM_BANKS, set()).add(w)
        deg = max(len(v) for v in words.values())
        worst = max(worst, deg)
        total += deg
    return worst, total


def column_read_degree(mode: str, col: int = 0) -> int:
    """Conflict degree of reading one 16 B column of an 8-row x 128 B tile.

    Rows are 128 B apart (8 cells of 16 B); the swizzle mode moves cell
    ``col`` of row r to cell ``col ^ (r & mask)``.
    """
    sw = SWIZZLE[mode]
    addrs = [sw(r * 128 + col * 16) for r in range(8)]
    return conflict_degree(addrs, 16)[0]


# ---------------------------------------------------------------------------
# "LBO, SBO and SWZ for a tcgen05 tile": the page's own A tile
# (BM=128, BK=32 fp16, K-major, SW64, 64-byte rows).
# ---------------------------------------------------------------------------


def p1_unswizzled_cell(m: int, q: int) -> int:
    """Section 2: byte of 16 B cell q of row m before swizzling: 64 m + 16 q."""
    return 64 * m + 16 * q


def p1_mbo(pattern_start: int) -> int:
    """Section 3: matrix base offset = (pattern start >> 7) & 7."""
    return (pattern_start >> 7) & 7


def p1_sw64_key(r: int, mbo: int = 0) -> int:
    """Section 3: SW64 XOR key of row r in an 8-row band, ((MBO & 3) + (r >> 1)) & 3."""
    return ((mbo & 3) + (r >> 1)) & 3


def p1_sw64_cell_addr(P: int, band: int, r: int, q: int, sbo: int = 512, mbo: int = 0) -> int:
    """Section 3: P + band*SBO + r*64 + (q ^ key(r)) * 16."""
    return P + band * sbo + r * 64 + (q ^ p1_sw64_key(r, mbo)) * 16


def p1_a_element_addr(P: int, m: int, k: int, esize: int = 2) -> int:
    """Byte address of A[m][k] in the page's SW64 K-major A tile."""
    cell_elems = 16 // esize
    return p1_sw64_cell_addr(P, m // 8, m % 8, k // cell_elems) + (k % cell_elems) * esize


# ---------------------------------------------------------------------------
# Shared-memory matrix descriptor (64-bit), reading c1 above.
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class SmemDesc:
    start: int          # byte address in the shared window (multiple of 16)
    lbo: int            # bytes (multiple of 16)
    sbo: int            # bytes (multiple of 16)
    base_offset: int    # raw 3-bit field
    swz: int            # raw 3-bit field (SWZ_CODE)
    lbo_mode: int = 0


def encode_smem_desc(d: SmemDesc) -> int:
    if d.start % 16 or d.lbo % 16 or d.sbo % 16:
        raise ValueError("start, LBO and SBO are encoded in 16-byte units")
    start = (d.start & 0x3FFFF) >> 4
    lbo, sbo = d.lbo >> 4, d.sbo >> 4
    if lbo >= 1 << 14 or sbo >= 1 << 14:
        raise ValueError("LBO/SBO field overflow")
    word = start
    word |= lbo << 16
    word |= sbo << 32
    word |= 0b001 << 46
    word |= (d.base_offset & 7) << 49
    word |= (d.lbo_mode & 1) << 52
    word |= (d.swz & 7) << 61
    return word


def decode_smem_desc(word: int) -> SmemDesc:
    return SmemDesc(
        start=(word & 0x3FFF) << 4,
        lbo=((word >> 16) & 0x3FFF) << 4,
        sbo=((word >> 32) & 0x3FFF) << 4,
        base_offset=(word >> 49) & 7,
        swz=(word >> 61) & 7,
        lbo_mode=(word >> 52) & 1,
    )


def desc_fixed_bits(word: int) -> int:
    return (word >> 46) & 7


# ---------------------------------------------------------------------------
# Descriptor interpreter: the byte address the MMA reads for element
# (mn, k) of one K slice described by a descriptor (reading c1/c3 above).
# ---------------------------------------------------------------------------


def _xor_field(mode: str) -> tuple[int, int]:
    """(width, lowest address bit) of the field the mode's XOR rewrites: the 16-byte
    cell index [4, 4+B) for the 16-byte-atom modes, the 32-byte unit [5, 7) for ATOM32."""
    if mode == ATOM32:
        return 2, 5
    return MODE_BITS[mode], 4


def _xor_absolute(addr: int, bits: int, lo: int = 4) -> int:
    """Flip address bits [lo, lo+B) with the bits of the 128-byte row above them, [7, 7+B)."""
    if bits == 0:
        return addr
    mask = (1 << bits) - 1
    return addr ^ (((addr >> 7) & mask) << lo)


def _xor_relative(addr: int, pattern_start: int, mbo: int, bits: int, lo: int = 4) -> int:
    """Same XOR, taking the row phase from the offset to the pattern start plus MBO."""
    if bits == 0:
        return addr
    mask = (1 << bits) - 1
    rel = addr - pattern_start
    key = ((rel >> 7) + mbo) & mask
    return addr ^ (key << lo)


def desc_pre_swizzle_addr(d: SmemDesc, major: str, esize: int, mn: int, k: int) -> int:
    mode = SWZ_MODE[d.swz]
    W = swizzle_width(mode)
    if mode == ATOM32:
        if major != "MN":
            raise ValueError("the 32-byte-atom mode is read for MN-major operands only")
        T, R = W // esize, ATOM32_K_BAND
        return d.start + (mn // T) * d.lbo + (k // R) * d.sbo + (k % R) * W + (mn % T) * esize
    if major == "K":
        if mode == "none":
            cell = 16 // esize
            return d.start + (mn // 8) * d.sbo + (mn % 8) * 16 + (k // cell) * d.lbo + (k % cell) * esize
        return d.start + (mn // 8) * d.sbo + (mn % 8) * W + k * esize
    if major == "MN":
        if mode == "none":
            cell = 16 // esize
            return d.start + (mn // cell) * d.sbo + (mn % cell) * esize + (k // 8) * d.lbo + (k % 8) * 16
        T = W // esize
        return d.start + (mn // T) * d.lbo + (k // 8) * d.sbo + (k % 8) * W + (mn % T) * esize
    raise ValueError(major)


def desc_element_addr(d: SmemDesc, major: str, esize: int, mn: int, k: int) -> int:
    """Physical byte address of element (mn, k) of the slice (absolute-address XOR)."""
    pre = desc_pre_swizzle_addr(d, major, esize, mn, k)
    return _xor_absolute(pre, *_xor_field(SWZ_MODE[d.swz]))


def desc_element_addr_relative(d: SmemDesc, major: str, esize: int, mn: int, k: int,
                               pattern_start: int) -> int:
    """Same address from the pattern-relative XOR with the descriptor's MBO."""
    pre = desc_pre_swizzle_addr(d, major, esize, mn, k)
    return _xor_relative(pre, pattern_start, d.base_offset, *_xor_field(SWZ_MODE[d.swz]))


# ---------------------------------------------------------------------------
# Where a TMA box lands in shared memory: the box is written row by row
# (inner dimension contiguous, rows of inner*esize bytes) and each 16 B
# chunk is moved by the swizzle functor of the tensor map's mode
# ("Tensor Cores, layouts, and swizzling", TMA section: the TMA applies the
# swizzle and the mode must match the shared-memory layout atom; the inner
# box may not exceed the swizzle width).
# ---------------------------------------------------------------------------


def tma_box_offset(mode: str, inner_elems: int, esize: int, row: int, col: int) -> int:
    """Byte offset (from a pattern-aligned base) of box element (row, col)."""
    row_bytes = inner_elems * esize
    if mode != "none" and row_bytes != swizzle_width(mode):
        raise ValueError("this model needs the inner box to span exactly one swizzle row")
    return SWIZZLE[mode](row * row_bytes + col * esize)


def tma_box_ok(mode: str, inner_elems: int, esize: int) -> bool:
    """TMA rule: inner box bytes a multiple of 16 and at most the swizzle width."""
    b = inner_elems * esize
    return b % 16 == 0 and (mode == "none" or b <= swizzle_width(mode))


def tma_stride_ok(stride_bytes: int) -> bool:
    """TMA rule: global strides are multiples of 16 B and below 2^40."""
    return stride_bytes % 16 == 0 and 0 < stride_bytes < (1 << 40)


# ---------------------------------------------------------------------------
# Operand packings of a BM x BK (or BN x BK) stage, built from TMA boxes.
# K-major: boxes of W/e K-elements x rows, one after another along K.
# MN-major: boxes of W/e MN-elements x BK K-rows, one after another along MN.
# The descriptor of slice j (K = 16 elements = 32 B for 16-bit types):
#   K-major : SBO = 8*W, LBO field 1 (unused), start = base + box*rows*W + (32 j mod W)
#   MN-major: LBO = BK*W (next MN atom), SBO = 8*W (next 8-row K band),
#             start = base + j * 2 * SBO
# ---------------------------------------------------------------------------


def stage_element_offset(major: str, mode: str, rows: int, bk: int, esize: int, mn: int, k: int) -> int:
    W = swizzle_width(mode)
    per_row = W // esize
    if major == "K":
        box = k // per_row
        return box * rows * W + tma_box_offset(mode, per_row, esize, mn, k % per_row)
    box = mn // per_row
    return box * bk * W + tma_box_offset(mode, per_row, esize, k, mn % per_row)


def stage_slice_desc(major: str, mode: str, rows: int, bk: int, esize: int, j: int, base: int) -> SmemDesc:
    """Descriptor of K slice j of a stage packed by ``stage_element_offset``.

    One MMA slice spans 32 bytes of K per row: 16 elements of a 16-bit type
    (kind::f16) or 32 of an 8-bit type (kind::f8f6f4). For MN-major operands
    the slice is that many K rows, i.e. kper / 8 bands of SBO.
    Without swizzle the 16 B cells are the atoms: K-major then needs LBO =
    the distance between K cells (one box, rows*16 B) and SBO = 128 B between
    8-row groups; MN-major needs SBO = one box (BK*16 B) between 8-element MN
    groups and LBO = 128 B between 8-row K bands.
    """
    W = swizzle_width(mode)
    kbytes = 32                 # K bytes per row consumed by one MMA
    kper = kbytes // esize      # K elements per MMA slice
    if major == "K":
        if mode == ATOM32:
            raise ValueError("the 32-byte-atom mode is read for MN-major operands only")
        off = j * kbytes
        start = base + (off // W) * rows * W + off % W
        lbo = rows * 16 if mode == "none" else 16
        return SmemDesc(start=start, lbo=lbo, sbo=8 * W, base_offset=0, swz=SWZ_CODE[mode])
    if mode == "none":
        return SmemDesc(start=base + j * (kper // 8) * 128, lbo=128, sbo=bk * 16, base_offset=0, swz=0)
    band = ATOM32_K_BAND if mode == ATOM32 else 8   # K rows between SBO steps
    # the slice's kper K rows start kper rows (of W bytes) into the box
    return SmemDesc(start=base + j * kper * W, lbo=bk * W, sbo=band * W, base_offset=0, swz=SWZ_CODE[mode])


# ---------------------------------------------------------------------------
# Instruction descriptor for kind::f16 (reading c2 above).
# ---------------------------------------------------------------------------

FMT_F16, FMT_BF16 = 0, 1        # kind::f16 A/B formats
FMT_E4M3, FMT_E5M2 = 0, 1       # kind::f8f6f4 A/B formats
DFMT_F16, DFMT_F32 = 0, 1


def encode_idesc(m: int, n: int, ab_fmt: int, d_fmt: int, a_mn_major: int, b_mn_major: int,
                 b_fmt: int | None = None) -> int:
    """Instruction descriptor; ``b_fmt`` defaults to A's format."""
    b_fmt = ab_fmt if b_fmt is None else b_fmt
    word = 0
    word |= (d_fmt & 3) << 4
    word |= (ab_fmt & 7) << 7
    word |= (b_fmt & 7) << 10
    word |= (a_mn_major & 1) << 15
    word |= (b_mn_major & 1) << 16
    word |= ((n >> 3) & 0x3F) << 17
    word |= ((m >> 4) & 0x1F) << 24
    return word


def legal_mma_n(cta_group: int, n: int) -> bool:
    """"06 Blackwell Tensor Core - tcgen05 MMA", cta_group section: f16/bf16 N ranges."""
    if cta_group == 1:
        return 8 <= n <= 256 and n % 8 == 0
    if cta_group == 2:
        return 16 <= n <= 256 and n % 16 == 0
    return False


# ---------------------------------------------------------------------------
# TMEM accumulator maps ("06 Blackwell Tensor Core - tcgen05 MMA",
# "How cta_group Sets the Operation Scope"). Each returns (cta, lane, col).
# ---------------------------------------------------------------------------

TMEM_LANES = 128
TMEM_COLS = 512


def tmem_cta1_m128(m: int, n: int) -> tuple[int, int, int]:
    return 0, m, n


def tmem_layout_f(m: int, n: int, align: int = 0) -> tuple[int, int, int]:
    if align not in (0, 16):
        raise ValueError("lane alignment is 0 or 16")
    return 0, (m // 16) * 32 + align + m % 16, n


def tmem_cta2_m256(m: int, n: int) -> tuple[int, int, int]:
    return m // 128, m % 128, n


def tmem_layout_b(m: int, n: int, N: int) -> tuple[int, int, int]:
    half = N // 2
    return m // 64, m % 64 + (64 if n >= half else 0), n % half


def tmem_ws(m: int, n: int, M: int, N: int) -> tuple[int, int, int]:
    """Accumulator map of the weight-stationary tcgen05.mma.ws (cta_group::1).

    The page lists .ws among the four choices that fix the accumulator layout
    but prints only the ordinary layouts. Reading (recorded with the other
    readings): for M = 128 the .ws accumulator is the M = 128 one (row m in
    lane m); for M = 32 and 64 the 128 lanes are filled by cutting N into
    4 / (M / 32) equal column parts. Lane quarter q holds row block q % (M/32)
    (rows 32 (q % (M/32)) .. +31) of column part q // (M/32), so every quarter
    holds whole 32-row blocks and the accumulator takes N / parts columns.
    """
    if M == 128:
        return 0, m, n
    if M not in (32, 64):
        raise ValueError(".ws accumulators have 32, 64 or 128 rows")
    row_blocks = M // 32
    width = N // (4 // row_blocks)
    q = (n // width) * row_blocks + m // 32
    return 0, 32 * q + m % 32, n % width


def tmem_two_half(m: int, n: int, N: int, half_col: int = 256) -> tuple[int, int, int]:
    """Accumulator map of a 256-row tile held by one CTA as two cta_group::1
    M = 128 MMAs on the same B slice (the page's M = 128 layout twice: rows
    0..127 in lanes 0..127 from column 0, rows 128..255 in the same lanes from
    column ``half_col``). The second half starts at a fixed column, not at N,
    so that N may be any width up to ``half_col``.
    """
    if not 0 < N <= half_col or half_col + N > TMEM_COLS:
        raise ValueError("both halves must fit the TMEM columns side by side")
    return 0, m % 128, (m // 128) * half_col + n


def tmem_warp_lanes(warp: int) -> range:
    """Lanes a warp may touch: warp w of a warpgroup owns lanes 32*(w%4) .. +31."""
    q = warp % 4
    return range(32 * q, 32 * q + 32)


# ---------------------------------------------------------------------------
# mbarrier ring ("Tensor Cores, layouts, and swizzling", 6.6.1): stage of
# iteration k is k % S and the parity to wait for is (k / S) & 1.
# ---------------------------------------------------------------------------


def ring_stage(k: int, S: int) -> int:
    return k % S


def ring_parity(k: int, S: int) -> int:
    return (k // S) & 1


# ---------------------------------------------------------------------------
# Global-to-shared traffic of a tiled GEMM when every output tile reloads
# its A row panel and B column panel ("Swizzling explained properly",
# "Output swizzle": each operand is copied dim / tile times).
# ---------------------------------------------------------------------------


def reload_traffic_bytes(M: int, N: int, K: int, BM: int, BN: int, esize: int) -> int:
    n_tiles_n = -(-N // BN)
    n_tiles_m = -(-M // BM)
    return n_tiles_n * M * K * esize + n_tiles_m * K * N * esize
