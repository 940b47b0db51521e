// Descriptor builder for tcgen05.mma operands.
//
// Shared-memory matrix descriptor ("LBO, SBO and SWZ for a tcgen05 tile",
// section 3): matrix start, leading-dimension byte offset (LBO) and stride
// byte offset (SBO) in 16-byte units, matrix base offset (MBO) and the
// swizzle code as raw 3-bit fields. Bit positions follow the public PTX
// description of the tcgen05 shared-memory descriptor (the page's field table
// did not survive): start [0,14), LBO [16,30), SBO [32,46), the fixed value
// 0b001 at [46,49), MBO [49,52), LBO mode 52, swizzle [61,64).
//
// Instruction descriptor for kind::f16 ("06 Blackwell Tensor Core - tcgen05
// MMA", "How tcgen05.mma Executes": idesc carries M, N, the A/B and D types
// and the operand majors): D format [4,6), A format [7,10), B format
// [10,13), A major 15, B major 16, N>>3 at [17,23), M>>4 at [24,29).
//
// Operand stage packing (what the producer's TMA boxes build, 1024-aligned):
//   K-major  (rows x BK): boxes of W/2 K-elements x rows, one after another
//            along K; each 8-row group of W-byte rows is one swizzle atom.
//            SBO = 8 W (next 8-row group), LBO unused (encoded 1), and the
//            K=16 slice j starts at (32 j / W) * rows * W + (32 j mod W).
//   MN-major (BK x rows): boxes of W/2 MN-elements x BK K-rows, one after
//            another along MN. LBO = BK W (next MN atom), SBO = 8 W (next
//            8-row K band; 4 W for the 32-byte-atom mode's 4-row bands), and
//            slice j starts at j * (32 / esize) * W.
// Without swizzle (bits 0, W = 16) the 16-byte core-matrix cells are the
// atoms: K-major LBO = rows * 16 (next K cell, one box away), SBO = 128 (next
// 8-row group); MN-major LBO = 128 (next 8-row K band), SBO = BK * 16 (next
// 8-element MN group, one box away).
// Stages start on 1024-byte boundaries, so MBO is always 0 (the start of a
// K slice inside a K-major row moves only bits below 128, page section 3).
#pragma once

#include <cstdint>

#ifndef G300_HD
#define G300_HD __host__ __device__ __forceinline__
#endif

namespace g300 {

// Swizzle "bits" B: 1 = 32 B, 2 = 64 B, 3 = 128 B rows of 16-byte atoms
// ("Swizzling explained properly": Swizzle<B,4,3>). The value kSwzAtom32
// stands for the 128-byte rows of 32-byte atoms (Swizzle<2,5,2>: the 32-byte
// unit of a row is XORed with the row index mod 4), descriptor code 1, read
// for MN-major operands whose K rows come in bands of kAtom32KBand. The GEMM
// kernels do not issue MMAs on such operands (a kind::f16 or kind::f8f6f4
// MMA reads them as zeros on GB300); the builder serves the inspection
// entry points.
constexpr int kSwzAtom32 = 4;
constexpr int kAtom32KBand = 4;

G300_HD uint32_t swizzle_row_bytes(int bits) { return bits == kSwzAtom32 ? 128u : 16u << bits; }

// Raw descriptor code of a swizzle mode (LBO/SBO page, section 4):
// none 0, SW32 6, SW64 4, SW128 2, 128 B with 32-byte atoms 1.
G300_HD uint32_t swizzle_code(int bits)
{
    return bits == kSwzAtom32 ? 1u : bits == 3 ? 2u : bits == 2 ? 4u : bits == 1 ? 6u : 0u;
}

G300_HD uint64_t make_smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                uint32_t swz_code)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // fixed 0b001
    d |= static_cast<uint64_t>(swz_code & 7u) << 61;
    return d;
}

struct OperandPacking {
    uint32_t lbo;
    uint32_t sbo;
    uint32_t swz;
};

G300_HD OperandPacking operand_packing(int mn_major, int swz_bits, int rows, int bk)
{
    const uint32_t W = swizzle_row_bytes(swz_bits);
    OperandPacking p;
    p.swz = swizzle_code(swz_bits);
    if (swz_bits == 0) {
        p.lbo = mn_major ? 128u : static_cast<uint32_t>(rows) * 16u;
        p.sbo = mn_major ? static_cast<uint32_t>(bk) * 16u : 128u;
        return p;
    }
    p.lbo = mn_major ? static_cast<uint32_t>(bk) * W : 16u;
    // SBO steps over one band of K rows (MN-major) or 8 rows (K-major); the
    // stage holds its rows contiguously, so a band is its rows times W
    p.sbo = static_cast<uint32_t>(swz_bits == kSwzAtom32 ? kAtom32KBand : 8) * W;
    return p;
}

// Byte offset of K slice j from the stage start. One MMA consumes 32 bytes of
// K per row: 16 elements of a 16-bit type (kind::f16) or 32 of an 8-bit type
// (kind::f8f6f4, esize 1). MN-major operands store one K row per W bytes
// (16 without swizzle), so a slice there is 32 / esize rows.
G300_HD uint32_t slice_byte_offset(int mn_major, int swz_bits, int rows, int j, int esize = 2)
{
    const uint32_t W = swizzle_row_bytes(swz_bits);
    if (mn_major)
        return static_cast<uint32_t>(j) * (32u / static_cast<uint32_t>(esize)) * W;
    const uint32_t off = 32u * static_cast<uint32_t>(j);
    return (off / W) * static_cast<uint32_t>(rows) * W + off % W;
}

// Instruction descriptor, fp32 accumulator. A/B format codes depend on the
// kind: kind::f16 0 = f16, 1 = bf16; kind::f8f6f4 0 = E4M3, 1 = E5M2.
G300_HD uint32_t make_idesc(int M, int N, int a_fmt, int b_fmt, int a_mn_major, int b_mn_major)
{
    uint32_t d = 0;
    d |= 1u << 4;  // D format: f32
    d |= static_cast<uint32_t>(a_fmt & 7) << 7;
    d |= static_cast<uint32_t>(b_fmt & 7) << 10;
    d |= static_cast<uint32_t>(a_mn_major & 1) << 15;
    d |= static_cast<uint32_t>(b_mn_major & 1) << 16;
    d |= static_cast<uint32_t>((N >> 3) & 0x3F) << 17;
    d |= static_cast<uint32_t>((M >> 4) & 0x1F) << 24;
    return d;
}

// Instruction descriptor of a block-scaled MMA (kind::mxf8f6f4, mxf4,
// mxf4nvf4): the same shape, format and major fields (E2M1 is format 1 in the
// fp4 kinds), the scale format at bit 23 (1 UE8M0, 0 UE4M3), and no D-format
// field: bits [4,6) and [29,31) carry the scale factor IDs of B and A (the
// first byte of each 32-bit scale column this MMA uses), added per MMA by
// idesc_sf_ids.
G300_HD uint32_t make_idesc_mx(int M, int N, int a_fmt, int b_fmt, int a_mn_major, int b_mn_major,
                               bool scale_ue8m0 = true)
{
    uint32_t d = 0;
    d |= static_cast<uint32_t>(a_fmt & 7) << 7;
    d |= static_cast<uint32_t>(b_fmt & 7) << 10;
    d |= static_cast<uint32_t>(a_mn_major & 1) << 15;
    d |= static_cast<uint32_t>(b_mn_major & 1) << 16;
    d |= static_cast<uint32_t>((N >> 3) & 0x3F) << 17;
    d |= (scale_ue8m0 ? 1u : 0u) << 23;
    d |= static_cast<uint32_t>((M >> 4) & 0x1F) << 24;
    return d;
}

G300_HD uint32_t idesc_sf_ids(uint32_t idesc, int a_sf_id, int b_sf_id)
{
    return idesc | (static_cast<uint32_t>(b_sf_id & 3) << 4) | (static_cast<uint32_t>(a_sf_id & 3) << 29);
}

G300_HD uint32_t make_idesc_f16(int M, int N, int in_bf16, int a_mn_major, int b_mn_major)
{
    return make_idesc(M, N, in_bf16, in_bf16, a_mn_major, b_mn_major);
}

}  // namespace g300
