// C ABI of the tcgen05 GEMM library: argument checks, TMA tensor-map
// encoding, kernel-variant choice and launch. Declarations and contracts are
// in include/gemm_gb300.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gemm_gb300.h"
#include "gemm_kernel.cuh"
#include "launch.cuh"
#include "variants.h"

using namespace g300;

namespace {

constexpr int kMaxDevices = 64;

// Device status word written by the kernels' bounded waits.
__device__ unsigned int g_status_word;

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_inject_timeout_ms{0};
std::atomic<int> g_inject_role{kRoleMma};
// Tag of the latest stream-K launch; a split tile's head accepts a partial
// sum only when the contributor's flag carries its own launch's tag.
std::atomic<uint32_t> g_sk_epoch{0};

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
unsigned int *g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

struct Variant {
    int cg, bn, bk, stages;
    bool grouped;
    int esize;
    int bm;
    int sf;  // scale kind (kScale*)
    int mode;  // kModeOrdinary, kModeWs (tcgen05.mma.ws) or kModeMcastB (B multicast in a 2-CTA cluster)
    cudaError_t (*launch)(const LaunchArgs &);
    cudaError_t (*resident)(int *);
    int resident_cache[kMaxDevices];
};

#define G300_VARIANT_ROW(CG, BN, BK, ST, GR, ES, BM, SF, MO) \
    {CG, BN, BK, ST, GR, ES, BM, SF, MO, &launch_gemm<CG, BN, BK, ST, GR, ES, BM, SF, MO>, &resident_ctas<CG, BN, BK, ST, GR, ES, BM, SF, MO>, {0}},
Variant g_variants[] = {G300_VARIANTS(G300_VARIANT_ROW)};
#undef G300_VARIANT_ROW

gemm_status_t cuda_fail(cudaError_t e)
{
    (void)e;
    return GEMM_ERR_CUDA;
}

gemm_status_t device_state(int *dev_out, unsigned int **status_out, int *sms_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return GEMM_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess)
            return GEMM_ERR_CUDA;
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        g_sms[dev] = sms;
    }
    *dev_out = dev;
    *status_out = g_status_ptr[dev];
    *sms_out = g_sms[dev];
    return GEMM_OK;
}

int resident_for(Variant &v, int dev)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (v.resident_cache[dev] == 0) {
        int n = 0;
        if (v.resident(&n) != cudaSuccess || n <= 0)
            n = -1;
        v.resident_cache[dev] = n;
    }
    return v.resident_cache[dev];
}

Variant *find_variant(int cg, int bn, int bk, bool grouped, int esize = 2, int bm = 128, int sf = kScaleNone,
                      int mode = kModeOrdinary)
{
    for (auto &v : g_variants)
        if (v.cg == cg && v.bn == bn && v.bk == bk && v.grouped == grouped && v.esize == esize && v.bm == bm &&
            v.sf == sf && v.mode == mode)
            return &v;
    return nullptr;
}

// Operand element type of a call: storage code for the tensor maps (0 fp16,
// 1 bf16, 2 bytes: fp8 or packed fp4), element size, the MMA format code of
// A and B, and the block-scale kind (kScale*).
struct InFmt {
    int dcode, esize, a_fmt, b_fmt;
    int sf;
};

InFmt fmt16(int in_bf16) { return InFmt{in_bf16, 2, in_bf16, in_bf16, kScaleNone}; }

InFmt fmt8(int a_fmt, int b_fmt) { return InFmt{2, 1, a_fmt, b_fmt, kScaleNone}; }

// TF32: fp32 words in memory (tensor-map type FLOAT32), MMA format code 2 in kind::tf32.
InFmt fmt32() { return InFmt{3, 4, 2, 2, kScaleNone}; }

// Block-scaled fp8: the same operand bytes plus E8M0 scale atoms.
InFmt fmtmx(int a_fmt, int b_fmt) { return InFmt{2, 1, a_fmt, b_fmt, kScaleMx8}; }

// Block-scaled fp4: packed E2M1 bytes (format code 1 in the fp4 kinds).
InFmt fmtfp4(int sf) { return InFmt{2, 1, 1, 1, sf}; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int out_bytes(int d_type) { return d_type == GEMM_OUT_F32 ? 4 : 2; }

CUtensorMapDataType out_dtype(int d_type)
{
    return d_type == GEMM_OUT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
           : d_type == GEMM_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

CUtensorMapSwizzle tma_swizzle(int bits)
{
    return bits == kSwzAtom32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B
           : bits == 3 ? CU_TENSOR_MAP_SWIZZLE_128B
           : bits == 2 ? CU_TENSOR_MAP_SWIZZLE_64B
           : bits == 1 ? CU_TENSOR_MAP_SWIZZLE_32B
                       : CU_TENSOR_MAP_SWIZZLE_NONE;
}

// Encoded tensor maps of recent calls, keyed on every encode argument: repeated
// GEMMs on the same buffers skip the driver's encode (a few microseconds each).
struct MapKey {
    const void *ptr;
    uint64_t inner, outer, stride;
    uint32_t box_inner, box_outer;
    int dt, swz, l2;
    bool operator==(const MapKey &o) const
    {
        return ptr == o.ptr && inner == o.inner && outer == o.outer && stride == o.stride &&
               box_inner == o.box_inner && box_outer == o.box_outer && dt == o.dt && swz == o.swz &&
               l2 == o.l2;
    }
};
constexpr int kMapCache = 32;
MapKey g_map_keys[kMapCache];
CUtensorMap g_map_vals[kMapCache];
int g_map_used = 0, g_map_next = 0;
std::mutex g_map_mu;

gemm_status_t encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner,
                        uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                        uint32_t box_outer, CUtensorMapSwizzle swz,
                        CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
{
    const MapKey key{ptr, inner, outer, row_stride_bytes, box_inner, box_outer, static_cast<int>(dt),
                     static_cast<int>(swz), static_cast<int>(l2)};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        for (int i = 0; i < g_map_used; ++i)
            if (g_map_keys[i] == key) {
                *m = g_map_vals[i];
                return GEMM_OK;
            }
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return GEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_map_keys[g_map_next] = key;
    g_map_vals[g_map_next] = *m;
    g_map_next = (g_map_next + 1) % kMapCache;
    if (g_map_used < kMapCache)
        ++g_map_used;
    return GEMM_OK;
}

// Operand tile map: boxes of one swizzled row (W/2 elements) along the
// contiguous dimension, `rows` (K-major) or `bk` (MN-major) along the other.
gemm_status_t encode_operand(CUtensorMap *m, int dcode, const void *ptr, int mn_major,
                             int swz_bits, int64_t mn_total, int64_t k_total, int64_t ld, int rows,
                             int bk)
{
    const CUtensorMapDataType dt = dcode == 3   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dcode == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dcode == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint32_t esize = dcode == 3 ? 4u : dcode == 2 ? 1u : 2u;
    const uint32_t per = swizzle_row_bytes(swz_bits) / esize;
    if (!mn_major)
        return encode_2d(m, dt, ptr, static_cast<uint64_t>(k_total), static_cast<uint64_t>(mn_total),
                         static_cast<uint64_t>(ld) * esize, per, static_cast<uint32_t>(rows),
                         tma_swizzle(swz_bits));
    return encode_2d(m, dt, ptr, static_cast<uint64_t>(mn_total), static_cast<uint64_t>(k_total),
                     static_cast<uint64_t>(ld) * esize, per, static_cast<uint32_t>(bk),
                     tma_swizzle(swz_bits));
}

// Scale-atom map of a block-scaled operand: the atoms viewed as rows of 256
// bytes (atom a = rows 2a, 2a + 1); one box holds the `groups` consecutive
// atoms a stage of the kernel needs for one row block.
gemm_status_t encode_scales(CUtensorMap *m, const void *ptr, int64_t rows, int64_t k_bytes, int sf, int groups)
{
    const int64_t per = sf_atom_kbytes(sf);
    const uint64_t atoms = static_cast<uint64_t>((rows + 127) / 128) * static_cast<uint64_t>((k_bytes + per - 1) / per);
    return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, 256, 2 * atoms, 256, 256,
                     static_cast<uint32_t>(2 * groups), CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Output (and C) map: boxes of 128 bytes x the rows one epilogue warp owns
// (32 for 128-row tiles, 16 for 64-row tiles).
gemm_status_t encode_output(CUtensorMap *m, int d_type, const void *ptr, int64_t M, int64_t N,
                            int64_t ld, int epi_swizzle, int rows = 32)
{
    const int ob = out_bytes(d_type);
    return encode_2d(m, out_dtype(d_type), ptr, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                     static_cast<uint64_t>(ld) * ob, static_cast<uint32_t>(128 / ob), static_cast<uint32_t>(rows),
                     epi_swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

struct Plan {
    int cg, bn, bk;
    int bm;  // accumulator rows per CTA: 128, 64 (M = 64 MMAs) or 32 (.ws only)
    int ws;  // 1: tcgen05.mma.ws
    int mcb;  // 1: clusters of two cta_group::1 CTAs sharing B by TMA multicast
    int a_swz, b_swz;
    int epi_swizzle;
    int max_ctas;
    int group_m;
    unsigned long long timeout_ns;
    int flags;
    unsigned long long *stats;
    int stream_k;
    void *workspace;
    size_t workspace_bytes;
};

// CTAs per cluster of a plan: CTA pairs and B-multicast clusters have two.
int cluster_ctas(const Plan &pl) { return (pl.cg == 2 || pl.mcb) ? 2 : 1; }

// gemm_swizzle_t -> swizzle bits (B of Swizzle<B,4,3>): 32B 1, 64B 2, 128B 3, none 0;
// 128B with 32-byte atoms kSwzAtom32.
int swz_bits_of(int opt)
{
    return opt == GEMM_SWIZZLE_NONE ? 0 : opt == GEMM_SWIZZLE_128B_ATOM32 ? kSwzAtom32 : opt;
}

// Choose the tile configuration; fills `plan` or returns an error for options
// the compiled kernel variants cannot honour.
gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, int a_mn, int b_mn, int sms,
                        const gemm_options_t *o, bool grouped, Plan *plan, int esize = 2, int sf = kScaleNone)
{
    gemm_options_t opt = {};
    if (o)
        opt = *o;
    if (opt.cta_group < 0 || opt.cta_group > 2 || opt.tile_n < 0 || opt.swizzle_a < 0 ||
        opt.swizzle_a > 5 || opt.swizzle_b < 0 || opt.swizzle_b > 5 || opt.max_ctas < 0 ||
        opt.group_m < 0 || opt.timeout_ms < 0 || opt.epilogue_swizzle < -1 ||
        opt.epilogue_swizzle > 1 || opt.flags < 0 || opt.flags > 127 || opt.block_k < 0 ||
        opt.stream_k < -1 || opt.stream_k > 3 || opt.mma_ws < -1 || opt.mma_ws > 1 || opt.multicast_b < -1 ||
        opt.multicast_b > 1)
        return GEMM_ERR_INVALID_ARG;
    if (opt.workspace && (reinterpret_cast<uintptr_t>(opt.workspace) & 255u) != 0)
        return GEMM_ERR_ALIGNMENT;

    if (opt.tile_m != 0 && opt.tile_m != 32 && opt.tile_m != 64 && opt.tile_m != 128 && opt.tile_m != 256)
        return GEMM_ERR_INVALID_ARG;
    int cg = opt.cta_group;
    if ((opt.tile_m == 64 || opt.tile_m == 32 || opt.tile_m == 256) && cg == 2)
        return GEMM_ERR_UNSUPPORTED;
    if (opt.tile_m == 64 || opt.tile_m == 32 || opt.tile_m == 256)
        cg = 1;
    if (cg == 0) {
        // CTA pairs for large problems: each SM then loads half of B.
        cg = (!grouped && M >= 2048 && N >= 2048) ? 2 : 1;
    }
    int bn = opt.tile_n;
    if (bn == 0 && opt.tile_m == 256) {
        bn = 256;  // the only width two-half tiles are built for
    } else if (bn == 0) {
        if (cg == 2) {
            bn = N <= 128 ? 128 : 256;
        } else {
            // 256-wide tiles when they still fill every SM and waste little of N;
            // otherwise 128 (measured faster than 64 even where 64 would give more
            // tiles than SMs: a 64-wide tile moves half the bytes per pipeline
            // stage for the same fixed per-stage cost)
            const int64_t tiles_m = (M + 127) / 128;
            const int64_t tn256 = (N + 255) / 256;
            const bool fill256 = tiles_m * tn256 >= sms && tn256 * 256 <= N + N / 8;
            bn = fill256 ? 256 : (N > 64 ? 128 : 64);
        }
    }
    // K block per stage: the per-stage cost of a TMA refill is nearly fixed, so
    // the deepest stages that still leave three of them in flight win; the
    // 128 x 256 single-CTA tile keeps BK = 64 to hold four stages.
    int bk = opt.block_k;
    if (bk == 0) {
        if (esize == 1)
            bk = (cg == 1 && bn == 256) ? 128 : 256;  // the same stage bytes as bf16
        else if (esize == 4)
            bk = (cg == 1 && bn == 256) ? 32 : 64;
        else if (!grouped && cg == 1 && bn == 128 && K <= 32 && opt.tile_n == 0)
            bk = 32;
        else
            bk = (cg == 1 && (bn == 256 || opt.tile_m == 256)) ? 64 : 128;  // two-half tiles: 64
    }
    // 64-row tiles (M = 64 MMAs) when asked, or for problems of at most 64 rows
    // (compiled for 128- and 256-wide N tiles)
    int bm = opt.tile_m ? opt.tile_m
                        : (cg == 1 && M <= 64 && esize == 2 && !grouped && bn >= 128 ? 64 : 128);
    if (bm == 64 && opt.block_k == 0)
        bk = bn == 256 ? 64 : 128;
    // Two-half tiles (256 rows on one CTA: two M = 128 MMAs per B slice, half
    // the operand bytes per flop of a 128 x 256 tile) for large single-CTA
    // 16-bit problems with long K. Measured, TFLOP/s, 128 x 256 (B multicast
    // where that is the default) -> 256 x 256: 8192^3 1666 -> 1843, 8192^3
    // MN-major 1482 -> 1697, 6144^3 1580 -> 1699, 3072^2 x 8192 1283 -> 1390,
    // 4096^3 1360 -> 1389, 4096^3 K/MN 1258 -> 1307; K = 2048 (8192^2) 1423 ->
    // 1344, where the epilogue, which no longer overlaps, weighs more.
    if (opt.tile_m == 0 && cg == 1 && esize == 2 && !grouped && sf == kScaleNone && bm == 128 &&
        (opt.tile_n == 0 || opt.tile_n == 256) && (opt.block_k == 0 || opt.block_k == 64) && opt.mma_ws != 1 &&
        M >= 2048 && N >= 2048 && K >= 4096 && find_variant(1, 256, 64, false, 2, 256)) {
        bm = 256;
        bn = 256;
        bk = 64;
        // 224 wide instead when that takes fewer column-rounds of the grid
        // (the time of a round goes with the tile width): 4096^2 is 128
        // B-sharing cluster tiles of 512 x 256 on 76 clusters, two rounds for
        // 1.68 waves of work, but exactly two rounds of 304 tiles of 256 x 224
        // on 152 CTAs. 224-wide tiles keep their own B: sharing it measured
        // slower there (4096^3, TFLOP/s: 256 wide shared 1389, 224 wide shared
        // 1449, 224 wide own 1481). A and B K-major only: with MN-major B 224 own
        // measured 941-954 against 1411-1418 for 256 shared, with MN-major A
        // 1259 against 1360.
        if (opt.tile_n == 0 && opt.multicast_b != 1 && !a_mn && !b_mn && find_variant(1, 224, 64, false, 2, 256)) {
            auto rounds = [&](int64_t rows, int64_t w, int64_t units) {
                const int64_t tiles = ((M + rows - 1) / rows) * ((N + w - 1) / w);
                return (tiles + units - 1) / units;
            };
            const bool shared256 = opt.multicast_b != -1;
            const int64_t r256 = shared256 ? rounds(512, 256, sms / 2) : rounds(256, 256, sms);
            if (rounds(256, 224, sms) * 224 < r256 * 256)
                bn = 224;
        }
    }
    // Weight-stationary tiles (tcgen05.mma.ws): 32 rows (M = 32 exists only in
    // the .ws form) when asked for, or 64 rows; single CTAs, 16-bit operands,
    // single problems. 32-row tiles are 256 wide so that each epilogue warp
    // holds whole 64-column chunks of its column part. The .ws form is the
    // default for the 64 x 128 tiles of M <= 64 (32 x 16384 x 8192: 0.79 of
    // the measured HBM rate against 0.77 for Layout F and 0.71 for 32 x 256
    // .ws tiles); an explicit tile_m 64 keeps the page's Layout F.
    int ws = 0;
    const bool ws_default = opt.mma_ws == 0 && opt.tile_m == 0 && bm == 64 && bn == 128;
    if (opt.tile_m == 32 || opt.mma_ws == 1 || ws_default) {
        if (opt.mma_ws == -1 || opt.tile_m >= 128 || sf != kScaleNone || esize != 2 || grouped || cg != 1)
            return GEMM_ERR_UNSUPPORTED;
        ws = 1;
        bm = opt.tile_m ? opt.tile_m : 64;
        if (bm == 32)
            bn = opt.tile_n ? opt.tile_n : 256;
        if (opt.block_k == 0)
            bk = bn == 256 ? 64 : 128;
    }
    if (sf != kScaleNone) {
        // Block-scaled tiles: 256 x 256 CTA pairs with one accumulator buffer
        // (the default from 2048 rows and columns; MXFP8 8192^3 2588 against
        // 1897 TFLOP/s for single CTAs), single CTAs of 128 x 128, and MXFP8
        // pairs of 256 x 128 (1773). K bytes per stage: MXFP8 256 (single CTAs
        // also 128), NVFP4 128, MXFP4 256 (pairs also 128); the variant lookup
        // below refuses anything else. A 128-byte fp4 stage on a pair holds
        // four MMAs, less tensor work than the MMA thread needs to issue a
        // stage, so MXFP4 pairs default to 256 bytes.
        if (opt.tile_m && opt.tile_m != 128)
            return GEMM_ERR_UNSUPPORTED;
        auto depth = [&](int) { return sf == kScaleNv4 ? 128 : 256; };
        const bool wide = opt.cta_group == 0 && opt.tile_n == 0 && M >= 2048 && N >= 2048;
        cg = opt.cta_group ? opt.cta_group : (wide ? 2 : 1);
        bn = opt.tile_n ? opt.tile_n : (cg == 2 && (wide || sf != kScaleMx8) ? 256 : 128);
        bk = opt.block_k ? opt.block_k : depth(cg);
        bm = 128;
        if (wide && !find_variant(cg, bn, bk, grouped, esize, bm, sf)) {
            cg = 1;  // a stage depth only single CTAs are built for
            bn = 128;
        }
    }
    // B multicast between two single-CTA tiles of one cluster: when asked for,
    // and by default for 128 x 256 single-CTA tiles whose B is MN-major or
    // whose operands overflow L2 (measured, TFLOP/s without -> with: 8192^3
    // K/MN fp32 out + C 914 -> 1452, 4096^3 K/MN 815 -> 1175, 8192^3 K/K
    // 1599 -> 1665, 6144^3 K/K 1383 -> 1433; 4096^3 and 8192^2 x 2048 K/K,
    // operands in L2: within 1 %)
    int mcb = 0;
    if (opt.multicast_b == 1) {
        // each CTA loads half of B: for MN-major B, whole swizzle atoms of it
        if (cg != 1 || (bm != 128 && bm != 256) || ws || sf != kScaleNone || grouped || (b_mn && bn % 256 != 0))
            return GEMM_ERR_UNSUPPORTED;
        mcb = 1;
    } else if (opt.multicast_b == 0 && cg == 1 && bm == 128 && bn == 256 && !ws && sf == kScaleNone && !grouped &&
               M > 128 && (b_mn || (M + N) * K * esize > (static_cast<int64_t>(128) << 20)) &&
               find_variant(cg, bn, bk, grouped, esize, bm, sf, kModeMcastB)) {
        mcb = 1;
    } else if (opt.multicast_b == 0 && bm == 256 && bn == 256 && M > 256 && !grouped &&
               find_variant(cg, bn, bk, grouped, esize, bm, sf, kModeMcastB)) {
        // two-half tiles share B in pairs of CTAs by default (measured, TFLOP/s
        // without -> with: 4096^3 1389 -> 1404-1417, K/MN 1295-1307 -> 1418,
        // 6144^3 1738 -> 1758-1765, 8192^3 1856-1862 -> 1888, MN/MN 1700 -> 1791)
        mcb = 1;
    }
    const int mode = ws ? kModeWs : mcb ? kModeMcastB : kModeOrdinary;
    if (!find_variant(cg, bn, bk, grouped, esize, bm, sf, mode))
        return GEMM_ERR_UNSUPPORTED;

    // the widest swizzle whose row fits the stage: along K for K-major
    // operands, along the tile's MN extent for MN-major ones
    auto pick_swz = [&](int requested, int mn_major, int rows) -> int {
        if (requested)
            return swz_bits_of(requested);
        if (esize == 4 && mn_major)
            return kSwzAtom32;  // the MN-major layout kind::tf32 reads
        // widest row that divides the extent (a 192-byte K stage takes 64-byte rows)
        const int span = (mn_major ? rows : bk) * esize;
        return span % 128 == 0 ? 3 : span % 64 == 0 ? 2 : 1;
    };
    plan->cg = cg;
    plan->bn = bn;
    plan->bk = bk;
    plan->a_swz = pick_swz(opt.swizzle_a, a_mn, bm);
    plan->b_swz = pick_swz(opt.swizzle_b, b_mn, bn / cg);
    // a K-major swizzled row may not be wider than the K block; an MN-major
    // atom may not be wider than the tile's MN extent. MN-major operands of
    // kind::tf32 take the 32-byte-atom mode and no other (on GB300 an MN-major
    // TF32 operand in SW128 reads as zeros), and 16- and 8-bit operands never
    // take it (kind::f16 and kind::f8f6f4 read it as zeros)
    auto fits = [&](int bits, int mn_major, int rows) {
        if ((bits == kSwzAtom32) != (esize == 4 && mn_major != 0))
            return false;
        const int per = static_cast<int>(swizzle_row_bytes(bits)) / esize;
        return mn_major ? (rows % per == 0) : (bk % per == 0);
    };
    if (!fits(plan->a_swz, a_mn, bm) || !fits(plan->b_swz, b_mn, bn / cg))
        return GEMM_ERR_UNSUPPORTED;
    plan->bm = bm;
    plan->ws = ws;
    plan->mcb = mcb;
    plan->epi_swizzle = opt.epilogue_swizzle == -1 ? 0 : 1;
    plan->max_ctas = opt.max_ctas;
    plan->group_m = opt.group_m ? opt.group_m : 8;
    plan->timeout_ns = static_cast<unsigned long long>(opt.timeout_ms ? opt.timeout_ms : 2000) * 1000000ull;
    plan->flags = opt.flags;
    // Problems of at most one wave of tiles with long K stream their operands
    // from HBM (each tile reads its own panel once): every CTA then starts its
    // K loop at its own offset, so that the CTAs do not all request the same
    // columns of their row panels at the same moment (16384 x 128 x 8192:
    // 0.70 -> 0.75 of the measured HBM rate). Explicit flags are kept as given.
    if (opt.flags == 0 && !grouped) {
        const int64_t rows = static_cast<int64_t>(bm) * (mcb ? 2 : cg);
        const int64_t tiles = ((M + rows - 1) / rows) * ((N + bn - 1) / bn);
        const int64_t kblocks = (K + bk - 1) / bk;
        if (tiles <= sms / (mcb ? 2 : cg) && kblocks >= 16)
            plan->flags |= kFlagRotateK;
    }
    plan->stats = opt.stats;
    plan->stream_k = opt.stream_k;
    plan->workspace = opt.workspace;
    plan->workspace_bytes = opt.workspace_bytes;
    return GEMM_OK;
}

// Stream-K workspace: a row of 4 flags per CTA, then one rows x BN fp32
// partial-sum slot per CTA (rows 128, or 256 for two-half tiles).
size_t sk_flag_bytes(int ctas) { return (static_cast<size_t>(ctas) * 4 * sizeof(uint32_t) + 1023) & ~size_t(1023); }

size_t sk_bytes(int ctas, int bn, int rows)
{
    return sk_flag_bytes(ctas) + static_cast<size_t>(ctas) * rows * bn * sizeof(float);
}

// Stream-K split of `tiles` tiles of `kbt` K blocks over `clusters` clusters:
// the number of tiles that stay data-parallel, or -1 for no split.
int64_t sk_split(int mode, int64_t tiles, int64_t clusters, int64_t kbt)
{
    if (mode < 0 || kbt <= 0 || clusters <= 1)
        return -1;
    // auto: a ragged last wave after at least two full ones (fewer tiles than
    // that leave split tiles whose short head pieces cannot hide the gather of
    // partial sums; eight waves or more lose little to the ragged one)
    if (mode == 0 && (tiles % clusters == 0 || tiles < 2 * clusters || tiles >= 8 * clusters))
        return -1;
    int64_t sk = tiles;
    if (mode == 3 && tiles > clusters)
        sk = tiles % clusters ? tiles % clusters : clusters;  // the ragged wave alone
    else if (mode != 2 && tiles >= 2 * clusters)
        sk = clusters + tiles % clusters;  // the ragged wave and one full wave
    if (sk * kbt < clusters)
        return -1;  // fewer K blocks than clusters: some would have no work
    return tiles - sk;
}

int grid_for(const Plan &pl, Variant &v, int dev, int sms, int64_t tiles)
{
    int cap = resident_for(v, dev);
    if (cap <= 0)
        cap = sms;
    if (pl.max_ctas > 0)
        cap = std::min(cap, pl.max_ctas);
    const int64_t per_cluster = cluster_ctas(pl);
    int64_t clusters = std::min<int64_t>(tiles, cap / per_cluster);
    if (clusters < 1)
        clusters = 1;
    return static_cast<int>(clusters * per_cluster);
}

void fill_common(KParams &p, const Plan &pl, const InFmt &f, int a_mn, int b_mn, int d_type,
                 float alpha, float beta, unsigned int *status)
{
    p.alpha = alpha;
    p.beta = beta;
    p.a_mn = a_mn;
    p.b_mn = b_mn;
    p.a_swz = pl.a_swz;
    p.b_swz = pl.b_swz;
    p.a_fmt = f.a_fmt;
    p.b_fmt = f.b_fmt;
    p.out_type = d_type;
    p.epi_swizzle = pl.epi_swizzle;
    p.group_m = pl.group_m;
    p.timeout_ns = pl.timeout_ns;
    p.flags = pl.flags;
    p.stats = pl.stats;
    p.status = status;
    const int inj = g_inject_timeout_ms.exchange(0);
    p.inject_timeout = inj > 0 ? g_inject_role.load() : 0;
    if (inj > 0)
        p.timeout_ns = static_cast<unsigned long long>(inj) * 1000000ull;
}

bool valid_enum(int major) { return major == GEMM_K_MAJOR || major == GEMM_MN_MAJOR; }

// Checks shared by single and grouped problems.
gemm_status_t check_problem(int64_t M, int64_t N, int64_t K, const void *A, int a_mn, int64_t lda,
                            const void *B, int b_mn, int64_t ldb, const void *C, int64_t ldc,
                            const void *D, int64_t ldd, int d_type, float beta, int esize = 2)
{
    const int64_t lim = (static_cast<int64_t>(1) << 31) - 1;
    if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim)
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return GEMM_OK;
    const int ob = out_bytes(d_type);
    if (!D || ldd < N)
        return GEMM_ERR_INVALID_ARG;
    if (!aligned16(D) || (ldd * ob) % 16 != 0 || ldd * ob >= (static_cast<int64_t>(1) << 40))
        return GEMM_ERR_ALIGNMENT;
    if (K > 0) {
        if (!A || !B)
            return GEMM_ERR_INVALID_ARG;
        if (lda < (a_mn ? M : K) || ldb < (b_mn ? N : K))
            return GEMM_ERR_INVALID_ARG;
        if (!aligned16(A) || !aligned16(B) || (lda * esize) % 16 != 0 || (ldb * esize) % 16 != 0 ||
            lda * esize >= (static_cast<int64_t>(1) << 40) || ldb * esize >= (static_cast<int64_t>(1) << 40))
            return GEMM_ERR_ALIGNMENT;
    }
    if (beta != 0.0f) {
        if (!C || ldc < N)
            return GEMM_ERR_INVALID_ARG;
        if (!aligned16(C) || (ldc * ob) % 16 != 0 || ldc * ob >= (static_cast<int64_t>(1) << 40))
            return GEMM_ERR_ALIGNMENT;
    }
    return GEMM_OK;
}

gemm_status_t run_single(const InFmt &f, int64_t M, int64_t N, int64_t K, const void *A, int a_major,
                         int64_t lda, const void *B, int b_major, int64_t ldb, const void *C,
                         int64_t ldc, void *D, int64_t ldd, int d_type, float alpha, float beta,
                         const gemm_options_t *opts, cudaStream_t stream, const void *sfa = nullptr,
                         const void *sfb = nullptr)
{
    if (!valid_enum(a_major) || !valid_enum(b_major) || d_type < 0 || d_type > 2)
        return GEMM_ERR_INVALID_ARG;
    const int a_mn = a_major, b_mn = b_major;
    gemm_status_t s = check_problem(M, N, K, A, a_mn, lda, B, b_mn, ldb, C, ldc, D, ldd, d_type, beta, f.esize);
    if (s != GEMM_OK || M == 0 || N == 0)
        return s;
    if (f.sf != kScaleNone && K > 0) {
        if (!sfa || !sfb)
            return GEMM_ERR_INVALID_ARG;
        if (!aligned16(sfa) || !aligned16(sfb))
            return GEMM_ERR_ALIGNMENT;
    }
    int dev = 0, sms = 0;
    unsigned int *status = nullptr;
    if ((s = device_state(&dev, &status, &sms)) != GEMM_OK)
        return s;
    Plan pl;
    if ((s = make_plan(M, N, K, a_mn, b_mn, sms, opts, false, &pl, f.esize, f.sf)) != GEMM_OK)
        return s;
    Variant *v = find_variant(pl.cg, pl.bn, pl.bk, false, f.esize, pl.bm, f.sf,
                              pl.ws ? kModeWs : pl.mcb ? kModeMcastB : kModeOrdinary);
    const int ccta = cluster_ctas(pl);
    // output rows one epilogue warp stores per chunk (two-half tiles: per half)
    const int epi_rows = (pl.ws || pl.bm == 256) ? 32 : pl.bm / 4;

    LaunchArgs la;
    std::memset(&la, 0, sizeof(la));
    if (K > 0) {
        if ((s = encode_operand(&la.a, f.dcode, A, a_mn, pl.a_swz, M, K, lda, pl.bm, pl.bk)) != GEMM_OK)
            return s;
        // B rows (K-major boxes) one CTA loads: half the tile for pairs and for B multicast
        if ((s = encode_operand(&la.b, f.dcode, B, b_mn, pl.b_swz, N, K, ldb, pl.bn / ccta, pl.bk)) != GEMM_OK)
            return s;
    }
    if ((s = encode_output(&la.d, d_type, D, M, N, ldd, pl.epi_swizzle, epi_rows)) != GEMM_OK)
        return s;
    if (beta != 0.0f) {
        if ((s = encode_output(&la.c, d_type, C, M, N, ldc, pl.epi_swizzle, epi_rows)) != GEMM_OK)
            return s;
    } else {
        la.c = la.d;
    }
    KParams &p = la.p;
    std::memset(&p, 0, sizeof(p));
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((M + pl.bm * ccta - 1) / (pl.bm * ccta));
    p.tiles_n = static_cast<int>((N + pl.bn - 1) / pl.bn);
    const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    if (tiles >= (static_cast<int64_t>(1) << 31))
        return GEMM_ERR_UNSUPPORTED;
    p.num_tiles = static_cast<int>(tiles);
    fill_common(p, pl, f, a_mn, b_mn, d_type, alpha, beta, status);
    p.c_ptr = beta != 0.0f ? C : nullptr;
    p.ldc = ldc;
    p.d_ptr = D;
    p.ldd = ldd;
    if (f.sf != kScaleNone && K > 0) {
        const int groups = pl.bk / sf_atom_kbytes(f.sf);  // atoms per stage and row block
        if ((s = encode_scales(&la.sfa, sfa, M, K, f.sf, groups)) != GEMM_OK ||
            (s = encode_scales(&la.sfb, sfb, N, K, f.sf, groups)) != GEMM_OK)
            return s;
        p.sf_groups = static_cast<int>((K + sf_atom_kbytes(f.sf) - 1) / sf_atom_kbytes(f.sf));
    }
    la.grid = grid_for(pl, *v, dev, sms, tiles);
    // stream-K: 128-row tiles gather partial sums in a spare accumulator buffer
    // (none for block-scaled 256-wide tiles); two-half tiles add them per chunk
    if (pl.workspace && (pl.bm == 128 || pl.bm == 256) && K > 0 && !(f.sf != kScaleNone && pl.bn == 256)) {
        // stream-K runs on every resident cluster
        const int full = grid_for(pl, *v, dev, sms, static_cast<int64_t>(1) << 40);
        const int64_t kbt = (K + pl.bk - 1) / pl.bk;
        // two-half tiles add the partial sums in the head's epilogue, chunk by
        // chunk: measured slower than the unsplit launch (4096^3 105 against
        // 97 us, 6144^3 308 against 266 us), so only an explicit mode splits them
        const int mode = (pl.bm == 256 && pl.stream_k == 0) ? -1 : pl.stream_k;
        const int64_t dp = sk_split(mode, tiles, full / ccta, kbt);
        if (dp >= 0) {
            if (pl.workspace_bytes < sk_bytes(full, pl.bn, pl.bm == 256 ? 256 : 128))
                return GEMM_ERR_INVALID_ARG;
            uint32_t epoch = g_sk_epoch.fetch_add(1) + 1;
            if (epoch == 0)
                epoch = g_sk_epoch.fetch_add(1) + 1;
            la.grid = full;
            p.sk_dp_tiles = static_cast<int>(dp);
            p.kb_per_tile = static_cast<int>(kbt);
            p.sk_iters = (tiles - dp) * kbt;
            p.sk_flags = static_cast<uint32_t *>(pl.workspace);
            p.sk_partials = reinterpret_cast<float *>(static_cast<unsigned char *>(pl.workspace) + sk_flag_bytes(full));
            p.sk_epoch = epoch;
        }
    }
    la.stream = stream;
    cudaError_t e = v->launch(la);
    if (e != cudaSuccess)
        return cuda_fail(e);
    g_launches.fetch_add(1);
    return GEMM_OK;
}

// Device-side problem table followed by four tensor maps per problem.
size_t table_bytes(int n) { return (static_cast<size_t>(n) * sizeof(GroupedProblemDev) + 127) & ~size_t(127); }

// A validated, planned grouped call, before its table exists anywhere.
struct GroupedCall {
    int in_bf16, a_mn, b_mn, d_type;
    float alpha, beta;
    int dev, sms;
    unsigned int *status;
    Plan pl;
    Variant *v;
};

// Argument checks of every problem, then the plan shared by all of them
// (from the largest M, N and K of the list).
gemm_status_t plan_grouped(int in_bf16, const gemm_problem_t *probs, int n, int a_major, int b_major, int d_type,
                           float alpha, float beta, const gemm_options_t *opts, GroupedCall *gc)
{
    const int a_mn = a_major, b_mn = b_major;
    int64_t maxM = 0, maxN = 0, maxK = 0;
    for (int i = 0; i < n; ++i) {
        const gemm_problem_t &q = probs[i];
        gemm_status_t s = check_problem(q.M, q.N, q.K, q.A, a_mn, q.lda, q.B, b_mn, q.ldb, q.C, q.ldc,
                                        q.D, q.ldd, d_type, beta);
        if (s != GEMM_OK)
            return s;
        maxM = std::max(maxM, q.M);
        maxN = std::max(maxN, q.N);
        maxK = std::max(maxK, q.K);
    }
    gemm_status_t s = device_state(&gc->dev, &gc->status, &gc->sms);
    if (s != GEMM_OK)
        return s;
    gemm_options_t o = {};
    if (opts)
        o = *opts;
    // CTA pairs for lists of wide problems, as for single ones (64 problems of
    // M_i in 128..4096, N = 4096, K = 2048: 1651 against 1596 TFLOP/s for
    // single CTAs); single CTAs otherwise
    if (o.cta_group == 0)
        o.cta_group = (maxN >= 2048 && maxM >= 256) ? 2 : 1;
    if (o.tile_n == 0)  // grouped pairs are built for 256-wide tiles only
        o.tile_n = (maxN >= 192 || o.cta_group == 2) ? 256 : 128;
    if ((s = make_plan(maxM, maxN, maxK, a_mn, b_mn, gc->sms, &o, true, &gc->pl)) != GEMM_OK)
        return s;
    gc->v = find_variant(gc->pl.cg, gc->pl.bn, gc->pl.bk, true);
    gc->in_bf16 = in_bf16;
    gc->a_mn = a_mn;
    gc->b_mn = b_mn;
    gc->d_type = d_type;
    gc->alpha = alpha;
    gc->beta = beta;
    return GEMM_OK;
}

// Writes the problem table and the tensor maps of `n` problems into the host
// buffer `img` (table_bytes(n) + n * 4 maps, zeroed by the caller) and counts
// the tiles of the launch.
gemm_status_t build_grouped_image(const GroupedCall &gc, const gemm_problem_t *probs, int n, unsigned char *img,
                                  int64_t *tiles_out)
{
    const Plan &pl = gc.pl;
    const int dcode = fmt16(gc.in_bf16).dcode;
    auto *table = reinterpret_cast<GroupedProblemDev *>(img);
    auto *maps = reinterpret_cast<CUtensorMap *>(img + table_bytes(n));
    int64_t tiles = 0;
    gemm_status_t s = GEMM_OK;
    for (int i = 0; i < n; ++i) {
        const gemm_problem_t &q = probs[i];
        GroupedProblemDev &g = table[i];
        g.M = static_cast<int>(q.M);
        g.N = static_cast<int>(q.N);
        g.K = static_cast<int>(q.K);
        const bool empty = q.M == 0 || q.N == 0;
        g.tiles_m = empty ? 0 : static_cast<int>((q.M + 128 * pl.cg - 1) / (128 * pl.cg));
        g.tiles_n = empty ? 0 : static_cast<int>((q.N + pl.bn - 1) / pl.bn);
        g.tile_start = static_cast<int>(tiles);
        tiles += static_cast<int64_t>(g.tiles_m) * g.tiles_n;
        if (tiles >= (static_cast<int64_t>(1) << 31))
            return GEMM_ERR_UNSUPPORTED;
        if (empty)
            continue;
        CUtensorMap *m = maps + 4 * i;
        if (q.K > 0) {
            if ((s = encode_operand(&m[0], dcode, q.A, gc.a_mn, pl.a_swz, q.M, q.K, q.lda, 128, pl.bk)) != GEMM_OK)
                return s;
            if ((s = encode_operand(&m[1], dcode, q.B, gc.b_mn, pl.b_swz, q.N, q.K, q.ldb, pl.bn / pl.cg, pl.bk)) !=
                GEMM_OK)
                return s;
        }
        if ((s = encode_output(&m[3], gc.d_type, q.D, q.M, q.N, q.ldd, pl.epi_swizzle)) != GEMM_OK)
            return s;
        if (gc.beta != 0.0f) {
            if ((s = encode_output(&m[2], gc.d_type, q.C, q.M, q.N, q.ldc, pl.epi_swizzle)) != GEMM_OK)
                return s;
        } else {
            m[2] = m[3];
        }
    }
    *tiles_out = tiles;
    return GEMM_OK;
}

// Copies the image (pageable source: staged before cudaMemcpyAsync returns)
// to `ws` on `stream` and launches the grouped kernel that reads it there.
gemm_status_t upload_and_launch_grouped(const GroupedCall &gc, int n, int64_t tiles, const unsigned char *img,
                                        size_t img_bytes, unsigned char *ws, cudaStream_t stream)
{
    cudaError_t e = cudaMemcpyAsync(ws, img, img_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return cuda_fail(e);
    LaunchArgs la;
    std::memset(&la, 0, sizeof(la));
    KParams &p = la.p;
    p.num_tiles = static_cast<int>(tiles);
    p.problems = reinterpret_cast<const GroupedProblemDev *>(ws);
    p.maps = reinterpret_cast<const CUtensorMap *>(ws + table_bytes(n));
    p.num_problems = n;
    fill_common(p, gc.pl, fmt16(gc.in_bf16), gc.a_mn, gc.b_mn, gc.d_type, gc.alpha, gc.beta, gc.status);
    la.grid = grid_for(gc.pl, *gc.v, gc.dev, gc.sms, tiles);
    la.stream = stream;
    e = gc.v->launch(la);
    if (e != cudaSuccess)
        return cuda_fail(e);
    g_launches.fetch_add(1);
    return GEMM_OK;
}

bool grouped_args_ok(const gemm_problem_t *probs, int n, int a_major, int b_major, int d_type)
{
    return n >= 0 && (n == 0 || probs) && valid_enum(a_major) && valid_enum(b_major) && d_type >= 0 && d_type <= 2;
}

gemm_status_t run_grouped(int in_bf16, const gemm_problem_t *probs, int n, int a_major, int b_major,
                          int d_type, float alpha, float beta, void *ws, size_t ws_bytes,
                          const gemm_options_t *opts, cudaStream_t stream)
{
    if (!grouped_args_ok(probs, n, a_major, b_major, d_type))
        return GEMM_ERR_INVALID_ARG;
    if (n == 0)
        return GEMM_OK;
    if (!ws || ws_bytes < gemm_grouped_workspace_size(n))
        return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 127u) != 0)
        return GEMM_ERR_ALIGNMENT;
    GroupedCall gc;
    gemm_status_t s = plan_grouped(in_bf16, probs, n, a_major, b_major, d_type, alpha, beta, opts, &gc);
    if (s != GEMM_OK)
        return s;
    std::vector<unsigned char> host(gemm_grouped_workspace_size(n), 0);
    int64_t tiles = 0;
    if ((s = build_grouped_image(gc, probs, n, host.data(), &tiles)) != GEMM_OK)
        return s;
    if (tiles == 0)
        return GEMM_OK;
    return upload_and_launch_grouped(gc, n, tiles, host.data(), host.size(), static_cast<unsigned char *>(ws),
                                     stream);
}

// ---------------------------------------------------------------- inspection kernels

__global__ void debug_descriptor_kernel(int major, int swz_bits, int rows, int bk, uint32_t stage_addr,
                                        int n_slices, int umma_m, int tile_n, int fmt, int esize,
                                        int a_mn, int b_mn, uint64_t *out)
{
    if (threadIdx.x != 0 || blockIdx.x != 0)
        return;
    // the same arithmetic as the MMA role: stage descriptor + slice offset / 16
    const OperandPacking pk = operand_packing(major, swz_bits, rows, bk);
    const uint64_t d0 = make_smem_desc(stage_addr, pk.lbo, pk.sbo, pk.swz);
    for (int j = 0; j < n_slices; ++j)
        out[j] = d0 + (slice_byte_offset(major, swz_bits, rows, j, esize) >> 4);
    out[n_slices] = make_idesc(umma_m, tile_n, fmt, fmt, a_mn, b_mn);
}

__global__ void debug_stage_kernel(const __grid_constant__ CUtensorMap map, int mn_major, int swz_bits,
                                   int rows, int bk, int mn0, int k0, uint8_t *out,
                                   unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    const uint32_t raw = smem_u32(sm_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bytes = static_cast<uint32_t>(rows * bk * 2);
    const uint32_t bar = base + bytes;
    __shared__ int ok_flag;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        ok_flag = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, bytes);
        load_operand_stage<1>(&map, base, bar, mn_major, swz_bits, rows, bk, mn0, k0);
        const uint64_t t0 = globaltimer_ns();
        bool ok = true;
        while (!mbar_try_wait(bar, 0)) {
            if (globaltimer_ns() - t0 > 1000000000ull) {
                ok = false;
                atomicCAS(status, 0u, kRoleProducer | kWaitFull);
                break;
            }
        }
        ok_flag = ok ? 1 : 0;
        if (!ok) {
            // let the copy land before the CTA can exit
            const uint64_t t1 = globaltimer_ns();
            while (globaltimer_ns() - t1 < 20000ull)
                __nanosleep(1000);
        }
    }
    __syncthreads();
    if (!ok_flag)
        return;
    const uint8_t *src = sm_raw + (base - raw);
    for (uint32_t i = threadIdx.x * 16u; i < bytes; i += blockDim.x * 16u)
        *reinterpret_cast<uint4 *>(out + i) = *reinterpret_cast<const uint4 *>(src + i);
}

// ---------------------------------------------------------------- grouped GEMM without allocation
//
// Some callers cannot allocate device memory at the moment they launch a
// GEMM: programs whose allocator has reserved the whole device and forbids
// side allocations, plug-ins that are handed their input and output buffers
// by a host runtime and own no memory budget of their own, and real-time
// loops that may not block in the driver's allocator (cudaMalloc can
// synchronise the device). For them the grouped GEMM's workspace (problem
// table plus one TMA descriptor per operand per problem) lives in the fixed
// array below, sized for kNoAllocMaxProblems problems. Every GPU that loads
// the library holds it until the process exits.

constexpr int kNoAllocMaxProblems = GEMM_NOALLOC_MAX_PROBLEMS;
constexpr size_t kNoAllocScratchBytes =
    ((static_cast<size_t>(kNoAllocMaxProblems) * sizeof(GroupedProblemDev) + 127) & ~size_t(127)) +
    static_cast<size_t>(kNoAllocMaxProblems) * 4 * sizeof(CUtensorMap);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host staging for the table; guarded by g_noalloc_mu. A pageable-source copy
// has consumed its source when cudaMemcpyAsync returns, so it can be reused.
static unsigned char g_noalloc_host[kNoAllocScratchBytes];
std::mutex g_noalloc_mu;
unsigned char *g_noalloc_dev[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name only stands in for the symbol, so the address is looked up once
// per device (with that device current) and cached.
gemm_status_t noalloc_scratch(int dev, unsigned char **out)
{
    if (!g_noalloc_dev[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return GEMM_ERR_CUDA;
        g_noalloc_dev[dev] = static_cast<unsigned char *>(ptr);
    }
    *out = g_noalloc_dev[dev];
    return GEMM_OK;
}

gemm_status_t run_grouped_noalloc(int in_bf16, const gemm_problem_t *probs, int n, int a_major,
                                  int b_major, int d_type, float alpha, float beta,
                                  cudaStream_t stream)
{
    if (!grouped_args_ok(probs, n, a_major, b_major, d_type))
        return GEMM_ERR_INVALID_ARG;
    if (n > kNoAllocMaxProblems)
        return GEMM_ERR_INVALID_ARG;  // more problems than the fixed scratch holds
    if (n == 0)
        return GEMM_OK;
    GroupedCall gc;
    gemm_status_t s = plan_grouped(in_bf16, probs, n, a_major, b_major, d_type, alpha, beta, nullptr, &gc);
    if (s != GEMM_OK)
        return s;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    unsigned char *ws = nullptr;
    if ((s = noalloc_scratch(gc.dev, &ws)) != GEMM_OK)
        return s;
    const size_t used = table_bytes(n) + static_cast<size_t>(n) * 4 * sizeof(CUtensorMap);
    // the whole used region is rewritten on every call: nothing is left over
    // from an earlier call with more problems or other pointers
    std::memset(g_noalloc_host, 0, used);
    int64_t tiles = 0;
    if ((s = build_grouped_image(gc, probs, n, g_noalloc_host, &tiles)) != GEMM_OK)
        return s;
    if (tiles == 0)
        return GEMM_OK;
    return upload_and_launch_grouped(gc, n, tiles, g_noalloc_host, used, ws, stream);
}

}  // namespace

// ---------------------------------------------------------------- C ABI

extern "C" {

gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K, const void *A, gemm_major_t a_major,
                        int64_t lda, const void *B, gemm_major_t b_major, int64_t ldb, const void *C,
                        int64_t ldc, void *D, int64_t ldd, gemm_out_t d_type, float alpha, float beta,
                        gemm_stream_t stream)
{
    return run_single(fmt16(1), M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd, d_type, alpha, beta,
                      nullptr, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K, const void *A, gemm_major_t a_major,
                       int64_t lda, const void *B, gemm_major_t b_major, int64_t ldb, const void *C,
                       int64_t ldc, void *D, int64_t ldd, gemm_out_t d_type, float alpha, float beta,
                       gemm_stream_t stream)
{
    return run_single(fmt16(0), M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd, d_type, alpha, beta,
                      nullptr, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_ex(int in_type, int64_t M, int64_t N, int64_t K, const void *A, gemm_major_t a_major,
                      int64_t lda, const void *B, gemm_major_t b_major, int64_t ldb, const void *C,
                      int64_t ldc, void *D, int64_t ldd, gemm_out_t d_type, float alpha, float beta,
                      const gemm_options_t *opts, gemm_stream_t stream)
{
    if (in_type < 0 || in_type > 2)
        return GEMM_ERR_INVALID_ARG;
    return run_single(in_type == 2 ? fmt32() : fmt16(in_type), M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc,
                      D, ldd, d_type, alpha, beta, opts, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_fp8_ex(int64_t M, int64_t N, int64_t K, const void *A, gemm_fp8_t a_format,
                          gemm_major_t a_major, int64_t lda, const void *B, gemm_fp8_t b_format,
                          gemm_major_t b_major, int64_t ldb, const void *C, int64_t ldc, void *D,
                          int64_t ldd, gemm_out_t d_type, float alpha, float beta,
                          const gemm_options_t *opts, gemm_stream_t stream)
{
    if ((a_format != GEMM_FP8_E4M3 && a_format != GEMM_FP8_E5M2) ||
        (b_format != GEMM_FP8_E4M3 && b_format != GEMM_FP8_E5M2))
        return GEMM_ERR_INVALID_ARG;
    return run_single(fmt8(a_format, b_format), M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd,
                      d_type, alpha, beta, opts, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_fp8(int64_t M, int64_t N, int64_t K, const void *A, gemm_fp8_t a_format,
                       gemm_major_t a_major, int64_t lda, const void *B, gemm_fp8_t b_format,
                       gemm_major_t b_major, int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd,
                       gemm_out_t d_type, float alpha, float beta, gemm_stream_t stream)
{
    return gemm_fp8_ex(M, N, K, A, a_format, a_major, lda, B, b_format, b_major, ldb, C, ldc, D, ldd, d_type,
                       alpha, beta, nullptr, stream);
}

size_t gemm_mx_scale_bytes(int64_t rows, int64_t K)
{
    if (rows <= 0 || K <= 0)
        return 0;
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((K + 127) / 128) * 512;
}

gemm_status_t gemm_mxfp8(int64_t M, int64_t N, int64_t K, const void *A, gemm_fp8_t a_format,
                         gemm_major_t a_major, int64_t lda, const void *SFA, const void *B, gemm_fp8_t b_format,
                         gemm_major_t b_major, int64_t ldb, const void *SFB, const void *C, int64_t ldc, void *D,
                         int64_t ldd, gemm_out_t d_type, float alpha, float beta, const gemm_options_t *opts,
                         gemm_stream_t stream)
{
    if ((a_format != GEMM_FP8_E4M3 && a_format != GEMM_FP8_E5M2) ||
        (b_format != GEMM_FP8_E4M3 && b_format != GEMM_FP8_E5M2))
        return GEMM_ERR_INVALID_ARG;
    return run_single(fmtmx(a_format, b_format), M, N, K, A, a_major, lda, B, b_major, ldb, C, ldc, D, ldd, d_type,
                      alpha, beta, opts, reinterpret_cast<cudaStream_t>(stream), SFA, SFB);
}

size_t gemm_fp4_scale_bytes(int64_t rows, int64_t K, gemm_fp4_scale_t kind)
{
    if (rows <= 0 || K <= 0 || (kind != GEMM_FP4_NVFP4 && kind != GEMM_FP4_MXFP4))
        return 0;
    const int64_t per = kind == GEMM_FP4_NVFP4 ? 64 : 128;  // K elements per atom (4 blocks)
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((K + per - 1) / per) * 512;
}

gemm_status_t gemm_fp4(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *SFA,
                       const void *B, int64_t ldb, const void *SFB, gemm_fp4_scale_t kind, const void *C,
                       int64_t ldc, void *D, int64_t ldd, gemm_out_t d_type, float alpha, float beta,
                       const gemm_options_t *opts, gemm_stream_t stream)
{
    if (kind != GEMM_FP4_NVFP4 && kind != GEMM_FP4_MXFP4)
        return GEMM_ERR_INVALID_ARG;
    // packed operands: two elements per byte, so K and the leading dimensions go in bytes
    if (K < 0 || (K & 1) || lda < 0 || ldb < 0 || (lda & 1) || (ldb & 1))
        return GEMM_ERR_INVALID_ARG;
    return run_single(fmtfp4(kind == GEMM_FP4_NVFP4 ? kScaleNv4 : kScaleMx4), M, N, K / 2, A, GEMM_K_MAJOR, lda / 2,
                      B, GEMM_K_MAJOR, ldb / 2, C, ldc, D, ldd, d_type, alpha, beta, opts,
                      reinterpret_cast<cudaStream_t>(stream), SFA, SFB);
}

size_t gemm_streamk_workspace_size(void)
{
    int dev = 0, sms = 0;
    unsigned int *status = nullptr;
    if (device_state(&dev, &status, &sms) != GEMM_OK || sms <= 0)
        return 0;
    return sk_bytes(sms, 256, 256);
}

size_t gemm_grouped_workspace_size(int num_problems)
{
    if (num_problems <= 0)
        return 0;
    return table_bytes(num_problems) + static_cast<size_t>(num_problems) * 4 * sizeof(CUtensorMap);
}

gemm_status_t gemm_bf16_grouped(const gemm_problem_t *problems, int num_problems, gemm_major_t a_major,
                                gemm_major_t b_major, gemm_out_t d_type, float alpha, float beta,
                                void *workspace, size_t workspace_bytes, gemm_stream_t stream)
{
    return run_grouped(1, problems, num_problems, a_major, b_major, d_type, alpha, beta, workspace,
                       workspace_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_grouped(const gemm_problem_t *problems, int num_problems, gemm_major_t a_major,
                               gemm_major_t b_major, gemm_out_t d_type, float alpha, float beta,
                               void *workspace, size_t workspace_bytes, gemm_stream_t stream)
{
    return run_grouped(0, problems, num_problems, a_major, b_major, d_type, alpha, beta, workspace,
                       workspace_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_bf16_grouped_noalloc(const gemm_problem_t *problems, int num_problems,
                                        gemm_major_t a_major, gemm_major_t b_major, gemm_out_t d_type,
                                        float alpha, float beta, gemm_stream_t stream)
{
    return run_grouped_noalloc(1, problems, num_problems, a_major, b_major, d_type, alpha, beta,
                               reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_grouped_ex(int in_type, const gemm_problem_t *problems, int num_problems,
                              gemm_major_t a_major, gemm_major_t b_major, gemm_out_t d_type, float alpha,
                              float beta, void *workspace, size_t workspace_bytes, const gemm_options_t *opts,
                              gemm_stream_t stream)
{
    if (in_type != 0 && in_type != 1)
        return GEMM_ERR_INVALID_ARG;
    return run_grouped(in_type, problems, num_problems, a_major, b_major, d_type, alpha, beta, workspace,
                       workspace_bytes, opts, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_last_device_status(gemm_stream_t stream, uint32_t *detail)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (detail)
        *detail = v;
    return v ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

const char *gemm_status_string(gemm_status_t s)
{
    switch (s) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_ALIGNMENT: return "pointer or leading dimension breaks a TMA alignment rule";
    case GEMM_ERR_UNSUPPORTED: return "unsupported configuration";
    case GEMM_ERR_CUDA: return "CUDA call failed";
    case GEMM_ERR_TIMEOUT: return "a bounded device wait ran out";
    }
    return "unknown status";
}

uint64_t gemm_launch_count(void) { return g_launches.load(); }

gemm_status_t gemm_debug_descriptors(int major, int swizzle, int rows, int bk, uint32_t stage_addr,
                                     int n_slices, int cta_group, int tile_n, int in_type, int a_major,
                                     int b_major, uint64_t *out, gemm_stream_t stream)
{
    if (!valid_enum(major) || swizzle < 1 || swizzle > 5 || rows <= 0 || bk <= 0 || n_slices < 0 ||
        (cta_group != 1 && cta_group != 2) || tile_n <= 0 || !out || in_type < 0 || in_type > 4 ||
        !valid_enum(a_major) || !valid_enum(b_major))
        return GEMM_ERR_INVALID_ARG;
    // in_type 0 fp16, 1 bf16 (kind::f16); 2 E4M3, 3 E5M2 (kind::f8f6f4); 4 TF32 (kind::tf32)
    const int esize = in_type == 4 ? 4 : in_type >= 2 ? 1 : 2;
    const int fmt = in_type == 4 ? 2 : in_type >= 2 ? in_type - 2 : in_type;
    debug_descriptor_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        major, swz_bits_of(swizzle), rows, bk, stage_addr, n_slices, 128 * cta_group, tile_n, fmt, esize,
        a_major, b_major, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e);
    g_launches.fetch_add(1);
    return GEMM_OK;
}

gemm_status_t gemm_debug_stage_image(const void *src, int major, int swizzle, int64_t rows_total,
                                     int64_t k_total, int64_t ld, int rows, int bk, int64_t mn0, int64_t k0,
                                     void *out, gemm_stream_t stream)
{
    if (!src || !out || !valid_enum(major) || swizzle < 1 || swizzle > 5 || rows <= 0 || rows > 256 ||
        bk <= 0 || bk > 256 || rows_total <= 0 || k_total <= 0 || mn0 < 0 || k0 < 0 ||
        mn0 > INT32_MAX || k0 > INT32_MAX || rows_total > INT32_MAX || k_total > INT32_MAX)
        return GEMM_ERR_INVALID_ARG;
    const int bits = swz_bits_of(swizzle);
    const int per = static_cast<int>(swizzle_row_bytes(bits)) / 2;
    if (major == GEMM_K_MAJOR ? (bk % per != 0) : (rows % per != 0))
        return GEMM_ERR_UNSUPPORTED;
    if (ld < (major == GEMM_K_MAJOR ? k_total : rows_total))
        return GEMM_ERR_INVALID_ARG;
    // the TMA box's inner coordinate must start on a 16-byte boundary
    if (!aligned16(src) || !aligned16(out) || ld % 8 != 0 || (major == GEMM_K_MAJOR ? k0 : mn0) % 8 != 0)
        return GEMM_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    unsigned int *status = nullptr;
    gemm_status_t s = device_state(&dev, &status, &sms);
    if (s != GEMM_OK)
        return s;
    CUtensorMap map;
    if ((s = encode_operand(&map, 1, src, major, bits, rows_total, k_total, ld, rows, bk)) != GEMM_OK)
        return s;
    const int smem = rows * bk * 2 + 1024 + 64;
    cudaError_t e = cudaFuncSetAttribute(debug_stage_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return cuda_fail(e);
    debug_stage_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
        map, major, bits, rows, bk, static_cast<int>(mn0), static_cast<int>(k0),
        static_cast<uint8_t *>(out), status);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e);
    g_launches.fetch_add(1);
    return GEMM_OK;
}

gemm_status_t gemm_debug_plan(int64_t M, int64_t N, int64_t K, int kind, int a_major, int b_major, int grouped,
                              const gemm_options_t *opts, int sms, int32_t *out)
{
    if (!out || sms <= 0 || kind < 0 || kind > 5 || !valid_enum(a_major) || !valid_enum(b_major) || M < 0 ||
        N < 0 || K < 0)
        return GEMM_ERR_INVALID_ARG;
    // kind: 0 fp16/bf16, 1 fp8, 2 MXFP8, 3 NVFP4, 4 MXFP4 (fp4: K counted in elements, planned in
    // bytes), 5 TF32
    const int esize = kind == 5 ? 4 : kind == 0 ? 2 : 1;
    const int sf = kind == 2 ? kScaleMx8 : kind == 3 ? kScaleNv4 : kind == 4 ? kScaleMx4 : kScaleNone;
    const int64_t k_plan = kind >= 3 ? K / 2 : K;
    Plan pl;
    const gemm_status_t s = make_plan(M, N, k_plan, a_major, b_major, sms, opts, grouped != 0, &pl, esize, sf);
    if (s != GEMM_OK)
        return s;
    out[0] = pl.cg;
    out[1] = pl.bn;
    out[2] = pl.bk;
    out[3] = pl.bm;
    out[4] = pl.a_swz;
    out[5] = pl.b_swz;
    out[6] = pl.epi_swizzle;
    out[7] = pl.group_m;
    out[8] = pl.ws;
    out[9] = pl.mcb;
    return GEMM_OK;
}

int gemm_debug_streamk_units(int mode, int64_t tiles, int clusters, int kb_per_tile, int cluster, int32_t *out,
                             int max_units)
{
    if (tiles < 0 || tiles >= (static_cast<int64_t>(1) << 31) || clusters < 1 || kb_per_tile < 1 || cluster < 0 ||
        cluster >= clusters || max_units < 0 || (max_units > 0 && !out))
        return -1;
    const int64_t dp = sk_split(mode, tiles, clusters, kb_per_tile);
    if (dp < 0)
        return -1;
    Sched sc;
    std::memset(&sc, 0, sizeof(sc));
    sc.num_tiles = static_cast<int>(tiles);
    sc.sk_dp = static_cast<int>(dp);
    sc.kbt = kb_per_tile;
    sc.sk_iters = (tiles - dp) * kb_per_tile;
    UnitIter it(sc, cluster, clusters);
    Unit u;
    int n = 0;
    while (it.next(u)) {
        if (n < max_units) {
            int32_t *o = out + 6 * n;
            const int kind = unit_kind(u, sc.kbt);
            o[0] = u.tile;
            o[1] = u.kb0;
            o[2] = u.kb1;
            o[3] = kind;
            o[4] = 0;
            o[5] = -1;
            if (kind == kUnitHead) {
                const long long first = static_cast<long long>(u.tile - sc.sk_dp) * sc.kbt;
                o[4] = sk_owner(first + u.kb1, sc.sk_iters, clusters);
                o[5] = sk_owner(first + sc.kbt - 1, sc.sk_iters, clusters);
            }
        }
        ++n;
    }
    return n;
}

void gemm_debug_inject_timeout(int timeout_ms) { gemm_debug_inject_timeout_at(timeout_ms, kRoleMma); }

void gemm_debug_inject_timeout_at(int timeout_ms, int role)
{
    if (role != kRoleProducer && role != kRoleMma)
        return;
    g_inject_role.store(role);
    g_inject_timeout_ms.store(timeout_ms > 0 ? timeout_ms : 0);
}

}  // extern "C"
