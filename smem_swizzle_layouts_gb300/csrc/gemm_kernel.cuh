// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   D = alpha * A * B + beta * C,  fp16/bf16 in, fp32 accumulate in TMEM.
//
// One CTA (cta_group::1) or one CTA pair (cta_group::2, cluster of 2) per
// SM / SM pair walks a static round-robin list of output tiles. Warp roles:
//   warp 0     TMA producer: one thread fills an S-stage shared-memory ring
//              (full/empty mbarriers, "Tensor Cores, layouts, and swizzling",
//              TMA section and 6.6.1: expect_tx bytes, parity (k/S)&1);
//   warp 1     TMEM allocator and MMA issuer: one thread issues
//              tcgen05.mma for every K slice and commits completion to
//              mbarriers ("06 Blackwell Tensor Core - tcgen05 MMA", "How
//              tcgen05.mma Executes"); the accumulator is double-buffered
//              in TMEM (2 x BN fp32 columns) so the epilogue of tile i
//              overlaps the main loop of tile i+1 (two-half 256-row tiles
//              on one CTA: two M=128 MMAs per K slice, both accumulators in
//              TMEM, one buffer);
//   warps 2-5  epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (the lane
//              quarter rule of "Tensor Cores, layouts, and swizzling",
//              tcgen05 section) with tcgen05.ld, applies alpha/beta against
//              C (TMA-loaded, or read into registers), converts, stages
//              32-row chunks in a swizzled shared-memory buffer and writes
//              them with TMA stores;
//   warp 6     block-scaled kinds only: scale copier (tcgen05.cp of each
//   (and 7)    stage's scale atoms into TMEM); NVFP4 runs two copiers on
//              alternate K groups;
//   last warp  second producer, issuing the B boxes when the loads are
//              split (kFlagSplitLoad; not in the NVFP4 kernels). So 224
//              threads, or 256 with copiers.
//
// CTA pairs: the even CTA holds accumulator rows 0-127 and the odd CTA rows
// 128-255 ("How cta_group Sets the Operation Scope", cta_group::2, M=256).
// Each CTA TMA-loads its own 128 rows of A and its own half of the tile's N
// columns of B into its own shared memory (no multicast); the .cta_group::2
// form of the load completes the bytes of both on the even CTA's full
// barrier, whose one thread issues the M=256 MMAs. Their completion reaches
// both CTAs through one multicast tcgen05.commit (mask 0b11) on the stage's
// empty barrier and on the accumulator-full barrier; the odd CTA's epilogue
// warps release accumulators by remote arrives on the even CTA's barrier.
// (Forwarding each release from the even CTA to the odd one by a remote
// mbarrier.arrive is kept as the kFlagPairForward ablation.)
//
// Every mbarrier wait is bounded: past the time limit the waiting role
// records a code in the status word, raises a CTA-wide abort flag and
// returns; the kernel then drains in-flight copies and MMAs (with short
// bounds), frees TMEM and exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "descriptors.cuh"
#include "ptx.cuh"

namespace g300 {

constexpr int kEpiWarps = 4;
// warp 0 producer, warp 1 MMA issuer, warps 2-5 epilogue, warp 6 scale copier (block-scaled only)
constexpr int kSfCopyWarp = 2 + kEpiWarps;
constexpr int kEpiBufBytes = 32 * 128;  // one 32-row x 128 B staging chunk

// Roles in the status word (bits 0-7) and waits (bits 8-15).
enum : uint32_t {
    kRoleProducer = 1,
    kRoleMma = 2,
    kRoleEpilogue = 3,
    kRoleSfCopy = 4,
    kWaitEmpty = 1 << 8,
    kWaitFull = 2 << 8,
    kWaitAccEmpty = 3 << 8,
    kWaitAccFull = 4 << 8,
    kWaitEpiC = 5 << 8,
    kWaitInjected = 6 << 8,
    kWaitDrain = 7 << 8,
    kWaitPartial = 8 << 8,
    kWaitSfReady = 9 << 8,
    kRoleSetup = 5,
    kSetupAlignment = 10 << 8,
};

struct GroupedProblemDev {
    int M, N, K;
    int tiles_m, tiles_n;
    int tile_start;  // first linear tile of this problem
    int pad0, pad1;
};

struct KParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles;
    float alpha, beta;
    int a_mn, b_mn;        // 0 K-major, 1 MN-major
    int a_swz, b_swz;      // swizzle bits: 0 none, 1 SW32, 2 SW64, 3 SW128, 4 SW128 with 32-byte atoms
    int a_fmt, b_fmt;      // MMA operand formats (kind::f16: 0 fp16, 1 bf16; kind::f8f6f4: 0 E4M3, 1 E5M2)
    int out_type;          // 0 f32, 1 bf16, 2 f16
    int epi_swizzle;       // 1: staging chunks in SW128 layout; 0: plain rows
    int group_m;           // raster group height (tiles)
    unsigned long long timeout_ns;
    int inject_timeout;    // test hook: role (kRoleProducer or kRoleMma) that waits on a barrier nothing arrives at
    unsigned int *status;
    const GroupedProblemDev *problems;  // grouped launches only
    const CUtensorMap *maps;            // [num_problems][4]: A, B, C, D
    int num_problems;
    int flags;                  // kFlag* tuning switches
    unsigned long long *stats;  // optional per-CTA wait counters (kStat* slots), or null
    // Stream-K (single problems). Tiles [0, sk_dp_tiles) run data-parallel,
    // one whole tile per unit; the K iterations of the remaining tiles
    // (sk_iters = (num_tiles - sk_dp_tiles) * kb_per_tile) are split evenly
    // across the clusters. A tile cut between clusters is finished by the one
    // holding its first K block (its head). The others leave their fp32
    // partial sums in sk_partials (slot cluster * CG + rank, 128 x BN, or
    // 256 x BN for two-half tiles) and
    // raise their flags (sk_flags[(cluster * CG + rank) * 4 + warp] =
    // sk_epoch). A head is always its cluster's last unit, so the other TMEM
    // accumulator buffer is free while the head's MMAs run: the epilogue
    // warps gather the partial sums into it meanwhile and add both buffers
    // in the head's epilogue. Two-half tiles have no other buffer: their
    // head adds the partial sums from the slots chunk by chunk.
    int sk_dp_tiles;
    int kb_per_tile;
    long long sk_iters;
    float *sk_partials;
    unsigned int *sk_flags;
    unsigned int sk_epoch;
    // Block-scaled operands: K groups (128 elements) per row block of the
    // scale tensors; atom (i * sf_groups + g) holds row block i, K group g
    int sf_groups;
    // C and D of a single problem (row-major, ldc / ldd elements per row), for
    // the epilogue reading C straight into registers (kFlagDirectC) and writing
    // D straight from them (kFlagDirectD)
    const void *c_ptr;
    long long ldc;
    void *d_ptr;
    long long ldd;
};

// Diagnostics: per-CTA counters written when KParams::stats is set.
enum : int {
    kStatProducerWaitCycles = 0,
    kStatProducerBlocked = 1,
    kStatMmaFullWaitCycles = 2,
    kStatMmaAccEmptyWaitCycles = 3,
    kStatMmaLoopCycles = 4,
    kStatEpiAccFullWaitCycles = 5,
    kStatEpiCWaitCycles = 6,
    kStatEpiLoopCycles = 7,
    kStatMmaFullBlocked = 8,
    kStatTiles = 9,
    kStatEpiPartialWaitCycles = 10,  // stream-K head: waiting for contributors' flags
    kStatEpiPartialCycles = 11,      // stream-K head: gathering partial sums into TMEM
    kStatEpiTailCycles = 12,         // from the last accumulator-full wait to the end
    kStatSfCopyWaitCycles = 13,      // scale copier: waiting for stages to land
    kStatMmaSfWaitCycles = 14,       // MMA issuer: waiting for a stage's scales in TMEM
    kStatSlots = 16,
};

enum : int {
    kFlagPairForward = 1,      // CTA pairs: forward releases with remote arrives (ablation)
    kFlagAllClusterWaits = 2,  // CTA pairs: cluster-scope acquire on every wait (ablation)
    kFlagRotateK = 4,          // start each tile's K loop at a per-cluster offset
    kFlagCacheHints = 8,       // operands evict_last, C loads and D stores evict_first in L2
    kFlagDirectC = 16,         // single problems, 128-row tiles: C read into registers, not staged
    kFlagSplitLoad = 32,       // two producer warps: A boxes (and scale atoms) from one, B boxes from the other
    kFlagDirectD = 64,         // single problems, 128- and 256-row tiles: D stored from registers, not staged
};

// K block processed at iteration `it` of a tile: with kFlagRotateK the
// cluster starts at its own offset, so CTAs that share an operand panel do not
// all read the same K block of it at the same moment.
__device__ __forceinline__ int kblock_at(int it, int num_kb, int flags, int cluster_id)
{
    if (!(flags & kFlagRotateK))
        return it;
    const int r = it + (cluster_id * 7) % num_kb;
    return r >= num_kb ? r - num_kb : r;
}

// Block-scaled operand kinds (the SF template argument). A scale atom holds
// 4 scale blocks of 128 rows; its K extent in bytes is 4 x block x element
// bytes: MXFP8 (E8M0 per 32 fp8) 128, NVFP4 (UE4M3 per 16 E2M1) 32, MXFP4
// (E8M0 per 32 E2M1) 64. fp4 operands are packed two to a byte, and their
// tiles count K in bytes (one 32-byte slice = one K = 64 MMA).
enum : int { kScaleNone = 0, kScaleMx8 = 1, kScaleNv4 = 2, kScaleMx4 = 3 };

__host__ __device__ constexpr int sf_atom_kbytes(int sf)
{
    return sf == kScaleMx8 ? 128 : sf == kScaleNv4 ? 32 : 64;
}

// ESIZE: bytes per operand element, 2 (fp16/bf16, tcgen05 kind::f16),
// 1 (fp8, kind::f8f6f4) or 4 (fp32 words read as TF32, kind::tf32). BK counts elements of K per stage. BMT: accumulator
// rows per CTA, 128 (row m in TMEM lane m) or 64 (cta_group::1 only, Layout F:
// rows 16g..16g+15 in lanes 32g+a..32g+a+15; the two accumulators of the
// double buffer take lane alignments a = 0 and 16 and share their columns).
// Tile modes (the MODE template argument): ordinary MMAs; the weight-stationary
// tcgen05.mma.ws (32- and 64-row tiles); or a cluster of two cta_group::1 CTAs
// on vertically adjacent tiles that each load half of the shared B panel and
// TMA-multicast it to both (B bytes read from L2 per CTA halved).
enum : int { kModeOrdinary = 0, kModeWs = 1, kModeMcastB = 2 };

template <int CG, int BN, int BK, int STAGES, int ESIZE = 2, int BMT = 128, int SF = 0, int MODE = 0>
struct Cfg {
    static constexpr bool WS = MODE == kModeWs;
    static constexpr bool MCB = MODE == kModeMcastB;
    static constexpr int BM = BMT;             // accumulator rows per CTA
    static constexpr int BN_LOCAL = BN / CG;   // B columns loaded by each CTA
    static constexpr int A_BYTES = BM * BK * ESIZE;
    static constexpr int B_BYTES = BN_LOCAL * BK * ESIZE;
    // Block-scaled stages also carry the scale atoms of their K range: one
    // 512-byte atom covers 128 rows x 4 scale blocks (128 elements of K)
    static constexpr int KGROUPS = SF ? BK / sf_atom_kbytes(SF) : 0;  // scale atoms per stage and row block
    static constexpr int SF_A_BYTES = 512 * KGROUPS * (BM / 128);
    static constexpr int SF_B_BYTES = 512 * KGROUPS * (BN / 128);  // every column of the tile, in each CTA
    static constexpr int SF_OFF = A_BYTES + B_BYTES;  // within a stage
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_A_BYTES + SF_B_BYTES;
    static constexpr int TX_BYTES = STAGE_BYTES * CG;  // bytes landing on one full barrier
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    // staging chunks per epilogue warp: two (a store may still read one while
    // the next is filled); block-scaled tiles keep one, to leave room for the
    // scale atoms of three 256-element K stages
    static constexpr int EPI_BUFS = SF ? 1 : 2;
    static constexpr int EPI_BYTES = kEpiWarps * EPI_BUFS * kEpiBufBytes;
    static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
    // full[S], empty[S], acc_full[2], acc_empty[2], epi[4][2], drain, inject, sf_ready[S], copier drain
    static constexpr int NUM_BARS = 3 * STAGES + 2 + 2 + 2 * kEpiWarps + 3;
    // threads per CTA: the scale copier warp exists only for block-scaled kinds
    // scale copier warps: NVFP4 stages carry three times the atoms of the others
    static constexpr int SF_COPIERS = SF == kScaleNv4 ? 2 : SF ? 1 : 0;
    // the second producer warp (B boxes when loads are split) comes last; the
    // NVFP4 kernels, with two copier warps, go without it: a ninth warp puts
    // three warps on one SM sub-partition and caps registers below their need
    static constexpr bool HAS_LOADB = kSfCopyWarp + SF_COPIERS < 8;
    static constexpr int LOADB_WARP = HAS_LOADB ? kSfCopyWarp + SF_COPIERS : -1;
    static constexpr int THREADS = 32 * (kSfCopyWarp + SF_COPIERS + (HAS_LOADB ? 1 : 0));
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    // + slack to round the base up to 1024 bytes; the dynamic shared memory is
    // declared 1024-aligned, so a variant that would not fit with the slack
    // goes without it and checks the alignment at launch instead
    static constexpr int ALIGN_SLACK = MISC_OFF + 16 + 1024 <= 232448 ? 1024 : 0;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + ALIGN_SLACK;
    // TMEM: two accumulators, then (block-scaled) per stage 4 columns of A
    // scales and 4 of B scales for each K group
    // Accumulator buffers: two (the epilogue of one tile overlaps the next
    // tile's MMAs), except for block-scaled 256-wide tiles, whose two
    // accumulators would leave no TMEM for the scale slots
    // Two-half tiles (BMT 256, single CTAs): two 128-row accumulators side by
    // side fill the TMEM columns, so they have one buffer and the epilogue of a
    // tile does not overlap the next tile's MMAs
    static constexpr int M_HALVES = BMT == 256 ? 2 : 1;
    // TMEM column of the second half's accumulator: 256 whatever the width,
    // so that a 64-column epilogue chunk of a 224-wide tile reads past its
    // own columns only into columns no accumulator uses
    static constexpr int HALF_COL = 256;
    static constexpr int ACC_BUFS = ((SF && BN == 256) || M_HALVES == 2) ? 1 : 2;
    static constexpr int SF_COL0 = ACC_BUFS * BN;
    static constexpr int SF_GROUP_COLS = 4 + 4 * (BN / 128);  // A atom, then the B atoms of one K group
    static constexpr int SF_COLS = SF_GROUP_COLS * KGROUPS;
    // Weight-stationary tiles (WS, tcgen05.mma.ws with M = BM = 32 or 64): the
    // accumulator is spread over the four TMEM lane quarters by column parts.
    // Quarter q holds rows 32 (q % RB) .. +31 (RB = BM / 32 row blocks) of
    // column part q / RB, COL_PARTS = 4 / RB parts of BN / COL_PARTS columns,
    // at TMEM column n - part * (BN / COL_PARTS); one buffer takes ACC_COLS.
    static constexpr int WS_ROW_BLOCKS = WS ? BM / 32 : 1;
    static constexpr int COL_PARTS = WS ? 4 / WS_ROW_BLOCKS : 1;
    static constexpr int ACC_COLS = BN / COL_PARTS;
    static constexpr int TMEM_COLS = WS ? (2 * ACC_COLS < 32 ? 32 : 2 * ACC_COLS) : BMT == 64 ? BN : (SF || M_HALVES == 2) ? 512 : 2 * BN;
    static constexpr int UMMA_M = BM / M_HALVES * CG;
    // CTAs per cluster (CTA pairs, or the two CTAs sharing B by multicast) and
    // the output rows of one cluster tile; B rows/atoms one CTA's TMA loads
    static constexpr int CLUSTER = (CG == 2 || MCB) ? 2 : 1;
    static constexpr int TILE_M = BM * CLUSTER;
    static constexpr int B_LOAD = MCB ? BN / 2 : BN_LOCAL;
    static_assert(!MCB || (CG == 1 && (BMT == 128 || BMT == 256) && SF == 0 && BN % 32 == 0),
                  "B multicast: two single-CTA 128- or 256-row tiles sharing a B panel split in halves of whole "
                  "8-row groups (MN-major halves of whole atoms are checked by the host)");
    static constexpr int EPI_ROWS = (WS || M_HALVES == 2) ? 32 : BM / 4;  // output rows per epilogue warp (and half)
    static_assert(BMT == 128 || BMT == 256 || (BMT == 64 && CG == 1) || (BMT == 32 && WS),
                  "64-row tiles are single-CTA");
    static_assert(M_HALVES == 1 || (CG == 1 && !WS && SF == 0 && ESIZE != 4 && BN <= HALF_COL && BN % 32 == 0),
                  "two-half tiles: single CTAs, ordinary kind::f16/f8f6f4 MMAs, both accumulators in TMEM");
    static_assert(!WS || ((BMT == 32 || BMT == 64) && CG == 1 && ESIZE == 2 && SF == 0 && (BN / COL_PARTS) % 64 == 0),
                  ".ws tiles: 32 or 64 rows, single CTA, 16-bit operands, whole 64-column chunks per warp");
    static constexpr int KSLICES = BK * ESIZE / 32;  // MMAs per stage (32 bytes of K each)
    static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-aligned");
    static_assert(A_BYTES % 1024 == 0, "B tile must start 1024-aligned");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation: power of two, 32..512 columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static_assert(CG == 1 || BN % 32 == 0, "pair tiles split N in halves of whole atoms");
    static_assert(!SF || (BMT == 128 && (BN == 128 || (BN == 256 && CG == 2)) && ESIZE == 1 &&
                          BK % sf_atom_kbytes(SF) == 0 && SF_COL0 + STAGES * SF_COLS <= 512),
                  "block-scaled tiles: 128-wide per CTA, or 256-wide for pairs; byte operands; whole atoms");
};

// ---------------------------------------------------------------- waits

struct Waiter {
    unsigned long long timeout_ns;
    volatile uint32_t *abort_flag;
    unsigned int *status;
    bool all_cluster_scope;  // tuning flag: cluster-scope acquire on every wait

    __device__ __forceinline__ bool probe(uint32_t bar, uint32_t parity, bool cluster) const
    {
        return (cluster || all_cluster_scope) ? mbar_try_wait_cluster(bar, parity)
                                              : mbar_try_wait(bar, parity);
    }

    __device__ __forceinline__ void fail(uint32_t code) const
    {
        *abort_flag = 1u;
        atomicCAS(status, 0u, code);
    }

    // Waits for the phase of parity `parity`; false if it gave up (timeout or abort).
    // `cluster`: the phase is completed by an arrive from another CTA of the
    // cluster, so the wait acquires at cluster scope.
    __device__ bool wait(uint32_t bar, uint32_t parity, uint32_t code, bool cluster = false) const
    {
        if (probe(bar, parity, cluster))
            return true;
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            for (int i = 0; i < 8; ++i)
                if (probe(bar, parity, cluster))
                    return true;
            if (*abort_flag)
                return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                fail(code);
                return false;
            }
        }
    }

    // Waits until a global flag holds `value` (acquire at GPU scope).
    __device__ bool wait_flag(const uint32_t *flag, uint32_t value, uint32_t code) const
    {
        if (ld_acquire_gpu(flag) == value)
            return true;
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            for (int i = 0; i < 4; ++i)
                if (ld_acquire_gpu(flag) == value)
                    return true;
            if (*abort_flag)
                return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                fail(code);
                return false;
            }
            __nanosleep(64);
        }
    }

    // Short wait used while tearing down; never records a code.
    __device__ bool drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) const
    {
        const uint64_t t0 = globaltimer_ns();
        while (!probe(bar, parity, true))
            if (globaltimer_ns() - t0 > limit_ns)
                return false;
        return true;
    }
};

// ---------------------------------------------------------------- tiles
//
// Kernel parameters live in the __grid_constant__ parameter block. Every
// inline-asm statement below clobbers "memory", so any field read through
// `p` inside a loop would be reloaded after each asm; the roles therefore
// copy what they need into registers once, before their loops.

struct Sched {
    int num_tiles;
    int M, N, K;
    int tiles_m, tiles_n;
    int group_m;
    int num_problems;
    const GroupedProblemDev *problems;
    int sk_dp;          // data-parallel tiles
    int kbt;            // K blocks per tile (stream-K)
    long long sk_iters; // stream-K iterations
};

__device__ __forceinline__ Sched make_sched(const KParams &p)
{
    Sched s;
    s.num_tiles = p.num_tiles;
    s.M = p.M;
    s.N = p.N;
    s.K = p.K;
    s.tiles_m = p.tiles_m;
    s.tiles_n = p.tiles_n;
    s.group_m = p.group_m;
    s.num_problems = p.num_problems;
    s.problems = p.problems;
    s.sk_dp = p.sk_iters > 0 ? p.sk_dp_tiles : p.num_tiles;
    s.kbt = p.kb_per_tile > 0 ? p.kb_per_tile : 1;
    s.sk_iters = p.sk_iters;
    return s;
}

// One unit of a cluster's work: a tile and the K blocks [kb0, kb1) of it to
// accumulate (kb1 < 0: all of the tile's K blocks).
struct Unit {
    int tile, kb0, kb1;
};

// A cluster's units in order: its data-parallel tiles c, c+G, ... below
// sk_dp, then its share [c*S/G, (c+1)*S/G) of the S stream-K iterations, cut
// at tile boundaries. Every role of every CTA of the cluster walks the same
// sequence.
struct UnitIter {
    int G, dp, dp_next, kbt;
    long long pos, end;

    __host__ __device__ __forceinline__ UnitIter(const Sched &s, int c, int g)
    {
        G = g;
        dp = s.sk_dp;
        dp_next = c;
        kbt = s.kbt;
        pos = s.sk_iters * c / g;
        end = s.sk_iters * (c + 1) / g;
    }

    __host__ __device__ __forceinline__ bool next(Unit &u)
    {
        if (dp_next < dp) {
            u.tile = dp_next;
            u.kb0 = 0;
            u.kb1 = -1;
            dp_next += G;
            return true;
        }
        if (pos >= end)
            return false;
        const long long t = pos / kbt;
        const int k0 = static_cast<int>(pos - t * kbt);
        const long long left = end - pos;
        const int k1 = static_cast<int>(left < static_cast<long long>(kbt - k0) ? k0 + left : kbt);
        u.tile = dp + static_cast<int>(t);
        u.kb0 = k0;
        u.kb1 = k1;
        pos += k1 - k0;
        return true;
    }
};

// Cluster whose stream-K share holds iteration i (shares start at floor(c*S/G)).
__host__ __device__ __forceinline__ int sk_owner(long long i, long long S, int G)
{
    return static_cast<int>(((i + 1) * G - 1) / S);
}

// Part a unit plays in a split tile.
enum : int { kUnitWhole = 0, kUnitContributor = 1, kUnitHead = 2 };

__host__ __device__ __forceinline__ int unit_kind(const Unit &u, int kbt)
{
    if (u.kb1 < 0 || (u.kb0 == 0 && u.kb1 == kbt))
        return kUnitWhole;
    return u.kb0 > 0 ? kUnitContributor : kUnitHead;
}

struct TileInfo {
    int prob;
    int m_blk, n_blk;
    int M, N, K;
};

template <bool GROUPED>
__device__ __forceinline__ void decode_tile(const Sched &p, int t, TileInfo &ti)
{
    int tiles_m, tiles_n, local;
    if constexpr (GROUPED) {
        int lo = 0, hi = p.num_problems - 1;
        while (lo < hi) {  // last problem whose first tile is <= t
            const int mid = (lo + hi + 1) >> 1;
            if (p.problems[mid].tile_start <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const GroupedProblemDev g = p.problems[lo];
        ti.prob = lo;
        ti.M = g.M;
        ti.N = g.N;
        ti.K = g.K;
        tiles_m = g.tiles_m;
        tiles_n = g.tiles_n;
        local = t - g.tile_start;
    } else {
        ti.prob = 0;
        ti.M = p.M;
        ti.N = p.N;
        ti.K = p.K;
        tiles_m = p.tiles_m;
        tiles_n = p.tiles_n;
        local = t;
    }
    // Raster in groups of group_m tile rows so that CTAs running at the same
    // time share A row panels and B column panels in L2.
    const int per_group = p.group_m * tiles_n;
    const int g = local / per_group;
    const int first_m = g * p.group_m;
    const int rows_in_group = min(tiles_m - first_m, p.group_m);
    const int r = local - g * per_group;
    ti.m_blk = first_m + r % rows_in_group;
    ti.n_blk = r / rows_in_group;
}

// Geometry of the TMA boxes that fill one operand of a stage (the packing of
// descriptors.cuh): box b lands at dst + b * smem_step and starts at
// (k0 + b * k_step, mn0) for K-major operands or (mn0 + b * mn_step, k0) for
// MN-major ones.
struct OperandBoxes {
    int nbox;
    uint32_t smem_step;
    int step;
    int mn_major;
};

__device__ __forceinline__ OperandBoxes operand_boxes(int mn_major, int swz_bits, int rows, int bk,
                                                      int esize)
{
    const int W = static_cast<int>(swizzle_row_bytes(swz_bits));
    const int per = W / esize;  // elements per swizzled row
    OperandBoxes o;
    o.mn_major = mn_major;
    o.step = per;
    if (!mn_major) {
        o.nbox = bk / per;
        o.smem_step = static_cast<uint32_t>(rows * W);
    } else {
        o.nbox = rows / per;
        o.smem_step = static_cast<uint32_t>(bk * W);
    }
    return o;
}

template <int CG>
__device__ __forceinline__ void issue_box(const CUtensorMap *map, uint32_t dst, uint32_t bar,
                                          const OperandBoxes &o, int b, int mn0, int k0)
{
    const int x = o.mn_major ? mn0 + b * o.step : k0 + b * o.step;
    const int y = o.mn_major ? k0 : mn0;
    if constexpr (CG == 1)
        tma_load_2d(dst + static_cast<uint32_t>(b) * o.smem_step, map, bar, x, y);
    else
        tma_load_2d_pair(dst + static_cast<uint32_t>(b) * o.smem_step, map, bar, x, y);
}

// issue_box with an L2 eviction policy.
template <int CG>
__device__ __forceinline__ void issue_box_hint(const CUtensorMap *map, uint32_t dst, uint32_t bar,
                                               const OperandBoxes &o, int b, int mn0, int k0, uint64_t policy)
{
    const int x = o.mn_major ? mn0 + b * o.step : k0 + b * o.step;
    const int y = o.mn_major ? k0 : mn0;
    if constexpr (CG == 1)
        tma_load_2d_hint(dst + static_cast<uint32_t>(b) * o.smem_step, map, bar, x, y, policy);
    else
        tma_load_2d_pair_hint(dst + static_cast<uint32_t>(b) * o.smem_step, map, bar, x, y, policy);
}

// Issue every TMA box of one operand stage (used by the inspection kernel).
template <int CG>
__device__ __forceinline__ void load_operand_stage(const CUtensorMap *map, uint32_t dst,
                                                   uint32_t bar, int mn_major, int swz_bits,
                                                   int rows, int bk, int mn0, int k0, int esize = 2)
{
    const OperandBoxes o = operand_boxes(mn_major, swz_bits, rows, bk, esize);
    for (int b = 0; b < o.nbox; ++b)
        issue_box<CG>(map, dst, bar, o, b, mn0, k0);
}

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- roles

// The producer's loads that may still be in flight when it stops: the last
// `inflight` stages it filled, the newest being the one before (stage, phase).
struct ProducerTail {
    int inflight;
    int stage;
    uint32_t phase;
};

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
__device__ ProducerTail role_producer(const KParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB,
                                      const CUtensorMap *tmSFA, const CUtensorMap *tmSFB,
                                      uint32_t smem, uint32_t bar_full, uint32_t bar_empty, uint32_t bar_inject,
                                      uint32_t rank, const Waiter &w, int part)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>;
    if (p.inject_timeout == kRoleProducer) {
        // Test hook: wait on a barrier nothing arrives at; the bound runs out.
        // The B warp of split loads stays idle, so nothing is in flight.
        if (part != 2)
            w.wait(bar_inject, 0u, kRoleProducer | kWaitInjected);
        return ProducerTail{0, 0, 0u};
    }
    // part 0 loads whole stages; with split loads part 1 loads the A boxes and
    // A scale atoms and part 2 the B boxes and B scale atoms, each arming the
    // stage's full barrier (two arrivals) with the bytes it loads
    const bool do_a = part != 2, do_b = part != 1;
    const uint32_t tx = part == 0   ? static_cast<uint32_t>(C::TX_BYTES)
                        : part == 1 ? static_cast<uint32_t>((C::A_BYTES + C::SF_A_BYTES) * CG)
                                    : static_cast<uint32_t>((C::B_BYTES + C::SF_B_BYTES) * CG);
    const Sched sched = make_sched(p);
    const int flags = p.flags;
    unsigned long long *const stats = p.stats;
    const CUtensorMap *const maps = p.maps;
    const OperandBoxes boxA = operand_boxes(p.a_mn, p.a_swz, C::BM, BK, ESIZE);
    OperandBoxes boxB = operand_boxes(p.b_mn, p.b_swz, C::B_LOAD, BK, ESIZE);
    // B multicast: this CTA loads half of the tile's B (rows of each K-major
    // box, or MN atoms) into its place in the full B tile of both CTAs
    uint32_t b_own = 0;
    if constexpr (C::MCB) {
        const uint32_t W = swizzle_row_bytes(p.b_swz);
        if (!p.b_mn) {
            boxB.smem_step = static_cast<uint32_t>(BN) * W;
            b_own = rank * static_cast<uint32_t>(C::B_LOAD) * W;
        } else {
            b_own = rank * static_cast<uint32_t>(boxB.nbox) * boxB.smem_step;
        }
    }
    const int nbox = boxA.nbox > boxB.nbox ? boxA.nbox : boxB.nbox;
    const bool forward = CG == 2 && rank == 0 && (flags & kFlagPairForward) && part != 2;
    const int sf_groups = p.sf_groups;
    // operand tiles are re-read by other tiles of the wave: keep them in L2
    const bool hints = (flags & kFlagCacheHints) != 0;
    const uint64_t keep = hints ? l2_policy_evict_last() : 0;

    const uint32_t full_target = (CG == 2) ? mapa_shared(bar_full, 0) : bar_full;
    const uint32_t peer_empty = (CG == 2 && rank == 0) ? mapa_shared(bar_empty, 1) : 0u;
    const int cluster_id = blockIdx.x / C::CLUSTER, num_clusters = gridDim.x / C::CLUSTER;
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool ok = true;
    int last_prob = -1;
    unsigned long long st_wait = 0, st_blocked = 0;
    UnitIter units(sched, cluster_id, num_clusters);
    Unit u;
    while (ok && units.next(u)) {
        TileInfo ti;
        decode_tile<GROUPED>(sched, u.tile, ti);
        const CUtensorMap *mA = tmA, *mB = tmB;
        if constexpr (GROUPED) {
            mA = maps + 4 * ti.prob;
            mB = mA + 1;
            if (ti.prob != last_prob) {
                fence_tensormap_acquire(mA);
                fence_tensormap_acquire(mB);
                last_prob = ti.prob;
            }
        }
        const int num_kb = ceil_div_i(ti.K, BK);
        const int kb_lo = u.kb0, kb_hi = u.kb1 < 0 ? num_kb : u.kb1;
        const bool whole = u.kb1 < 0;
        const int m0 = ti.m_blk * C::TILE_M + C::BM * static_cast<int>(rank);
        const int n0 = ti.n_blk * BN + C::B_LOAD * static_cast<int>(rank);
        // a stage is released by arrivals from the other CTA of the cluster too
        // (pairs: the odd CTA's; B multicast: both CTAs' MMA commits)
        const bool remote_release = rank != 0 || C::MCB;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (stats) {
                const long long t0 = clock64();
                const bool ready = mbar_try_wait(bar_empty + 8 * stage, phase ^ 1u);
                ok = ready || w.wait(bar_empty + 8 * stage, phase ^ 1u, kRoleProducer | kWaitEmpty, remote_release);
                st_wait += static_cast<unsigned long long>(clock64() - t0);
                st_blocked += ready ? 0 : 1;
            } else {
                ok = w.wait(bar_empty + 8 * stage, phase ^ 1u, kRoleProducer | kWaitEmpty, remote_release);
            }
            if (!ok)
                break;
            // pass a real release (not the first trip round the ring) on to the odd CTA
            if (forward && issued >= STAGES)
                mbar_arrive_cluster(peer_empty + 8 * stage);
            if (rank == 0 || C::MCB)
                mbar_arrive_expect_tx(bar_full + 8 * stage, tx);
            const uint32_t sA = smem + stage * C::STAGE_BYTES;
            const uint32_t sB = sA + C::A_BYTES;
            const uint32_t fb = full_target + 8 * stage;
            const int k0 = (whole ? kblock_at(kb, num_kb, flags, cluster_id) : kb) * BK;
            // A and B boxes alternate, so both operands of the stage are in flight together
            if constexpr (C::MCB) {
                for (int b = 0; b < nbox; ++b) {
                    if (do_a && b < boxA.nbox)
                        issue_box<1>(mA, sA, fb, boxA, b, m0, k0);
                    if (do_b && b < boxB.nbox) {
                        const int x = boxB.mn_major ? n0 + b * boxB.step : k0 + b * boxB.step;
                        const int y = boxB.mn_major ? k0 : n0;
                        tma_load_2d_mcast2(sB + b_own + static_cast<uint32_t>(b) * boxB.smem_step, mB, fb, x, y);
                    }
                }
            } else if (hints) {
                for (int b = 0; b < nbox; ++b) {
                    if (do_a && b < boxA.nbox)
                        issue_box_hint<CG>(mA, sA, fb, boxA, b, m0, k0, keep);
                    if (do_b && b < boxB.nbox)
                        issue_box_hint<CG>(mB, sB, fb, boxB, b, n0, k0, keep);
                }
            } else {
                for (int b = 0; b < nbox; ++b) {
                    if (do_a && b < boxA.nbox)
                        issue_box<CG>(mA, sA, fb, boxA, b, m0, k0);
                    if (do_b && b < boxB.nbox)
                        issue_box<CG>(mB, sB, fb, boxB, b, n0, k0);
                }
            }
            if constexpr (SF) {
                // the scale atoms of this K range: this CTA's A rows (with the A
                // boxes), and every B column of the tile (with the B boxes; the
                // pair's MMA reads all of them from each CTA). The scale tensors
                // are viewed as rows of 256 bytes, atom a being rows 2a and 2a + 1;
                // a row block's atoms of consecutive K groups are adjacent, so one
                // box of 2 x KGROUPS rows brings all of a stage's atoms of one row
                // block. Atoms past the last K group (the tail of the last stage:
                // the next row block's, or TMA's zero fill past the end) multiply
                // only the zeros TMA fills in for K. Pair CTAs signal the even
                // CTA's barrier like the operand boxes.
                const uint32_t sSF = sA + C::SF_OFF;
                const int g0 = k0 / sf_atom_kbytes(SF);
                const int ra = m0 / 128, rb = ti.n_blk * BN / 128;
                if (do_a) {
                    if constexpr (CG == 1)
                        tma_load_2d(sSF, tmSFA, fb, 0, 2 * (ra * sf_groups + g0));
                    else
                        tma_load_2d_pair(sSF, tmSFA, fb, 0, 2 * (ra * sf_groups + g0));
                }
                if (do_b) {
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h) {
                        const uint32_t dst = sSF + C::SF_A_BYTES + 512 * C::KGROUPS * h;
                        if constexpr (CG == 1)
                            tma_load_2d(dst, tmSFB, fb, 0, 2 * ((rb + h) * sf_groups + g0));
                        else
                            tma_load_2d_pair(dst, tmSFB, fb, 0, 2 * ((rb + h) * sf_groups + g0));
                    }
                }
            }
            ++issued;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (stats && part != 2) {
        stats[blockIdx.x * kStatSlots + kStatProducerWaitCycles] = st_wait;
        stats[blockIdx.x * kStatSlots + kStatProducerBlocked] = st_blocked;
    }
    return ProducerTail{issued < STAGES ? issued : STAGES, stage, phase};
}

// After an abort: wait (bounded) until the loads of the last stages the
// producer filled have landed, so that no copy writes into shared memory of a
// CTA that has exited. The full barrier of a stage completes once all its
// bytes arrived (for a CTA pair, the even CTA's barrier counts the bytes of
// both CTAs); a stage already consumed has completed its phase and returns at
// once.
template <int STAGES>
__device__ void drain_producer_tail(const ProducerTail &t, uint32_t bar_full, const Waiter &w)
{
    for (int i = 1; i <= t.inflight; ++i) {
        int s = t.stage - i;
        uint32_t ph = t.phase;
        if (s < 0) {
            s += STAGES;
            ph ^= 1u;
        }
        w.drain(bar_full + 8 * s, ph, 2000000ull);
    }
}

// Scale copier (block-scaled kinds, warp 6 of the even CTA): for every stage
// of every unit, in the order the MMA issuer consumes them, waits until the
// stage has landed, copies its scale atoms from shared memory into the stage's
// TMEM scale columns (tcgen05.cp, 32x128b.warpx4) and commits to sf_ready of
// the stage, which arrives once the copies have completed. The MMA issuer
// waits on sf_ready before the stage's MMAs and so issues only MMAs. A
// stage's scale columns are rewritten only after the stage was refilled, that
// is after the MMAs that read their previous contents completed.
template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
__device__ void role_sf_copy(const KParams &p, uint32_t smem, uint32_t bar_full, uint32_t bar_sf,
                             uint32_t tmem_base, const Waiter &w, int copier)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>;
    if constexpr (SF != 0) {
        if (p.inject_timeout == kRoleMma)
            return;
        const Sched sched = make_sched(p);
        unsigned long long *const stats = p.stats;
        unsigned long long st_wait = 0;
        const int cluster_id = blockIdx.x / C::CLUSTER, num_clusters = gridDim.x / C::CLUSTER;
        int stage = 0;
        uint32_t phase = 0;
        UnitIter units(sched, cluster_id, num_clusters);
        Unit u;
        while (units.next(u)) {
            TileInfo ti;
            decode_tile<GROUPED>(sched, u.tile, ti);
            const int num_kb = ceil_div_i(ti.K, BK);
            const int kb_lo = u.kb0, kb_hi = u.kb1 < 0 ? num_kb : u.kb1;
            for (int kb = kb_lo; kb < kb_hi; ++kb) {
                const long long t0 = stats ? clock64() : 0;
                if (!w.wait(bar_full + 8 * stage, phase, kRoleSfCopy | kWaitFull))
                    return;
                if (stats)
                    st_wait += static_cast<unsigned long long>(clock64() - t0);
                tc_fence_after_sync();
                const uint32_t sSF = smem + stage * C::STAGE_BYTES + C::SF_OFF;
                const uint32_t tsf = tmem_base + static_cast<uint32_t>(C::SF_COL0 + stage * C::SF_COLS);
                // with several copiers, copier c takes the K groups g = c mod copiers
#pragma unroll
                for (int g = 0; g < C::KGROUPS; ++g) {
                    if (g % C::SF_COPIERS != copier)
                        continue;
                    const uint32_t tg = tsf + static_cast<uint32_t>(C::SF_GROUP_COLS * g);
                    tmem_cp_32x128b_warpx4<CG>(tg, make_smem_desc(sSF + 512 * g, 128, 128, 0));
                    // B scales of columns 128h..128h+127 in the next 4 columns each
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h)
                        tmem_cp_32x128b_warpx4<CG>(
                            tg + 4 + 4 * h, make_smem_desc(sSF + C::SF_A_BYTES + 512 * (C::KGROUPS * h + g), 128, 128, 0));
                }
                mma_commit<CG>(bar_sf + 8 * stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (stats && copier == 0)
            stats[blockIdx.x * kStatSlots + kStatSfCopyWaitCycles] = st_wait;
    } else {
        (void)p;
        (void)smem;
        (void)bar_full;
        (void)bar_sf;
        (void)tmem_base;
        (void)w;
        (void)copier;
    }
}

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
__device__ void role_mma(const KParams &p, uint32_t smem, uint32_t bar_full, uint32_t bar_empty,
                         uint32_t bar_acc_full, uint32_t bar_acc_empty, uint32_t bar_inject, uint32_t bar_sf,
                         uint32_t tmem_base, const Waiter &w)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>;
    if (p.inject_timeout == kRoleMma) {
        // Test hook: wait on a barrier nothing arrives at; the bound runs out.
        w.wait(bar_inject, 0u, kRoleMma | kWaitInjected);
        return;
    }
    const Sched sched = make_sched(p);
    unsigned long long *const stats = p.stats;
    const bool multicast = CG == 2 && !(p.flags & kFlagPairForward);
    // B multicast: a stage is refilled in both CTAs at once, so each CTA's MMA
    // completion releases the stage in both
    const uint32_t idesc = SF ? make_idesc_mx(C::UMMA_M, BN, p.a_fmt, p.b_fmt, p.a_mn, p.b_mn, SF != kScaleNv4)
                              : make_idesc(C::UMMA_M, BN, p.a_fmt, p.b_fmt, p.a_mn, p.b_mn);
    const OperandPacking pa = operand_packing(p.a_mn, p.a_swz, C::BM, BK);
    const OperandPacking pb = operand_packing(p.b_mn, p.b_swz, C::BN_LOCAL, BK);
    const uint64_t a_desc0 = make_smem_desc(smem, pa.lbo, pa.sbo, pa.swz);
    const uint64_t b_desc0 = make_smem_desc(smem + C::A_BYTES, pb.lbo, pb.sbo, pb.swz);
    uint32_t a_off[C::KSLICES], b_off[C::KSLICES];
    // two-half tiles: rows 128..255 of the A tile start 128 * W bytes further
    // on in a K-major stage (rows of W bytes), 128 * ESIZE * BK bytes in an
    // MN-major one (each MN element holds BK rows of K)
    const uint32_t a_half = C::M_HALVES == 2 ? (p.a_mn ? 128u * ESIZE * BK : 128u * swizzle_row_bytes(p.a_swz)) >> 4 : 0u;
#pragma unroll
    for (int j = 0; j < C::KSLICES; ++j) {
        a_off[j] = slice_byte_offset(p.a_mn, p.a_swz, C::BM, j, ESIZE) >> 4;
        b_off[j] = slice_byte_offset(p.b_mn, p.b_swz, C::BN_LOCAL, j, ESIZE) >> 4;
    }
    const int cluster_id = blockIdx.x / C::CLUSTER, num_clusters = gridDim.x / C::CLUSTER;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    unsigned long long st_full = 0, st_acc = 0, st_blocked = 0, st_tiles = 0, st_sf = 0;
    const long long t_start = clock64();
    UnitIter units(sched, cluster_id, num_clusters);
    Unit u;
    while (units.next(u)) {
        TileInfo ti;
        decode_tile<GROUPED>(sched, u.tile, ti);
        const int num_kb = ceil_div_i(ti.K, BK);
        const int kb_lo = u.kb0, kb_hi = u.kb1 < 0 ? num_kb : u.kb1;
        if (kb_hi <= kb_lo)
            continue;  // K == 0: the epilogue writes beta * C without the accumulator
        {
            const long long t0 = stats ? clock64() : 0;
            if (!w.wait(bar_acc_empty + 8 * acc, acc_phase ^ 1u, kRoleMma | kWaitAccEmpty, CG == 2))
                return;
            if (stats)
                st_acc += static_cast<unsigned long long>(clock64() - t0);
            ++st_tiles;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = C::WS        ? tmem_base + static_cast<uint32_t>(acc * C::ACC_COLS)
                                : C::BM == 64 ? tmem_base + (static_cast<uint32_t>(16 * acc) << 16)
                                              : tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (stats) {
                const long long t0 = clock64();
                const bool ready = mbar_try_wait(bar_full + 8 * stage, phase);
                if (!ready && !w.wait(bar_full + 8 * stage, phase, kRoleMma | kWaitFull))
                    return;
                st_full += static_cast<unsigned long long>(clock64() - t0);
                st_blocked += ready ? 0 : 1;
            } else if (!mbar_try_wait(bar_full + 8 * stage, phase) &&
                       !w.wait(bar_full + 8 * stage, phase, kRoleMma | kWaitFull)) {
                return;
            }
            tc_fence_after_sync();
            const uint64_t sdelta = static_cast<uint64_t>((stage * C::STAGE_BYTES) >> 4);
            if constexpr (SF) {
                // the copier warp has put this stage's scale atoms in its TMEM
                // scale columns; its commit arrives once the copies completed
                const long long t0 = stats ? clock64() : 0;
                if (!mbar_try_wait(bar_sf + 8 * stage, phase) &&
                    !w.wait(bar_sf + 8 * stage, phase, kRoleMma | kWaitSfReady))
                    return;
                if (stats)
                    st_sf += static_cast<unsigned long long>(clock64() - t0);
                tc_fence_after_sync();
                const uint32_t tsf = tmem_base + static_cast<uint32_t>(C::SF_COL0 + stage * C::SF_COLS);
                // each 32-byte K slice (one MMA) reads the atom holding its blocks
                // and, by its scale factor ID, the first of its bytes in each column
                constexpr int kPerAtom = sf_atom_kbytes(SF) / 32;  // MMAs per atom: 4, 1, 2
#pragma unroll
                for (int j = 0; j < C::KSLICES; ++j) {
                    const uint32_t ts = tsf + static_cast<uint32_t>(C::SF_GROUP_COLS * (j / kPerAtom));
                    const int id = (j % kPerAtom) * (4 / kPerAtom);
                    mma_scaled<CG, SF>(d_tmem, a_desc0 + sdelta + a_off[j], b_desc0 + sdelta + b_off[j],
                                       idesc_sf_ids(idesc, id, id), ts, ts + 4, ((kb - kb_lo) | j) != 0);
                }
            } else {
#pragma unroll
                for (int j = 0; j < C::KSLICES; ++j) {
                    // the first MMA of a unit overwrites the accumulator, the rest add
                    if constexpr (C::WS)
                        mma_ws_f16(d_tmem, a_desc0 + sdelta + a_off[j], b_desc0 + sdelta + b_off[j], idesc,
                                   ((kb - kb_lo) | j) != 0);
                    else if constexpr (ESIZE == 2) {
                        mma_f16<CG>(d_tmem, a_desc0 + sdelta + a_off[j], b_desc0 + sdelta + b_off[j], idesc,
                                    ((kb - kb_lo) | j) != 0);
                        if constexpr (C::M_HALVES == 2)  // the same B slice, rows 128..255 of A
                            mma_f16<CG>(d_tmem + C::HALF_COL, a_desc0 + sdelta + a_off[j] + a_half, b_desc0 + sdelta + b_off[j],
                                        idesc, ((kb - kb_lo) | j) != 0);
                    }
                    else if constexpr (ESIZE == 4)
                        mma_tf32<CG>(d_tmem, a_desc0 + sdelta + a_off[j], b_desc0 + sdelta + b_off[j], idesc,
                                     ((kb - kb_lo) | j) != 0);
                    else {
                        mma_f8<CG>(d_tmem, a_desc0 + sdelta + a_off[j], b_desc0 + sdelta + b_off[j], idesc,
                                   ((kb - kb_lo) | j) != 0);
                        if constexpr (C::M_HALVES == 2)
                            mma_f8<CG>(d_tmem + C::HALF_COL, a_desc0 + sdelta + a_off[j] + a_half, b_desc0 + sdelta + b_off[j],
                                       idesc, ((kb - kb_lo) | j) != 0);
                    }
                }
            }
            if constexpr (C::MCB)
                mma_commit_cg1_multicast(bar_empty + 8 * stage);
            else if (multicast)
                mma_commit_pair_multicast(bar_empty + 8 * stage);
            else
                mma_commit<CG>(bar_empty + 8 * stage);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (multicast)
            mma_commit_pair_multicast(bar_acc_full + 8 * acc);
        else
            mma_commit<CG>(bar_acc_full + 8 * acc);
        if (++acc == C::ACC_BUFS) {
            acc = 0;
            acc_phase ^= 1u;
        }
    }
    if (stats) {
        unsigned long long *o = stats + blockIdx.x * kStatSlots;
        o[kStatMmaFullWaitCycles] = st_full;
        o[kStatMmaAccEmptyWaitCycles] = st_acc;
        o[kStatMmaLoopCycles] = static_cast<unsigned long long>(clock64() - t_start);
        o[kStatMmaFullBlocked] = st_blocked;
        o[kStatTiles] = st_tiles;
        o[kStatMmaSfWaitCycles] = st_sf;
    }
}

// Convert 8 fp32 values to a 16-byte chunk of the output type.
__device__ __forceinline__ void pack_out(const float *v, int out_type, uint32_t (&o)[4])
{
    if (out_type == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            o[i] = *reinterpret_cast<uint32_t *>(&h);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            o[i] = *reinterpret_cast<uint32_t *>(&h);
        }
    }
}

__device__ __forceinline__ void unpack_in(const uint32_t (&c)[4], int out_type, float *v)
{
    if (out_type == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&c[i]);
            float2 f = __bfloat1622float2(h);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&c[i]);
            float2 f = __half22float2(h);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
}

struct EpiConst {
    float alpha, beta;
    int out_type;
    uint32_t key_mask;  // 7 when staging rows are SW128-swizzled, else 0
};

// This thread's 128 bytes of C for one chunk (row `row`, columns col0..),
// read from global memory into registers: whole 16-byte units inside N,
// single elements (predicated, fixed indices) at the N edge, zeros past the
// matrix.
template <int CW>
__device__ __forceinline__ void load_c_row(uint32_t (&cr)[32], const void *c_ptr, long long ldc, int row, int col0,
                                           int M, int N)
{
    constexpr int OB = CW == 32 ? 4 : 2;  // output element bytes
#pragma unroll
    for (int i = 0; i < 32; ++i)
        cr[i] = 0u;
    if (row >= M)
        return;
    const char *rp = static_cast<const char *>(c_ptr) + (static_cast<long long>(row) * ldc + col0) * OB;
    const int nv = N - col0;  // valid columns of the chunk
    if (nv >= CW) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 x = __ldg(reinterpret_cast<const uint4 *>(rp) + u);
            cr[4 * u] = x.x;
            cr[4 * u + 1] = x.y;
            cr[4 * u + 2] = x.z;
            cr[4 * u + 3] = x.w;
        }
    } else if constexpr (OB == 4) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nv)
                cr[i] = __ldg(reinterpret_cast<const uint32_t *>(rp) + i);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t lo = 2 * i < nv ? __ldg(reinterpret_cast<const unsigned short *>(rp) + 2 * i) : 0u;
            const uint32_t hi = 2 * i + 1 < nv ? __ldg(reinterpret_cast<const unsigned short *>(rp) + 2 * i + 1) : 0u;
            cr[i] = lo | (hi << 16);
        }
    }
}

// This thread's 128 bytes of D for one chunk (row `row`, columns col0..),
// written from registers: whole 16-byte units inside N, single elements at
// the N edge, nothing past the matrix. `o` holds the chunk in the output type.
template <int CW>
__device__ __forceinline__ void store_d_row(const uint32_t (&o)[32], void *d_ptr, long long ldd, int row, int col0,
                                            int M, int N)
{
    constexpr int OB = CW == 32 ? 4 : 2;  // output element bytes
    if (row >= M)
        return;
    char *rp = static_cast<char *>(d_ptr) + (static_cast<long long>(row) * ldd + col0) * OB;
    const int nv = N - col0;  // valid columns of the chunk
    constexpr int PER16 = 16 / OB;  // elements per 16-byte unit
    if (nv >= CW || nv % PER16 == 0) {  // whole 16-byte units (all, or the first nv / PER16)
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u * PER16 < nv)
                reinterpret_cast<uint4 *>(rp)[u] = make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
    } else if constexpr (OB == 4) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nv)
                reinterpret_cast<uint32_t *>(rp)[i] = o[i];
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (2 * i < nv)
                reinterpret_cast<unsigned short *>(rp)[2 * i] = static_cast<unsigned short>(o[i] & 0xFFFFu);
            if (2 * i + 1 < nv)
                reinterpret_cast<unsigned short *>(rp)[2 * i + 1] = static_cast<unsigned short>(o[i] >> 16);
        }
    }
}

// alpha * acc + beta * C for one chunk of this thread's row, in the output
// type, C from registers (`creg`, as load_c_row leaves it)
template <int CW>
__device__ __forceinline__ void chunk_math_regs(float (&acc)[CW], const EpiConst &e, bool use_c, const uint32_t (&creg)[32],
                                                uint32_t (&o)[32])
{
    constexpr int PER16 = (CW == 32) ? 4 : 8;  // elements per 16-byte unit
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        float *v = acc + u * PER16;
#pragma unroll
        for (int i = 0; i < PER16; ++i)
            v[i] *= e.alpha;
        if (use_c) {
            const uint32_t c[4] = {creg[4 * u], creg[4 * u + 1], creg[4 * u + 2], creg[4 * u + 3]};
            if constexpr (CW == 32) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    v[i] = fmaf(e.beta, __uint_as_float(c[i]), v[i]);
            } else {
                float cf[8];
                unpack_in(c, e.out_type, cf);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = fmaf(e.beta, cf[i], v[i]);
            }
        }
        uint32_t w[4];
        if constexpr (CW == 32) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = __float_as_uint(v[i]);
        } else {
            pack_out(v, e.out_type, w);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[4 * u + i] = w[i];
    }
}

// One 32-row x 128-byte chunk: fp32 output covers 32 columns, 16-bit output 64.
// `acc` holds this thread's row (lane) of the chunk in fp32. C comes from the
// staging buffer (swizzled like the output), or from `creg` when CREG. The
// output type (OT: 0 fp32, 1 bf16, 2 fp16) and alpha == 1 (A1) are fixed at
// compile time, and the eight stores follow all the arithmetic, so that a
// lone epilogue warp is not held by a branch or a store between conversions
// (measured: 690 -> 590 cycles per bf16 chunk, 512 -> 340 per fp32 chunk).
template <int CW, bool CREG, int OT, bool A1>
__device__ __forceinline__ void chunk_math_staged(float (&acc)[CW], const EpiConst &e, uint32_t sbuf, int r,
                                                  bool use_c, const uint32_t *creg)
{
    const uint32_t row = sbuf + static_cast<uint32_t>(r) * 128u;
    const uint32_t key = static_cast<uint32_t>(r) & e.key_mask;
    constexpr int PER16 = (CW == 32) ? 4 : 8;  // elements per 16-byte unit
    uint32_t o[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        float *v = acc + u * PER16;
        if constexpr (!A1) {
#pragma unroll
            for (int i = 0; i < PER16; ++i)
                v[i] *= e.alpha;
        }
        if (use_c) {
            uint32_t c[4];
            if constexpr (CREG) {
                c[0] = creg[4 * u];
                c[1] = creg[4 * u + 1];
                c[2] = creg[4 * u + 2];
                c[3] = creg[4 * u + 3];
            } else {
                ld_shared_v4(row + ((static_cast<uint32_t>(u) ^ key) << 4), c[0], c[1], c[2], c[3]);
            }
            if constexpr (CW == 32) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    v[i] = fmaf(e.beta, __uint_as_float(c[i]), v[i]);
            } else {
                float cf[8];
                unpack_in(c, OT, cf);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = fmaf(e.beta, cf[i], v[i]);
            }
        }
        if constexpr (CW == 32) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[u][i] = __float_as_uint(v[i]);
        } else {
            pack_out(v, OT, o[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
        st_shared_v4(row + ((static_cast<uint32_t>(u) ^ key) << 4), o[u][0], o[u][1], o[u][2], o[u][3]);
}

template <int CW, bool CREG = false>
__device__ __forceinline__ void epilogue_chunk_math(float (&acc)[CW], const EpiConst &e,
                                                    uint32_t sbuf, int r, bool use_c, const uint32_t *creg = nullptr)
{
    const bool a1 = e.alpha == 1.0f;
    if constexpr (CW == 32) {
        if (a1)
            chunk_math_staged<CW, CREG, 0, true>(acc, e, sbuf, r, use_c, creg);
        else
            chunk_math_staged<CW, CREG, 0, false>(acc, e, sbuf, r, use_c, creg);
    } else if (e.out_type == 1) {
        if (a1)
            chunk_math_staged<CW, CREG, 1, true>(acc, e, sbuf, r, use_c, creg);
        else
            chunk_math_staged<CW, CREG, 1, false>(acc, e, sbuf, r, use_c, creg);
    } else {
        if (a1)
            chunk_math_staged<CW, CREG, 2, true>(acc, e, sbuf, r, use_c, creg);
        else
            chunk_math_staged<CW, CREG, 2, false>(acc, e, sbuf, r, use_c, creg);
    }
}

// The clusters that hold the rest of split tile `ua` (its head): [*lo, *hi];
// a cluster whose share of the split iterations is empty holds nothing.
__device__ __forceinline__ void sk_contributors(const Sched &sched, const Unit &ua, int num_clusters, int *lo, int *hi)
{
    const long long first = static_cast<long long>(ua.tile - sched.sk_dp) * sched.kbt;
    *lo = sk_owner(first + ua.kb1, sched.sk_iters, num_clusters);
    *hi = sk_owner(first + sched.kbt - 1, sched.sk_iters, num_clusters);
}

__device__ __forceinline__ bool sk_share_empty(long long S, int cc, int num_clusters)
{
    return S * cc / num_clusters == S * (cc + 1) / num_clusters;
}

// Waits until every contributor of split tile `ua` has published the partial
// sum of this warp's lane quarter (flag row of CTA cc * CL + rank, word q).
template <int CL>
__device__ bool sk_wait_contributors(const Sched &sched, const Unit &ua, int q, const uint32_t *sk_flags,
                                     uint32_t epoch, int rank, int num_clusters, const Waiter &w,
                                     unsigned long long *st_wait)
{
    int c_lo, c_hi;
    sk_contributors(sched, ua, num_clusters, &c_lo, &c_hi);
    const long long t0 = st_wait ? clock64() : 0;
    bool ok = true;
    for (int cc = c_lo; cc <= c_hi && ok; ++cc) {
        if (sk_share_empty(sched.sk_iters, cc, num_clusters))
            continue;  // empty share: nothing to wait for
        ok = w.wait_flag(sk_flags + (cc * CL + rank) * 4 + q, epoch, kRoleEpilogue | kWaitPartial);
    }
    if (!__all_sync(0xffffffffu, ok))
        return false;
    if (st_wait)
        *st_wait += static_cast<unsigned long long>(clock64() - t0);
    return true;
}

// Stream-K head gather, one epilogue warp (TMEM lane quarter q, rows
// 32q..32q+31): waits for the flags of the clusters that hold the rest of
// split tile `ua`, then writes the sum of their fp32 partial sums into TMEM
// accumulator buffer `buf` (the first n32 32-column groups), the buffer the
// head's own MMAs do not use. False if a flag did not come in time.
template <int CL, int BN>
__device__ bool sk_gather(const Sched &sched, const Unit &ua, int n32, int buf, uint32_t tmem_base, int q,
                          int prow, const float4 *partials, const uint32_t *sk_flags, uint32_t epoch, int rank,
                          int num_clusters, const Waiter &w, unsigned long long *st_wait)
{
    const long long S = sched.sk_iters;
    if (!sk_wait_contributors<CL>(sched, ua, q, sk_flags, epoch, rank, num_clusters, w, st_wait))
        return false;
    int c_lo, c_hi;
    sk_contributors(sched, ua, num_clusters, &c_lo, &c_hi);
    constexpr int kSlotVec = 128 * BN / 4;  // float4 per slot
    constexpr int kGroups = 2;              // 32-column groups per batch of loads
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * BN);
    for (int c0 = 0; c0 < n32; c0 += kGroups) {
        float v[kGroups][32];
#pragma unroll
        for (int b = 0; b < kGroups; ++b)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                v[b][i] = 0.0f;
#pragma unroll 1
        for (int cc = c_lo; cc <= c_hi; ++cc) {
            if (sk_share_empty(S, cc, num_clusters))
                continue;
            const float4 *slot = partials + static_cast<size_t>(cc * CL + rank) * kSlotVec + prow;
#pragma unroll
            for (int b = 0; b < kGroups; ++b) {
                // groups past n32 reload the last one (in the slot) and are not stored
                const int cb = min(c0 + b, n32 - 1);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const float4 x = __ldcg(slot + (cb * 8 + g) * 128);
                    v[b][4 * g] += x.x;
                    v[b][4 * g + 1] += x.y;
                    v[b][4 * g + 2] += x.z;
                    v[b][4 * g + 3] += x.w;
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kGroups; ++b)
            if (c0 + b < n32)
                tmem_st_32x32b_x32(tbase + static_cast<uint32_t>((c0 + b) * 32), v[b]);
    }
    tmem_st_wait();  // the head's epilogue (this warp) reads the buffer back
    return true;
}

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE, int CW>
__device__ void role_epilogue(const KParams &p, const CUtensorMap *tmC, const CUtensorMap *tmD,
                              uint32_t epi_base, uint32_t bar_acc_full, uint32_t bar_acc_empty,
                              uint32_t bar_epi, uint32_t tmem_base, uint32_t rank, int warp,
                              int lane, const Waiter &w)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>;
    const Sched sched = make_sched(p);
    unsigned long long *const stats = p.stats;
    const CUtensorMap *const maps = p.maps;
    EpiConst ec;
    ec.alpha = p.alpha;
    ec.beta = p.beta;
    ec.out_type = p.out_type;
    ec.key_mask = p.epi_swizzle ? 7u : 0u;
    const bool forward = CG == 2 && rank == 0 && (p.flags & kFlagPairForward);
    const int q = warp & 3;   // TMEM lane quarter 32q..32q+31
    constexpr int R = C::EPI_ROWS;
    // The rows and column chunks this warp stores: 128-row tiles and Layout F
    // give each warp R rows (lane quarter q = rows R q..) of every chunk; .ws
    // tiles give it 32 rows of one column part (rows 32 (q % RB) .., chunks
    // [part * NCH / COL_PARTS, (part + 1) * NCH / COL_PARTS))
    // chunks per row; a two-half tile 224 wide ends in a chunk of 32 columns
    // (16-bit output), which the epilogue writes from registers
    constexpr int NCH = (BN + CW - 1) / CW;
    const int wrow = C::WS ? 32 * (q % C::WS_ROW_BLOCKS) : R * q;
    const int c_lo = C::WS ? (q / C::WS_ROW_BLOCKS) * (NCH / C::COL_PARTS) : 0;
    const int c_hi = c_lo + NCH / C::COL_PARTS;
    const int ew = warp - 2;  // staging slot
    const uint32_t buf0 = epi_base + static_cast<uint32_t>(ew * C::EPI_BUFS * kEpiBufBytes);
    const uint32_t ebar0 = bar_epi + static_cast<uint32_t>(16 * ew);
    const bool use_c = ec.beta != 0.0f;
    // C straight into registers: single problems with 128-row tiles (each
    // thread owns one output row of a chunk)
    // D straight from registers (single problems, tiles whose rows are the
    // threads' lanes); C then comes into registers too
    const bool direct_d = !GROUPED && C::BM >= 128 && !C::WS && (p.flags & kFlagDirectD) != 0;
    const bool direct_c = use_c && !GROUPED && C::BM >= 128 && !C::WS && ((p.flags & kFlagDirectC) != 0 || direct_d);
    const void *const c_ptr = p.c_ptr;
    const long long ldc = p.ldc;
    void *const d_ptr = p.d_ptr;
    const long long ldd = p.ldd;
    // C and D pass through once: let them leave L2 first
    const bool hints = (p.flags & kFlagCacheHints) != 0;
    const uint64_t stream_once = hints ? l2_policy_evict_first() : 0;
    const uint32_t acc_empty_target = (CG == 2) ? mapa_shared(bar_acc_empty, 0) : bar_acc_empty;
    const uint32_t peer_acc_full = (CG == 2 && rank == 0) ? mapa_shared(bar_acc_full, 1) : 0u;
    const int cluster_id = blockIdx.x / C::CLUSTER, num_clusters = gridDim.x / C::CLUSTER;
    uint32_t epi_phase[2] = {0u, 0u};
    int sel = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    unsigned long long st_accw = 0, st_cw = 0, st_pw = 0, st_pe = 0;
    long long t_last_acc = 0;
    const long long t_start = clock64();
    // stream-K: this CTA's partial-sum slot, and its row in every slot
    // 128-row tiles gather partial sums into the spare accumulator buffer;
    // two-half tiles (no spare buffer) add them from the workspace per chunk
    constexpr bool kStreamK = !GROUPED && ((C::BM == 128 && C::ACC_BUFS == 2) || C::M_HALVES == 2);
    const bool split = kStreamK && sched.sk_iters > 0;
    float4 *const partials = reinterpret_cast<float4 *>(p.sk_partials);
    uint32_t *const sk_flags = p.sk_flags;
    const uint32_t epoch = p.sk_epoch;
    const int prow = R * q + lane;
    constexpr int kSlotRows = 128 * C::M_HALVES;   // rows of a partial-sum slot
    constexpr int kSlotVec = kSlotRows * BN / 4;   // float4 per slot
    int sk_lo = 0, sk_hi = -1;                     // a two-half head's contributors
    int last_prob = -1;                            // grouped: problem whose C/D maps were acquired
    UnitIter units(sched, cluster_id, num_clusters);
    Unit u;
    while (units.next(u)) {
        TileInfo ti;
        decode_tile<GROUPED>(sched, u.tile, ti);
        // a contributor leaves its partial sum for the tile's head; the head
        // adds those partials (gathered into the spare accumulator buffer)
        const int kind = split ? unit_kind(u, sched.kbt) : kUnitWhole;
        const bool contributor = kind == kUnitContributor;
        const bool head = kind == kUnitHead;
        if (head) {
            const int n_cols = min(BN, ti.N - ti.n_blk * BN);
            const long long t0 = stats ? clock64() : 0;
            bool ok;
            if constexpr (C::M_HALVES == 2) {
                ok = sk_wait_contributors<C::CLUSTER>(sched, u, q, sk_flags, epoch, static_cast<int>(rank),
                                                      num_clusters, w, stats ? &st_pw : nullptr);
                sk_contributors(sched, u, num_clusters, &sk_lo, &sk_hi);
            } else {
                ok = sk_gather<C::CLUSTER, BN>(sched, u, (n_cols + 31) / 32, acc ^ 1, tmem_base, q, prow, partials,
                                               sk_flags, epoch, static_cast<int>(rank), num_clusters, w,
                                               stats ? &st_pw : nullptr);
            }
            if (stats)
                st_pe += static_cast<unsigned long long>(clock64() - t0);
            if (!ok)
                return;
        }
        const CUtensorMap *mC = tmC, *mD = tmD;
        if constexpr (GROUPED) {
            mC = maps + 4 * ti.prob + 2;
            mD = mC + 1;
            if (ti.prob != last_prob) {  // once per problem, as the producer does for A and B
                fence_tensormap_acquire(mC);
                fence_tensormap_acquire(mD);
                last_prob = ti.prob;
            }
        }
        const bool has_acc = ti.K > 0;
        const int m0 = ti.m_blk * C::TILE_M + C::BM * static_cast<int>(rank) + wrow;
        // 128-row and .ws tiles: thread t holds row t of the warp's rows. 64-row
        // tiles (Layout F): the accumulator with lane alignment 16*acc sits in
        // threads 16*acc..+15.
        const bool active = C::WS || C::BM >= 128 || (lane >> 4) == acc;
        const int trow = (C::WS || C::BM >= 128) ? lane : (lane & 15);
        if (has_acc) {
            const long long tw = stats ? clock64() : 0;
            bool ok = w.wait(bar_acc_full + 8 * acc, acc_phase, kRoleEpilogue | kWaitAccFull, rank != 0);
            if (stats) {
                t_last_acc = clock64();
                st_accw += static_cast<unsigned long long>(t_last_acc - tw);
            }
            if (!__all_sync(0xffffffffu, ok))
                return;
            if (forward && ew == 0 && lane == 0)
                mbar_arrive_cluster(peer_acc_full + 8 * acc);  // the odd CTA's half is complete too
            tc_fence_after_sync();
        }
        if (contributor) {
            // contributor: the accumulator goes to this CTA's slot as fp32,
            // laid out [column / 4][row][4] so that a warp writes 512
            // contiguous bytes per store
            float4 *const slot = partials + static_cast<size_t>(blockIdx.x) * kSlotVec;
            for (int half = 0; half < C::M_HALVES; ++half) {
                // 32-column groups of the tile (BN is a multiple of 32)
                for (int c32 = 0; c32 < BN / 32; ++c32) {
                    if (ti.n_blk * BN + c32 * 32 >= ti.N)
                        break;
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                           static_cast<uint32_t>((C::M_HALVES == 2 ? half * C::HALF_COL : acc * BN) +
                                                                 c32 * 32);
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        __stcg(slot + (c32 * 8 + g) * kSlotRows + 128 * half + prow,
                               make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                           __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])));
                }
            }
            tc_fence_before_sync();
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                st_release_gpu(sk_flags + blockIdx.x * 4 + q, epoch);
                if constexpr (CG == 2)
                    mbar_arrive_cluster(acc_empty_target + 8 * acc);
                else
                    mbar_arrive(bar_acc_empty + 8 * acc);
            }
            if (++acc == C::ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
            continue;
        }
        if constexpr (C::ACC_BUFS == 1 && C::BM == 128 && CW == 64) {
            if (has_acc && !use_c && !head) {
                // One accumulator buffer, 16-bit output, no C: read the whole row
                // and round it in registers first, then release the accumulator,
                // so that the next tile's MMAs run while the stores drain.
                uint32_t pk[NCH][32];
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(c * CW);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(taddr + 32 * h, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            float v[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                v[i] = ec.alpha * __uint_as_float(r[8 * u + i]);
                            uint32_t o[4];
                            pack_out(v, ec.out_type, o);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                pk[c][16 * h + 4 * u + i] = o[i];
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (CG == 2)
                        mbar_arrive_cluster(acc_empty_target + 8 * acc);
                    else
                        mbar_arrive(bar_acc_empty + 8 * acc);
                }
                if (++acc == C::ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                const uint32_t key = static_cast<uint32_t>(trow) & ec.key_mask;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    const int col0 = ti.n_blk * BN + c * CW;
                    if (col0 >= ti.N)
                        break;
                    const uint32_t sbuf = buf0 + static_cast<uint32_t>(sel * kEpiBufBytes);
                    if (lane == 0)
                        bulk_wait_group_read<C::EPI_BUFS - 1>();
                    __syncwarp();
                    const uint32_t row = sbuf + static_cast<uint32_t>(trow) * 128u;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(row + ((static_cast<uint32_t>(u) ^ key) << 4), pk[c][4 * u], pk[c][4 * u + 1],
                                     pk[c][4 * u + 2], pk[c][4 * u + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (hints)
                            tma_store_2d_hint(mD, sbuf, col0, m0, stream_once);
                        else
                            tma_store_2d(mD, sbuf, col0, m0);
                        bulk_commit_group();
                    }
                    if constexpr (C::EPI_BUFS == 2)
                        sel ^= 1;
                }
                continue;
            }
        }
        // two-half tiles store the rows of one half after the other (row
        // offset 128 h, accumulator columns from h HALF_COL); other tiles have one
        for (int half = 0; half < C::M_HALVES; ++half) {
            for (int c = c_lo; c < c_hi; ++c) {
                const int col0 = ti.n_blk * BN + c * CW;
                if (col0 >= ti.N)
                    break;
                const int m0h = m0 + 128 * half;
                // a chunk that runs past the tile (the last one of a 224-wide
                // tile with 16-bit output) is read and written from registers,
                // its columns cut at the tile's edge
                const bool part = (c + 1) * CW > BN;
                const bool dd = direct_d || part, dc = direct_c || (part && use_c);
                const int n_lim = part ? min(ti.N, ti.n_blk * BN + BN) : ti.N;
                const uint32_t sbuf = buf0 + static_cast<uint32_t>(sel * kEpiBufBytes);
                const uint32_t sbar = ebar0 + static_cast<uint32_t>(8 * sel);
                // the store issued from this buffer (EPI_BUFS chunks ago) must have read it
                if (lane == 0 && !dd)
                    bulk_wait_group_read<C::EPI_BUFS - 1>();
                __syncwarp();
                uint32_t creg[32];
                if (dc)  // issued before the TMEM load so that the two overlap
                    load_c_row<CW>(creg, c_ptr, ldc, m0h + trow, col0, ti.M, n_lim);
                if (use_c && !dc && lane == 0) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(sbar, R * 128);
                    if (hints)
                        tma_load_2d_hint(sbuf, mC, sbar, col0, m0h, stream_once);
                    else
                        tma_load_2d(sbuf, mC, sbar, col0, m0h);
                }
                __syncwarp();  // tcgen05.ld is .sync.aligned: the warp must be converged
                float v[CW];
                if (has_acc) {
                    const uint32_t col = static_cast<uint32_t>(
                        C::WS ? acc * C::ACC_COLS + (c - c_lo) * CW
                              : (C::BM == 128 ? acc * BN : C::M_HALVES == 2 ? half * C::HALF_COL : 0) + c * CW);
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + col;
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr, r);
                    if constexpr (CW == 64) {
                        uint32_t r2[32];
                        tmem_ld_32x32b_x32(taddr + 32, r2);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            v[i] = __uint_as_float(r[i]);
                            v[32 + i] = __uint_as_float(r2[i]);
                        }
                    } else {
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = __uint_as_float(r[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        v[i] = 0.0f;
                }
                if (head && C::M_HALVES == 2) {
                    // the contributors' partial sums of this chunk, from their slots
#pragma unroll 1
                    for (int cc = sk_lo; cc <= sk_hi; ++cc) {
                        if (sk_share_empty(sched.sk_iters, cc, num_clusters))
                            continue;
                        const float4 *slot = partials + static_cast<size_t>(cc * C::CLUSTER + rank) * kSlotVec +
                                             128 * half + prow;
                        float4 x[CW / 4];
#pragma unroll
                        for (int g = 0; g < CW / 4; ++g)  // the slot holds BN columns
                            x[g] = c * CW + 4 * g < BN ? __ldcg(slot + (c * (CW / 4) + g) * kSlotRows)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int g = 0; g < CW / 4; ++g) {
                            v[4 * g] += x[g].x;
                            v[4 * g + 1] += x[g].y;
                            v[4 * g + 2] += x[g].z;
                            v[4 * g + 3] += x[g].w;
                        }
                    }
                } else if (head) {
                    // the contributors' partial sums, gathered into the other buffer
                    const uint32_t paddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                           static_cast<uint32_t>((acc ^ 1) * BN + c * CW);
#pragma unroll
                    for (int h = 0; h < CW / 32; ++h) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(paddr + 32 * h, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[32 * h + i] += __uint_as_float(r[i]);
                    }
                }
                if (use_c && !dc) {
                    const long long tw = stats ? clock64() : 0;
                    bool ok = w.wait(sbar, epi_phase[sel], kRoleEpilogue | kWaitEpiC);
                    if (stats)
                        st_cw += static_cast<unsigned long long>(clock64() - tw);
                    epi_phase[sel] ^= 1u;
                    if (!__all_sync(0xffffffffu, ok))
                        return;
                }
                if (dd) {
                    uint32_t o[32];
                    chunk_math_regs<CW>(v, ec, use_c, creg, o);
                    store_d_row<CW>(o, d_ptr, ldd, m0h + trow, col0, ti.M, n_lim);
                    continue;
                }
                if (dc)
                    epilogue_chunk_math<CW, true>(v, ec, sbuf, trow, true, creg);
                else if (active)
                    epilogue_chunk_math<CW>(v, ec, sbuf, trow, use_c);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (hints)
                        tma_store_2d_hint(mD, sbuf, col0, m0h, stream_once);
                    else
                        tma_store_2d(mD, sbuf, col0, m0h);
                    bulk_commit_group();
                }
                if constexpr (C::EPI_BUFS == 2)
                    sel ^= 1;
            }
        }
        if (has_acc) {
            // all tcgen05.ld of this accumulator have completed (wait::ld above)
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 2)
                    mbar_arrive_cluster(acc_empty_target + 8 * acc);
                else
                    mbar_arrive(bar_acc_empty + 8 * acc);
            }
            if (++acc == C::ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }
    if (stats && ew == 0 && lane == 0) {
        unsigned long long *o = stats + blockIdx.x * kStatSlots;
        o[kStatEpiAccFullWaitCycles] = st_accw;
        o[kStatEpiCWaitCycles] = st_cw;
        const long long t_end = clock64();
        o[kStatEpiLoopCycles] = static_cast<unsigned long long>(t_end - t_start);
        o[kStatEpiPartialWaitCycles] = st_pw;
        o[kStatEpiPartialCycles] = st_pe;
        o[kStatEpiTailCycles] = static_cast<unsigned long long>(t_last_acc ? t_end - t_last_acc : 0);
    }
}

// ---------------------------------------------------------------- kernel

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
__global__ void __launch_bounds__(Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>::THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmD,
                        const __grid_constant__ CUtensorMap tmSFA,
                        const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ KParams p)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    if (C::ALIGN_SLACK == 0 && (raw & 1023u) != 0u) {
        // no room to round the base up: report and leave before any setup
        if (threadIdx.x == 0)
            atomicCAS(p.status, 0u, kRoleSetup | kSetupAlignment);
        return;
    }
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    uint32_t rank = 0;
    if constexpr (C::CLUSTER == 2)
        rank = cluster_ctarank() & 1u;

    const uint32_t bar_full = base + C::BAR_OFF;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_epi = bar_acc_empty + 16;
    const uint32_t bar_drain = bar_epi + 8 * 2 * kEpiWarps;
    const uint32_t bar_inject = bar_drain + 8;
    const uint32_t bar_sf = bar_inject + 8;  // sf_ready[STAGES]
    const uint32_t bar_cp_drain = bar_sf + 8 * STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::MISC_OFF + 4);

    const bool split = C::HAS_LOADB && (p.flags & kFlagSplitLoad) != 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, split ? 2 : 1);  // split loads: both producer warps arm it
            mbar_init(bar_empty + 8 * s, C::MCB ? 2 : 1);  // B multicast: both CTAs' MMAs release it
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, kEpiWarps * CG);
        }
        for (int i = 0; i < 2 * kEpiWarps; ++i)
            mbar_init(bar_epi + 8 * i, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_inject, 1);
        for (int s = 0; s < STAGES; ++s)
            mbar_init(bar_sf + 8 * s, C::SF_COPIERS > 0 ? C::SF_COPIERS : 1);
        mbar_init(bar_cp_drain, C::SF_COPIERS > 0 ? C::SF_COPIERS : 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && !GROUPED) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmD);
        if constexpr (SF) {
            prefetch_tensormap(&tmSFA);
            prefetch_tensormap(&tmSFB);
        }
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (C::CLUSTER == 2)
        cluster_sync_all();  // the peer's barriers exist before anything signals them
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    Waiter w;
    w.timeout_ns = p.timeout_ns;
    w.abort_flag = abort_flag;
    w.status = p.status;
    w.all_cluster_scope = (CG == 2) && (p.flags & kFlagAllClusterWaits);

    const uint32_t stage_base = base;
    ProducerTail tail{0, 0, 0u};
    if (warp == 0) {
        if (lane == 0)
            tail = role_producer<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>(
                p, &tmA, &tmB, &tmSFA, &tmSFB, stage_base, bar_full, bar_empty, bar_inject, rank, w, split ? 1 : 0);
    } else if (warp == C::LOADB_WARP) {
        if (lane == 0 && split)
            tail = role_producer<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>(
                p, &tmA, &tmB, &tmSFA, &tmSFB, stage_base, bar_full, bar_empty, bar_inject, rank, w, 2);
    } else if (warp == 1) {
        // CTA pairs: the even CTA issues the pair's MMAs; every other CTA its own
        if (lane == 0 && (CG == 1 || rank == 0)) {
            role_mma<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>(p, stage_base, bar_full, bar_empty,
                                                  bar_acc_full, bar_acc_empty, bar_inject, bar_sf,
                                                  tmem_base, w);
            // every MMA issued by this thread has completed before TMEM is freed
            mma_commit<CG>(bar_drain);
            w.drain(bar_drain, 0u, 100000000ull);
        }
    } else if (warp >= kSfCopyWarp) {
        // the even CTA copies the scales of both CTAs of a pair (cta_group::2)
        if (lane == 0 && rank == 0) {
            role_sf_copy<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>(p, stage_base, bar_full, bar_sf, tmem_base, w,
                                                                    warp - kSfCopyWarp);
            // arrives once every tcgen05.cp this thread issued has completed
            mma_commit<CG>(bar_cp_drain);
        }
    } else {
        if (p.out_type == 0)
            role_epilogue<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE, 32>(p, &tmC, &tmD, base + C::EPI_OFF,
                                                           bar_acc_full, bar_acc_empty, bar_epi,
                                                           tmem_base, rank, warp, lane, w);
        else
            role_epilogue<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE, 64>(p, &tmC, &tmD, base + C::EPI_OFF,
                                                           bar_acc_full, bar_acc_empty, bar_epi,
                                                           tmem_base, rank, warp, lane, w);
        if (lane == 0)
            bulk_wait_group<0>();  // stores have finished reading shared memory
    }
    __syncwarp();
    __syncthreads();  // every role has returned: the abort flag is final

    if (*abort_flag) {
        // The MMA thread has already waited for its MMAs (bar_drain). Wait for
        // the producer's loads in flight (this CTA's full barriers; for a pair
        // the even CTA's, which count both CTAs' bytes) and for the scale
        // copiers' tcgen05.cp, each with a bound, before TMEM is freed.
        if ((warp == 0 || warp == C::LOADB_WARP) && lane == 0 && (CG == 1 || rank == 0))
            drain_producer_tail<STAGES>(tail, bar_full, w);
        if constexpr (C::SF_COPIERS > 0)
            if (warp == kSfCopyWarp && lane == 0 && rank == 0)
                w.drain(bar_cp_drain, 0u, 100000000ull);
        // loads an odd CTA issued for a stage its even CTA never armed land on
        // no barrier this kernel can observe: a short pause covers them
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 20000ull)
            __nanosleep(1000);
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (C::CLUSTER == 2)
        cluster_sync_all();  // no CTA exits while the other may still write into it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace g300
