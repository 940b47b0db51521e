// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   D = alpha * A * B + beta * C,  fp16/bf16 in, fp32 accumulate in TMEM.
//
// One CTA (cta_group::1) or one CTA pair (cta_group::2, cluster of 2) per
// SM / SM pair walks a static round-robin list of output tiles. Six warps:
//   warp 0     TMA producer: one thread fills an S-stage shared-memory ring
//              (full/empty mbarriers, "Tensor Cores, layouts, and swizzling",
//              TMA section and 6.6.1: expect_tx bytes, parity (k/S)&1);
//   warp 1     TMEM allocator and MMA issuer: one thread issues
//              tcgen05.mma for every K=16 slice and commits completion to
//              mbarriers ("06 Blackwell Tensor Core - tcgen05 MMA", "How
//              tcgen05.mma Executes"); the accumulator is double-buffered
//              in TMEM (2 x BN fp32 columns) so the epilogue of tile i
//              overlaps the main loop of tile i+1;
//   warps 2-5  epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (the lane
//              quarter rule of "Tensor Cores, layouts, and swizzling",
//              tcgen05 section) with tcgen05.ld, applies alpha/beta against
//              C (TMA-loaded), converts, stages 32-row chunks in a
//              swizzled shared-memory buffer and writes them with TMA stores.
//
// CTA pairs: the even CTA holds accumulator rows 0-127 and the odd CTA rows
// 128-255 ("How cta_group Sets the Operation Scope", cta_group::2, M=256).
// Each CTA TMA-loads its own 128 rows of A and its own half of the tile's N
// columns of B into its own shared memory (no multicast); completion bytes
// of both land on the even CTA's full barrier, whose one thread issues the
// M=256 MMAs and commits their completion to the even CTA's barriers. The
// even CTA forwards each release to the odd CTA with a remote
// mbarrier.arrive: its producer, once a stage is free again, and its first
// epilogue warp, once an accumulator is complete. The odd CTA's epilogue
// warps release accumulators by remote arrives on the even CTA's barrier.
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

constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kEpiBufBytes = 32 * 128;  // one 32-row x 128 B staging chunk

// Roles in the status word (bits 0-7) and waits (bits 8-15).
enum : uint32_t {
    kRoleProducer = 1,
    kRoleMma = 2,
    kRoleEpilogue = 3,
    kWaitEmpty = 1 << 8,
    kWaitFull = 2 << 8,
    kWaitAccEmpty = 3 << 8,
    kWaitAccFull = 4 << 8,
    kWaitEpiC = 5 << 8,
    kWaitInjected = 6 << 8,
    kWaitDrain = 7 << 8,
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
    int a_swz, b_swz;      // swizzle bits: 0 none, 1 SW32, 2 SW64, 3 SW128
    int a_fmt, b_fmt;      // MMA operand formats (kind::f16: 0 fp16, 1 bf16; kind::f8f6f4: 0 E4M3, 1 E5M2)
    int out_type;          // 0 f32, 1 bf16, 2 f16
    int epi_swizzle;       // 1: staging chunks in SW128 layout; 0: plain rows
    int group_m;           // raster group height (tiles)
    unsigned long long timeout_ns;
    int inject_timeout;
    unsigned int *status;
    const GroupedProblemDev *problems;  // grouped launches only
    const CUtensorMap *maps;            // [num_problems][4]: A, B, C, D
    int num_problems;
    int flags;                  // kFlag* tuning switches
    unsigned long long *stats;  // optional per-CTA wait counters (kStat* slots), or null
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
    kStatSlots = 16,
};

enum : int {
    kFlagPairForward = 1,      // CTA pairs: forward releases with remote arrives (ablation)
    kFlagAllClusterWaits = 2,  // CTA pairs: cluster-scope acquire on every wait (ablation)
    kFlagRotateK = 4,          // start each tile's K loop at a per-cluster offset
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

// ESIZE: bytes per operand element, 2 (fp16/bf16, tcgen05 kind::f16) or
// 1 (fp8, kind::f8f6f4). BK counts elements of K per stage. BMT: accumulator
// rows per CTA, 128 (row m in TMEM lane m) or 64 (cta_group::1 only, Layout F:
// rows 16g..16g+15 in lanes 32g+a..32g+a+15; the two accumulators of the
// double buffer take lane alignments a = 0 and 16 and share their columns).
template <int CG, int BN, int BK, int STAGES, int ESIZE = 2, int BMT = 128>
struct Cfg {
    static constexpr int BM = BMT;             // accumulator rows per CTA
    static constexpr int BN_LOCAL = BN / CG;   // B columns loaded by each CTA
    static constexpr int A_BYTES = BM * BK * ESIZE;
    static constexpr int B_BYTES = BN_LOCAL * BK * ESIZE;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TX_BYTES = STAGE_BYTES * CG;  // bytes landing on one full barrier
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr int EPI_BYTES = kEpiWarps * 2 * kEpiBufBytes;
    static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
    // full[S], empty[S], acc_full[2], acc_empty[2], epi[4][2], drain, inject
    static constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 2 * kEpiWarps + 2;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base
    static constexpr int TMEM_COLS = BMT == 64 ? BN : 2 * BN;
    static constexpr int UMMA_M = BM * CG;
    static constexpr int EPI_ROWS = BM / 4;    // output rows per epilogue warp
    static_assert(BMT == 128 || (BMT == 64 && CG == 1), "64-row tiles are single-CTA");
    static constexpr int KSLICES = BK * ESIZE / 32;  // MMAs per stage (32 bytes of K each)
    static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-aligned");
    static_assert(A_BYTES % 1024 == 0, "B tile must start 1024-aligned");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation: power of two, 32..512 columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static_assert(CG == 1 || BN % 32 == 0, "pair tiles split N in halves of whole atoms");
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
    return s;
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
    const int W = 16 << swz_bits;
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

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT>
__device__ void role_producer(const KParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB,
                              uint32_t smem, uint32_t bar_full, uint32_t bar_empty,
                              uint32_t rank, const Waiter &w)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT>;
    const Sched sched = make_sched(p);
    const int flags = p.flags;
    unsigned long long *const stats = p.stats;
    const CUtensorMap *const maps = p.maps;
    const OperandBoxes boxA = operand_boxes(p.a_mn, p.a_swz, C::BM, BK, ESIZE);
    const OperandBoxes boxB = operand_boxes(p.b_mn, p.b_swz, C::BN_LOCAL, BK, ESIZE);
    const int nbox = boxA.nbox > boxB.nbox ? boxA.nbox : boxB.nbox;
    const bool forward = CG == 2 && rank == 0 && (flags & kFlagPairForward);

    const uint32_t full_target = (CG == 2) ? mapa_shared(bar_full, 0) : bar_full;
    const uint32_t peer_empty = (CG == 2 && rank == 0) ? mapa_shared(bar_empty, 1) : 0u;
    const int cluster_id = blockIdx.x / CG, num_clusters = gridDim.x / CG;
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool ok = true;
    int last_prob = -1;
    unsigned long long st_wait = 0, st_blocked = 0;
    for (int t = cluster_id; t < sched.num_tiles && ok; t += num_clusters) {
        TileInfo ti;
        decode_tile<GROUPED>(sched, t, ti);
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
        const int m0 = ti.m_blk * C::UMMA_M + C::BM * static_cast<int>(rank);
        const int n0 = ti.n_blk * BN + C::BN_LOCAL * static_cast<int>(rank);
        for (int kb = 0; kb < num_kb; ++kb) {
            if (stats) {
                const long long t0 = clock64();
                const bool ready = mbar_try_wait(bar_empty + 8 * stage, phase ^ 1u);
                ok = ready || w.wait(bar_empty + 8 * stage, phase ^ 1u, kRoleProducer | kWaitEmpty, rank != 0);
                st_wait += static_cast<unsigned long long>(clock64() - t0);
                st_blocked += ready ? 0 : 1;
            } else {
                ok = w.wait(bar_empty + 8 * stage, phase ^ 1u, kRoleProducer | kWaitEmpty, rank != 0);
            }
            if (!ok)
                break;
            // pass a real release (not the first trip round the ring) on to the odd CTA
            if (forward && issued >= STAGES)
                mbar_arrive_cluster(peer_empty + 8 * stage);
            if (rank == 0)
                mbar_arrive_expect_tx(bar_full + 8 * stage, C::TX_BYTES);
            const uint32_t sA = smem + stage * C::STAGE_BYTES;
            const uint32_t sB = sA + C::A_BYTES;
            const uint32_t fb = full_target + 8 * stage;
            const int k0 = kblock_at(kb, num_kb, flags, cluster_id) * BK;
            // A and B boxes alternate, so both operands of the stage are in flight together
            for (int b = 0; b < nbox; ++b) {
                if (b < boxA.nbox)
                    issue_box<CG>(mA, sA, fb, boxA, b, m0, k0);
                if (b < boxB.nbox)
                    issue_box<CG>(mB, sB, fb, boxB, b, n0, k0);
            }
            ++issued;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (stats) {
        stats[blockIdx.x * kStatSlots + kStatProducerWaitCycles] = st_wait;
        stats[blockIdx.x * kStatSlots + kStatProducerBlocked] = st_blocked;
    }
    if (!ok && CG == 1) {
        // Let the loads still in flight land before the CTA can exit.
        const int n = issued < STAGES ? issued : STAGES;
        for (int i = 1; i <= n; ++i) {
            int s = stage - i, ph = static_cast<int>(phase);
            if (s < 0) {
                s += STAGES;
                ph ^= 1;
            }
            w.drain(bar_full + 8 * s, static_cast<uint32_t>(ph), 20000000ull);
        }
    }
}

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT>
__device__ void role_mma(const KParams &p, uint32_t smem, uint32_t bar_full, uint32_t bar_empty,
                         uint32_t bar_acc_full, uint32_t bar_acc_empty, uint32_t bar_inject,
                         uint32_t tmem_base, const Waiter &w)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT>;
    if (p.inject_timeout) {
        // Test hook: wait on a barrier nothing arrives at; the bound runs out.
        w.wait(bar_inject, 0u, kRoleMma | kWaitInjected);
        return;
    }
    const Sched sched = make_sched(p);
    unsigned long long *const stats = p.stats;
    const bool multicast = CG == 2 && !(p.flags & kFlagPairForward);
    const uint32_t idesc = make_idesc(C::UMMA_M, BN, p.a_fmt, p.b_fmt, p.a_mn, p.b_mn);
    const OperandPacking pa = operand_packing(p.a_mn, p.a_swz, C::BM, BK);
    const OperandPacking pb = operand_packing(p.b_mn, p.b_swz, C::BN_LOCAL, BK);
    const uint64_t a_desc0 = make_smem_desc(smem, pa.lbo, pa.sbo, pa.swz);
    const uint64_t b_desc0 = make_smem_desc(smem + C::A_BYTES, pb.lbo, pb.sbo, pb.swz);
    uint32_t a_off[C::KSLICES], b_off[C::KSLICES];
#pragma unroll
    for (int j = 0; j < C::KSLICES; ++j) {
        a_off[j] = slice_byte_offset(p.a_mn, p.a_swz, C::BM, j, ESIZE) >> 4;
        b_off[j] = slice_byte_offset(p.b_mn, p.b_swz, C::BN_LOCAL, j, ESIZE) >> 4;
    }
    const int cluster_id = blockIdx.x / CG, num_clusters = gridDim.x / CG;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    unsigned long long st_full = 0, st_acc = 0, st_blocked = 0, st_tiles = 0;
    const long long t_start = clock64();
    for (int t = cluster_id; t < sched.num_tiles; t += num_clusters) {
        TileInfo ti;
        decode_tile<GROUPED>(sched, t, ti);
        const int num_kb = ceil_div_i(ti.K, BK);
        if (num_kb == 0)
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
        const uint32_t d_tmem = C::BM == 64 ? tmem_base + (static_cast<uint32_t>(16 * acc) << 16)
                                            : tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
            if (stats) {
                const long long t0 = clock64();
                const bool ready = mbar_try_wait(bar_full + 8 * stage, phase);
                if (!ready && !w.wait(bar_full + 8 * stage, phase, kRoleMma | kWaitFull))
                    return;
                st_full += static_cast<unsigned long long>(clock64() - t0);
                st_blocked += ready ? 0 : 1;
            } else if (!w.wait(bar_full + 8 * stage, phase, kRoleMma | kWaitFull)) {
                return;
            }
            tc_fence_after_sync();
            const uint64_t sdelta = static_cast<uint64_t>((stage * C::STAGE_BYTES) >> 4);
#pragma unroll
            for (int j = 0; j < C::KSLICES; ++j) {
                if constexpr (ESIZE == 2)
                    mma_f16<CG>(d_tmem, a_desc0 + sdelta + a_off[j], b_desc0 + sdelta + b_off[j], idesc,
                                (kb | j) != 0);
                else
                    mma_f8<CG>(d_tmem, a_desc0 + sdelta + a_off[j], b_desc0 + sdelta + b_off[j], idesc,
                               (kb | j) != 0);
            }
            if (multicast)
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
        acc ^= 1;
        if (acc == 0)
            acc_phase ^= 1u;
    }
    if (stats) {
        unsigned long long *o = stats + blockIdx.x * kStatSlots;
        o[kStatMmaFullWaitCycles] = st_full;
        o[kStatMmaAccEmptyWaitCycles] = st_acc;
        o[kStatMmaLoopCycles] = static_cast<unsigned long long>(clock64() - t_start);
        o[kStatMmaFullBlocked] = st_blocked;
        o[kStatTiles] = st_tiles;
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

// One 32-row x 128-byte chunk: fp32 output covers 32 columns, 16-bit output 64.
// `acc` holds this thread's row (lane) of the chunk in fp32.
template <int CW>
__device__ __forceinline__ void epilogue_chunk_math(float (&acc)[CW], const EpiConst &e,
                                                    uint32_t sbuf, int r, bool use_c)
{
    const uint32_t row = sbuf + static_cast<uint32_t>(r) * 128u;
    const uint32_t key = static_cast<uint32_t>(r) & e.key_mask;
    constexpr int PER16 = (CW == 32) ? 4 : 8;  // elements per 16-byte unit
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t addr = row + ((static_cast<uint32_t>(u) ^ key) << 4);
        float *v = acc + u * PER16;
#pragma unroll
        for (int i = 0; i < PER16; ++i)
            v[i] *= e.alpha;
        if (use_c) {
            uint32_t c[4];
            ld_shared_v4(addr, c[0], c[1], c[2], c[3]);
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
        uint32_t o[4];
        if constexpr (CW == 32) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = __float_as_uint(v[i]);
        } else {
            pack_out(v, e.out_type, o);
        }
        st_shared_v4(addr, o[0], o[1], o[2], o[3]);
    }
}

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int CW>
__device__ void role_epilogue(const KParams &p, const CUtensorMap *tmC, const CUtensorMap *tmD,
                              uint32_t epi_base, uint32_t bar_acc_full, uint32_t bar_acc_empty,
                              uint32_t bar_epi, uint32_t tmem_base, uint32_t rank, int warp,
                              int lane, const Waiter &w)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT>;
    const Sched sched = make_sched(p);
    unsigned long long *const stats = p.stats;
    const CUtensorMap *const maps = p.maps;
    EpiConst ec;
    ec.alpha = p.alpha;
    ec.beta = p.beta;
    ec.out_type = p.out_type;
    ec.key_mask = p.epi_swizzle ? 7u : 0u;
    const bool forward = CG == 2 && rank == 0 && (p.flags & kFlagPairForward);
    const int q = warp & 3;   // TMEM lane quarter 32q..32q+31 = output rows EPI_ROWS*q..
    constexpr int R = C::EPI_ROWS;
    const int ew = warp - 2;  // staging slot
    const uint32_t buf0 = epi_base + static_cast<uint32_t>(ew * 2 * kEpiBufBytes);
    const uint32_t ebar0 = bar_epi + static_cast<uint32_t>(16 * ew);
    const bool use_c = ec.beta != 0.0f;
    const uint32_t acc_empty_target = (CG == 2) ? mapa_shared(bar_acc_empty, 0) : bar_acc_empty;
    const uint32_t peer_acc_full = (CG == 2 && rank == 0) ? mapa_shared(bar_acc_full, 1) : 0u;
    const int cluster_id = blockIdx.x / CG, num_clusters = gridDim.x / CG;
    uint32_t epi_phase[2] = {0u, 0u};
    int sel = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    unsigned long long st_accw = 0, st_cw = 0;
    const long long t_start = clock64();
    for (int t = cluster_id; t < sched.num_tiles; t += num_clusters) {
        TileInfo ti;
        decode_tile<GROUPED>(sched, t, ti);
        const CUtensorMap *mC = tmC, *mD = tmD;
        if constexpr (GROUPED) {
            mC = maps + 4 * ti.prob + 2;
            mD = mC + 1;
            fence_tensormap_acquire(mC);
            fence_tensormap_acquire(mD);
        }
        const bool has_acc = ti.K > 0;
        const int m0 = ti.m_blk * C::UMMA_M + C::BM * static_cast<int>(rank) + R * q;
        // 128-row tiles: thread t holds row t. 64-row tiles (Layout F): the
        // accumulator with lane alignment 16*acc sits in threads 16*acc..+15.
        const bool active = C::BM == 128 || (lane >> 4) == acc;
        const int trow = C::BM == 128 ? lane : (lane & 15);
        if (has_acc) {
            const long long tw = stats ? clock64() : 0;
            bool ok = w.wait(bar_acc_full + 8 * acc, acc_phase, kRoleEpilogue | kWaitAccFull, rank != 0);
            if (stats)
                st_accw += static_cast<unsigned long long>(clock64() - tw);
            if (!__all_sync(0xffffffffu, ok))
                return;
            if (forward && ew == 0 && lane == 0)
                mbar_arrive_cluster(peer_acc_full + 8 * acc);  // the odd CTA's half is complete too
            tc_fence_after_sync();
        }
        for (int c = 0; c < BN / CW; ++c) {
            const int col0 = ti.n_blk * BN + c * CW;
            if (col0 >= ti.N)
                break;
            const uint32_t sbuf = buf0 + static_cast<uint32_t>(sel * kEpiBufBytes);
            const uint32_t sbar = ebar0 + static_cast<uint32_t>(8 * sel);
            // the store issued from this buffer two chunks ago must have read it
            if (lane == 0)
                bulk_wait_group_read<1>();
            __syncwarp();
            if (use_c && lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(sbar, R * 128);
                tma_load_2d(sbuf, mC, sbar, col0, m0);
            }
            __syncwarp();  // tcgen05.ld is .sync.aligned: the warp must be converged
            float v[CW];
            if (has_acc) {
                const uint32_t col = static_cast<uint32_t>((C::BM == 128 ? acc * BN : 0) + c * CW);
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
            if (use_c) {
                const long long tw = stats ? clock64() : 0;
                bool ok = w.wait(sbar, epi_phase[sel], kRoleEpilogue | kWaitEpiC);
                if (stats)
                    st_cw += static_cast<unsigned long long>(clock64() - tw);
                epi_phase[sel] ^= 1u;
                if (!__all_sync(0xffffffffu, ok))
                    return;
            }
            if (active)
                epilogue_chunk_math<CW>(v, ec, sbuf, trow, use_c);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(mD, sbuf, col0, m0);
                bulk_commit_group();
            }
            sel ^= 1;
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
            acc ^= 1;
            if (acc == 0)
                acc_phase ^= 1u;
        }
    }
    if (stats && ew == 0 && lane == 0) {
        unsigned long long *o = stats + blockIdx.x * kStatSlots;
        o[kStatEpiAccFullWaitCycles] = st_accw;
        o[kStatEpiCWaitCycles] = st_cw;
        o[kStatEpiLoopCycles] = static_cast<unsigned long long>(clock64() - t_start);
    }
}

// ---------------------------------------------------------------- kernel

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmD, const __grid_constant__ KParams p)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    uint32_t rank = 0;
    if constexpr (CG == 2)
        rank = cluster_ctarank() & 1u;

    const uint32_t bar_full = base + C::BAR_OFF;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_epi = bar_acc_empty + 16;
    const uint32_t bar_drain = bar_epi + 8 * 2 * kEpiWarps;
    const uint32_t bar_inject = bar_drain + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::MISC_OFF + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, kEpiWarps * CG);
        }
        for (int i = 0; i < 2 * kEpiWarps; ++i)
            mbar_init(bar_epi + 8 * i, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_inject, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && !GROUPED) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmD);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync_all();  // the peer's barriers exist before anything signals them
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    Waiter w;
    w.timeout_ns = p.timeout_ns;
    w.abort_flag = abort_flag;
    w.status = p.status;
    w.all_cluster_scope = (CG == 2) && (p.flags & kFlagAllClusterWaits);

    const uint32_t stage_base = base;
    if (warp == 0) {
        if (lane == 0)
            role_producer<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT>(p, &tmA, &tmB, stage_base, bar_full,
                                                              bar_empty, rank, w);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            role_mma<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT>(p, stage_base, bar_full, bar_empty,
                                                  bar_acc_full, bar_acc_empty, bar_inject,
                                                  tmem_base, w);
            // every MMA issued by this thread has completed before TMEM is freed
            mma_commit<CG>(bar_drain);
            w.drain(bar_drain, 0u, 100000000ull);
        }
    } else {
        if (p.out_type == 0)
            role_epilogue<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, 32>(p, &tmC, &tmD, base + C::EPI_OFF,
                                                           bar_acc_full, bar_acc_empty, bar_epi,
                                                           tmem_base, rank, warp, lane, w);
        else
            role_epilogue<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, 64>(p, &tmC, &tmD, base + C::EPI_OFF,
                                                           bar_acc_full, bar_acc_empty, bar_epi,
                                                           tmem_base, rank, warp, lane, w);
        if (lane == 0)
            bulk_wait_group<0>();  // stores have finished reading shared memory
    }
    __syncwarp();

    if (*abort_flag) {
        // give copies and MMAs still in flight time to land before teardown
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 20000ull)
            __nanosleep(1000);
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace g300
