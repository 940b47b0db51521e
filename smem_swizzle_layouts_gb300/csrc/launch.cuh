// Host-side launch of one compiled kernel variant (cluster attribute for
// CTA pairs, dynamic shared memory opt-in). Included by the instantiation
// units only.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "gemm_kernel.cuh"

namespace g300 {

struct LaunchArgs {
    CUtensorMap a, b, c, d;
    CUtensorMap sfa, sfb;  // block-scaled operands' scale atoms (else unused)
    KParams p;
    int grid;  // CTAs (a multiple of the cluster size)
    cudaStream_t stream;
};

// Opt a kernel into its dynamic shared memory once per device (the attribute
// is per device; setting it on every launch costs host time on short GEMMs).
// `done` is the caller's per-variant record: one bit per device 0..127.
template <typename Kern>
cudaError_t ensure_smem_attribute(Kern kern, int bytes, std::atomic<uint64_t> (&done)[2])
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 128)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    const uint64_t bit = uint64_t(1) << (dev & 63);
    if (done[dev >> 6].load(std::memory_order_acquire) & bit)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        done[dev >> 6].fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// One record per kernel variant.
template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
std::atomic<uint64_t> smem_attribute_set[2] = {{0}, {0}};

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
cudaError_t launch_gemm(const LaunchArgs &a)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>;
    auto kern = gemm_tcgen05_kernel<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>;
    cudaError_t e = ensure_smem_attribute(kern, C::SMEM_BYTES, smem_attribute_set<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    if (C::CLUSTER == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a.a, a.b, a.c, a.d, a.sfa, a.sfb, a.p);
}

// Largest number of CTAs of this variant that can be resident at once.
template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
cudaError_t resident_ctas(int *ctas)
{
    using C = Cfg<CG, BN, BK, STAGES, ESIZE, BMT, SF, MODE>;
    auto kern = gemm_tcgen05_kernel<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>;
    cudaError_t e = ensure_smem_attribute(kern, C::SMEM_BYTES, smem_attribute_set<CG, BN, BK, STAGES, GROUPED, ESIZE, BMT, SF, MODE>);
    if (e != cudaSuccess)
        return e;
    if (C::CLUSTER == 1) {
        int per_sm = 0, sms = 0, dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::THREADS, C::SMEM_BYTES);
        *ctas = per_sm * sms;
        return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    *ctas = 2 * clusters;
    return e;
}

}  // namespace g300

#define G300_INSTANTIATE(CG, BN, BK, ST, GR, ES, BM, SF, MO)                                             \
    template cudaError_t g300::launch_gemm<CG, BN, BK, ST, GR, ES, BM, SF, MO>(const g300::LaunchArgs &); \
    template cudaError_t g300::resident_ctas<CG, BN, BK, ST, GR, ES, BM, SF, MO>(int *);
