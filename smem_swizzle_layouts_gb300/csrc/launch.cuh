// Host-side launch of one compiled kernel variant (cluster attribute for
// CTA pairs, dynamic shared memory opt-in). Included by the instantiation
// units only.
#pragma once

#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace g300 {

struct LaunchArgs {
    CUtensorMap a, b, c, d;
    KParams p;
    int grid;  // CTAs (a multiple of the cluster size)
    cudaStream_t stream;
};

template <int CG, int BN, int BK, int STAGES, bool GROUPED>
cudaError_t launch_gemm(const LaunchArgs &a)
{
    using C = Cfg<CG, BN, BK, STAGES>;
    auto kern = gemm_tcgen05_kernel<CG, BN, BK, STAGES, GROUPED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    if (CG == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a.a, a.b, a.c, a.d, a.p);
}

// Largest number of CTAs of this variant that can be resident at once.
template <int CG, int BN, int BK, int STAGES, bool GROUPED>
cudaError_t resident_ctas(int *ctas)
{
    using C = Cfg<CG, BN, BK, STAGES>;
    auto kern = gemm_tcgen05_kernel<CG, BN, BK, STAGES, GROUPED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    if (CG == 1) {
        int per_sm = 0, sms = 0, dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, C::SMEM_BYTES);
        *ctas = per_sm * sms;
        return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
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

#define G300_INSTANTIATE(CG, BN, BK, ST, GR)                                             \
    template cudaError_t g300::launch_gemm<CG, BN, BK, ST, GR>(const g300::LaunchArgs &); \
    template cudaError_t g300::resident_ctas<CG, BN, BK, ST, GR>(int *);
