// Tensor-pipe instruction rates of tcgen05.mma on this GPU (a diagnostic, not
// part of the library): one CTA (or CTA pair) per SM issues back-to-back MMAs
// of 128 rows per SM x N = 256 on one TMEM accumulator, operands fixed in
// shared memory (SW128, K-major), and times them with clock64. Block-scaled
// kinds optionally copy their scale atoms into TMEM before every MMA
// (tcgen05.cp, as a 128-byte NVFP4 stage does). Prints one line per case:
//   <kind> cg<1|2> cp<0|1> <cycles per MMA> <flop per SM per cycle>
// Every wait is bounded; a wait that runs out sets the error word and the
// program exits non-zero.
#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_runtime.h>

#include "../descriptors.cuh"
#include "../ptx.cuh"

using namespace g300;

namespace {

constexpr int kIters = 8192;                           // MMAs per CTA (pair)
constexpr int kSmem = 1024 + 16384 + 32768 + 8192;     // align slack, A, B, scale atoms
enum Kind { kBf16 = 0, kE4m3 = 1, kMx8 = 2, kNv4 = 3, kMx4 = 4 };

template <int CG, int KIND, bool CP>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(unsigned long long *cycles, unsigned int *err)
{
    extern __shared__ __align__(1024) uint8_t raw[];
    __shared__ uint32_t tslot;
    __shared__ __align__(8) uint64_t bar;
    const uint32_t base = (smem_u32(raw) + 1023u) & ~1023u;
    const uint32_t sA = base, sB = base + 16384, sSF = base + 16384 + 32768;
    // finite operand bytes in every format; scale codes 1.0 (UE4M3 0x38, E8M0 0x7F)
    for (int i = threadIdx.x * 16; i < 16384 + 32768; i += 128 * 16)
        st_shared_v4(sA + i, 0x22222222u, 0x22222222u, 0x22222222u, 0x22222222u);
    const uint32_t sf = KIND == kNv4 ? 0x38383838u : 0x7F7F7F7Fu;
    for (int i = threadIdx.x * 16; i < 8192; i += 128 * 16)
        st_shared_v4(sSF + i, sf, sf, sf, sf);
    fence_proxy_async_smem();
    const uint32_t barp = smem_u32(&bar);
    const uint32_t rank = CG == 2 ? (cluster_ctarank() & 1u) : 0u;
    if (threadIdx.x == 0) {
        mbar_init(barp, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc<CG>(smem_u32(&tslot), 512);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem = tslot;
    if (threadIdx.x == 0 && rank == 0) {
        const uint64_t ad = make_smem_desc(sA, 16, 1024, 2);
        const uint64_t bd = make_smem_desc(sB, 16, 1024, 2);
        constexpr int M = 128 * CG;
        uint32_t idesc;
        if constexpr (KIND == kBf16)
            idesc = make_idesc(M, 256, 1, 1, 0, 0);
        else if constexpr (KIND == kE4m3)
            idesc = make_idesc(M, 256, 0, 0, 0, 0);
        else if constexpr (KIND == kMx8)
            idesc = make_idesc_mx(M, 256, 0, 0, 0, 0, true);
        else if constexpr (KIND == kNv4)
            idesc = make_idesc_mx(M, 256, 1, 1, 0, 0, false);
        else
            idesc = make_idesc_mx(M, 256, 1, 1, 0, 0, true);
        const uint32_t tsf = tmem + 256;  // A scales, then B scales of columns 0-127 and 128-255
        auto copy_scales = [&]() {
            tmem_cp_32x128b_warpx4<CG>(tsf, make_smem_desc(sSF, 128, 128, 0));
            tmem_cp_32x128b_warpx4<CG>(tsf + 4, make_smem_desc(sSF + 512, 128, 128, 0));
            tmem_cp_32x128b_warpx4<CG>(tsf + 8, make_smem_desc(sSF + 1024, 128, 128, 0));
        };
        if constexpr (KIND >= kMx8)
            copy_scales();
        const long long t0 = clock64();
        for (int i = 0; i < kIters; ++i) {
            const uint32_t j = static_cast<uint32_t>(i & 3);  // the four 32-byte K slices of a 128-byte row
            if constexpr (KIND == kBf16) {
                mma_f16<CG>(tmem, ad + 2 * j, bd + 2 * j, idesc, i != 0);
            } else if constexpr (KIND == kE4m3) {
                mma_f8<CG>(tmem, ad + 2 * j, bd + 2 * j, idesc, i != 0);
            } else {
                if constexpr (CP)
                    copy_scales();
                mma_scaled<CG, KIND - 1>(tmem, ad + 2 * j, bd + 2 * j, idesc, tsf, tsf + 4, i != 0);
            }
        }
        if constexpr (CG == 2)
            mma_commit_pair_multicast(barp);
        else
            mma_commit<1>(barp);
        bool ok = false;
        for (uint32_t it = 0; it < (1u << 26) && !ok; ++it)
            ok = mbar_try_wait(barp, 0);
        const long long t1 = clock64();
        if (!ok)
            atomicExch(err, 1u);
        cycles[blockIdx.x / CG] = ok ? static_cast<unsigned long long>(t1 - t0) : 0ull;
    } else if (threadIdx.x == 0) {
        bool ok = false;  // the odd CTA of a pair waits for the multicast commit
        for (uint32_t it = 0; it < (1u << 26) && !ok; ++it)
            ok = mbar_try_wait_cluster(barp, 0);
        if (!ok)
            atomicExch(err, 2u);
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync_all();
    tc_fence_after_sync();
    if (threadIdx.x < 32)
        tmem_dealloc<CG>(tmem, 512);
}

template <int CG, int KIND, bool CP>
bool run(const char *name, int sms, unsigned long long *d_cycles, unsigned int *d_err)
{
    auto k = mma_rate_kernel<CG, KIND, CP>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
        return false;
    const int grid = sms / 2 * 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    for (int rep = 0; rep < 2; ++rep)
        if (cudaLaunchKernelEx(&cfg, k, d_cycles, d_err) != cudaSuccess)
            return false;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return false;
    const int units = grid / CG;
    std::vector<unsigned long long> h(units);
    unsigned int herr = 0;
    cudaMemcpy(h.data(), d_cycles, units * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaMemcpy(&herr, d_err, sizeof(herr), cudaMemcpyDeviceToHost);
    if (herr)
        return false;
    double mean = 0;
    for (unsigned long long v : h)
        mean += static_cast<double>(v);
    mean /= units;
    const int k_per_mma = KIND == kBf16 ? 16 : KIND <= kMx8 ? 32 : 64;
    const double flop_per_sm = 2.0 * 128 * 256 * k_per_mma;  // a pair MMA covers two SMs
    printf("%s cg%d cp%d %.1f %.0f\n", name, CG, CP ? 1 : 0, mean / kIters, flop_per_sm * kIters / mean);
    return true;
}

}  // namespace

int main()
{
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess)
        return 2;
    unsigned long long *d_cycles = nullptr;
    unsigned int *d_err = nullptr;
    if (cudaMalloc(&d_cycles, sms * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMalloc(&d_err, sizeof(unsigned int)) != cudaSuccess)
        return 2;
    cudaMemset(d_err, 0, sizeof(unsigned int));
    bool ok = run<1, kBf16, false>("bf16", sms, d_cycles, d_err) && run<2, kBf16, false>("bf16", sms, d_cycles, d_err) &&
              run<1, kE4m3, false>("e4m3", sms, d_cycles, d_err) && run<2, kE4m3, false>("e4m3", sms, d_cycles, d_err) &&
              run<2, kMx8, false>("mxfp8", sms, d_cycles, d_err) && run<2, kMx4, false>("mxfp4", sms, d_cycles, d_err) &&
              run<2, kNv4, false>("nvfp4", sms, d_cycles, d_err) && run<2, kNv4, true>("nvfp4", sms, d_cycles, d_err);
    return ok ? 0 : 1;
}
