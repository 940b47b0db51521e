// The compiled kernel variants (tile shape, pipeline depth, CTA pairing).
#pragma once

#include <cuda_runtime.h>

namespace g300 {

struct LaunchArgs;

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
cudaError_t launch_gemm(const LaunchArgs &a);

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, int SF, int MODE>
cudaError_t resident_ctas(int *ctas);

// X(cta_group, BN, BK, stages, grouped, element bytes, tile rows, scale kind, mode).
// BN is the MMA N of one tile, BK counts elements; stages fill ~192 KB of
// shared memory next to 32 KB of epilogue staging. Element bytes 2 =
// fp16/bf16, 1 = fp8, 4 = fp32 words read as TF32. Tile rows 128, or 64 for single-CTA M=64 MMAs (TMEM
// Layout F), or 256 for single CTAs that issue two 128-row MMAs per K slice on one B slice. Scale kind 0 = none; 1 = MXFP8 (fp8, one E8M0 scale per 32
// elements of K for each row of A and column of B, kind::mxf8f6f4); 2 = NVFP4
// (packed E2M1, one UE4M3 scale per 16, kind::mxf4nvf4); 3 = MXFP4 (packed
// E2M1, one E8M0 per 32, kind::mxf4). fp4 tiles count BK in bytes; the scale
// atoms ride in each stage next to the operand tiles. Mode 1: tcgen05.mma.ws
// (weight-stationary accumulator layout) on 32- or 64-row single-CTA tiles;
// mode 2: clusters of two cta_group::1 CTAs sharing B by TMA multicast.
#define G300_VARIANTS(X)        \
    X(1, 256, 64, 4, false, 2, 128, 0, 0)     \
    X(1, 128, 64, 6, false, 2, 128, 0, 0)     \
    X(1, 128, 128, 3, false, 2, 128, 0, 0)    \
    X(1, 64, 64, 8, false, 2, 128, 0, 0)      \
    X(1, 64, 128, 4, false, 2, 128, 0, 0)     \
    X(1, 128, 32, 8, false, 2, 128, 0, 0)     \
    X(2, 256, 64, 6, false, 2, 128, 0, 0)     \
    X(2, 256, 128, 3, false, 2, 128, 0, 0)    \
    X(2, 128, 128, 4, false, 2, 128, 0, 0)    \
    X(1, 256, 64, 4, true, 2, 128, 0, 0)      \
    X(1, 128, 128, 3, true, 2, 128, 0, 0)     \
    X(2, 256, 128, 3, true, 2, 128, 0, 0)  \
    X(2, 256, 256, 3, false, 1, 128, 0, 0) \
    X(1, 256, 128, 4, false, 1, 128, 0, 0) \
    X(1, 128, 256, 3, false, 1, 128, 0, 0) \
    X(1, 128, 128, 4, false, 2, 64, 0, 0) \
    X(1, 256, 64, 4, false, 2, 64, 0, 0) \
    X(2, 256, 256, 3, false, 1, 128, 1, 0) \
    X(2, 128, 256, 4, false, 1, 128, 1, 0) \
    X(1, 128, 256, 3, false, 1, 128, 1, 0) \
    X(1, 128, 128, 5, false, 1, 128, 1, 0) \
    X(1, 128, 128, 5, false, 1, 128, 2, 0) \
    X(1, 128, 256, 3, false, 1, 128, 3, 0) \
    X(2, 256, 128, 5, false, 1, 128, 2, 0) \
    X(2, 256, 128, 5, false, 1, 128, 3, 0) \
    X(2, 256, 256, 3, false, 1, 128, 3, 0) \
    X(1, 256, 64, 5, false, 2, 32, 0, 1) \
    X(1, 128, 128, 4, false, 2, 64, 0, 1) \
    X(1, 256, 64, 4, false, 2, 64, 0, 1) \
    X(1, 256, 32, 4, false, 4, 128, 0, 0) \
    X(1, 128, 64, 3, false, 4, 128, 0, 0) \
    X(2, 256, 64, 3, false, 4, 128, 0, 0) \
    X(1, 256, 64, 4, false, 2, 128, 0, 2) \
    X(1, 256, 128, 4, false, 1, 128, 0, 2) \
    X(1, 256, 64, 3, false, 2, 256, 0, 0) \
    X(1, 256, 64, 3, false, 2, 256, 0, 2) \
    X(1, 224, 64, 3, false, 2, 256, 0, 0) \
    X(1, 224, 64, 3, false, 2, 256, 0, 2)

}  // namespace g300
