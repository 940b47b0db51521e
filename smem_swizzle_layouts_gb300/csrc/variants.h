// The compiled kernel variants (tile shape, pipeline depth, CTA pairing).
#pragma once

#include <cuda_runtime.h>

namespace g300 {

struct LaunchArgs;

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, bool MX>
cudaError_t launch_gemm(const LaunchArgs &a);

template <int CG, int BN, int BK, int STAGES, bool GROUPED, int ESIZE, int BMT, bool MX>
cudaError_t resident_ctas(int *ctas);

// X(cta_group, BN, BK, stages, grouped, element bytes, tile rows, block-scaled).
// BN is the MMA N of one tile, BK counts elements; stages fill ~192 KB of
// shared memory next to 32 KB of epilogue staging. Element bytes 2 =
// fp16/bf16, 1 = fp8. Tile rows 128, or 64 for single-CTA M=64 MMAs (TMEM
// Layout F). Block-scaled: fp8 with one E8M0 scale per 32 elements of K for
// each row of A and column of B (tcgen05 kind::mxf8f6f4), the scales riding
// in each stage next to the operand tiles.
#define G300_VARIANTS(X)        \
    X(1, 256, 64, 4, false, 2, 128, false)     \
    X(1, 128, 64, 6, false, 2, 128, false)     \
    X(1, 128, 128, 3, false, 2, 128, false)    \
    X(1, 64, 64, 8, false, 2, 128, false)      \
    X(1, 64, 128, 4, false, 2, 128, false)     \
    X(1, 128, 32, 8, false, 2, 128, false)     \
    X(2, 256, 64, 6, false, 2, 128, false)     \
    X(2, 256, 128, 3, false, 2, 128, false)    \
    X(2, 128, 128, 4, false, 2, 128, false)    \
    X(1, 256, 64, 4, true, 2, 128, false)      \
    X(1, 128, 128, 3, true, 2, 128, false)     \
    X(2, 256, 128, 3, true, 2, 128, false)  \
    X(2, 256, 256, 3, false, 1, 128, false) \
    X(1, 256, 128, 4, false, 1, 128, false) \
    X(1, 128, 256, 3, false, 1, 128, false) \
    X(1, 128, 128, 4, false, 2, 64, false) \
    X(1, 256, 64, 4, false, 2, 64, false) \
    X(2, 128, 256, 4, false, 1, 128, true) \
    X(1, 128, 256, 3, false, 1, 128, true) \
    X(1, 128, 128, 5, false, 1, 128, true)

}  // namespace g300
