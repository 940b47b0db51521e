// Instantiations: 64-row tiles (tcgen05.mma M = 64, TMEM Layout F accumulators).
#include "launch.cuh"

G300_INSTANTIATE(1, 128, 128, 4, false, 2, 64, 0, 0)
G300_INSTANTIATE(1, 256, 64, 4, false, 2, 64, 0, 0)
