// Instantiations: weight-stationary tcgen05.mma.ws tiles (M = 32 and 64 rows, kind::f16).
#include "launch.cuh"

G300_INSTANTIATE(1, 256, 64, 5, false, 2, 32, 0, 1)
G300_INSTANTIATE(1, 128, 128, 4, false, 2, 64, 0, 1)
G300_INSTANTIATE(1, 256, 64, 4, false, 2, 64, 0, 1)
