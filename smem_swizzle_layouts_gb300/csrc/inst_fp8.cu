// Instantiations: fp8 (E4M3/E5M2) operands, tcgen05 kind::f8f6f4.
#include "launch.cuh"

G300_INSTANTIATE(2, 256, 256, 3, false, 1, 128, 0, 0)
G300_INSTANTIATE(1, 256, 128, 4, false, 1, 128, 0, 0)
G300_INSTANTIATE(1, 128, 256, 3, false, 1, 128, 0, 0)
