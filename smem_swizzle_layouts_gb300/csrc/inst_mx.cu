// Instantiations: block-scaled fp8 (MXFP8), tcgen05 kind::mxf8f6f4.
#include "launch.cuh"

G300_INSTANTIATE(2, 256, 256, 3, false, 1, 128, 1, 0)
G300_INSTANTIATE(2, 128, 256, 4, false, 1, 128, 1, 0)
G300_INSTANTIATE(1, 128, 256, 3, false, 1, 128, 1, 0)
G300_INSTANTIATE(1, 128, 128, 5, false, 1, 128, 1, 0)
