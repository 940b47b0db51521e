// Instantiations: block-scaled fp4 (NVFP4, kind::mxf4nvf4; MXFP4, kind::mxf4).
#include "launch.cuh"

G300_INSTANTIATE(1, 128, 128, 5, false, 1, 128, 2, 0)
G300_INSTANTIATE(1, 128, 256, 3, false, 1, 128, 3, 0)
G300_INSTANTIATE(2, 256, 128, 5, false, 1, 128, 2, 0)
G300_INSTANTIATE(2, 256, 128, 5, false, 1, 128, 3, 0)
