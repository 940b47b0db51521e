// Instantiations: block-scaled fp4 pair tiles with 256 bytes of K per stage (MXFP4).
#include "launch.cuh"

G300_INSTANTIATE(2, 256, 256, 3, false, 1, 128, 3, 0)
