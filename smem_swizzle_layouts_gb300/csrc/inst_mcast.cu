// Instantiations: cta_group::1 128 x 256 tiles in clusters of two sharing B by TMA multicast (bf16, fp8).
#include "launch.cuh"

G300_INSTANTIATE(1, 256, 64, 4, false, 2, 128, 0, 2)
G300_INSTANTIATE(1, 256, 128, 4, false, 1, 128, 0, 2)
