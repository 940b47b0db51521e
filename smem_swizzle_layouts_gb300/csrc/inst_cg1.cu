// Instantiations: one CTA per 128-row tile (tcgen05 cta_group::1), single problem.
#include "launch.cuh"

G300_INSTANTIATE(1, 256, 64, 4, false, 2, 128, 0, 0)
G300_INSTANTIATE(1, 128, 64, 6, false, 2, 128, 0, 0)
G300_INSTANTIATE(1, 128, 128, 3, false, 2, 128, 0, 0)
G300_INSTANTIATE(1, 64, 64, 8, false, 2, 128, 0, 0)
G300_INSTANTIATE(1, 64, 128, 4, false, 2, 128, 0, 0)
G300_INSTANTIATE(1, 128, 32, 8, false, 2, 128, 0, 0)
