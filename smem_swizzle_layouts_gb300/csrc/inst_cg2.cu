// Instantiations: CTA pairs on 256-row tiles (tcgen05 cta_group::2), single problem.
#include "launch.cuh"

G300_INSTANTIATE(2, 256, 64, 6, false, 2, 128, 0, 0)
G300_INSTANTIATE(2, 256, 128, 3, false, 2, 128, 0, 0)
G300_INSTANTIATE(2, 128, 128, 4, false, 2, 128, 0, 0)
