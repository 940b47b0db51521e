// Instantiations: two-half single-CTA tiles (256 rows as two 128-row kind::f16 MMAs sharing B),
// alone and in clusters of two that share B by TMA multicast.
#include "launch.cuh"

G300_INSTANTIATE(1, 256, 64, 3, false, 2, 256, 0, 0)
G300_INSTANTIATE(1, 256, 64, 3, false, 2, 256, 0, 2)
G300_INSTANTIATE(1, 224, 64, 3, false, 2, 256, 0, 0)
G300_INSTANTIATE(1, 224, 64, 3, false, 2, 256, 0, 2)
