// Instantiations: two-half single-CTA tiles (256 rows as two 128-row kind::f16 MMAs sharing B).
#include "launch.cuh"

G300_INSTANTIATE(1, 256, 64, 3, false, 2, 256, 0, 0)
