// Instantiations: grouped problem lists (device-side problem table and tensor maps).
#include "launch.cuh"

G300_INSTANTIATE(1, 256, 64, 4, true, 2, 128, 0, 0)
G300_INSTANTIATE(1, 128, 128, 3, true, 2, 128, 0, 0)
G300_INSTANTIATE(2, 256, 128, 3, true, 2, 128, 0, 0)
