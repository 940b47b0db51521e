// Instantiations: TF32 operands (fp32 words, tcgen05 kind::tf32, K = 8 per MMA).
#include "launch.cuh"

G300_INSTANTIATE(1, 256, 32, 4, false, 4, 128, 0, 0)
G300_INSTANTIATE(1, 128, 64, 3, false, 4, 128, 0, 0)
G300_INSTANTIATE(2, 256, 64, 3, false, 4, 128, 0, 0)
