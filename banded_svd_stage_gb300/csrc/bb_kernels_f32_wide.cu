// float pass kernels for reflector lengths 32, 33 and up to 65.
#include "bb_launch.cuh"

namespace bb {
BB_INSTANTIATE_W(float, 32) BB_INSTANTIATE_W(float, 33) BB_INSTANTIATE_W(float, 65)
}  // namespace bb
