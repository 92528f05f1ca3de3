// float pass kernels for reflector lengths up to 17.
#include "bb_launch.cuh"

namespace bb {
BB_INSTANTIATE_W(float, 8) BB_INSTANTIATE_W(float, 9) BB_INSTANTIATE_W(float, 16) BB_INSTANTIATE_W(float, 17)
}  // namespace bb
