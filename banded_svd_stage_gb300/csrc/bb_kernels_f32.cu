// float instantiation of the reduction kernels and their launchers.
#include "bb_launch.cuh"

namespace bb {
BB_INSTANTIATE(float)
}  // namespace bb
