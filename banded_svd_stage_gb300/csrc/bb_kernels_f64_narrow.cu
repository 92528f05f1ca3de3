// double pass kernels for reflector lengths up to 17.
#include "bb_launch.cuh"

namespace bb {
BB_INSTANTIATE_W(double, 8) BB_INSTANTIATE_W(double, 9) BB_INSTANTIATE_W(double, 16) BB_INSTANTIATE_W(double, 17)
}  // namespace bb
