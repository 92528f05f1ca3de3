// double group kernels of the symmetric chase (reflector lengths up to 9, 17
// and 33).
#include "bb_sym_group.cuh"

namespace bb {
BB_SYM_GROUP_INSTANTIATE(double, 9) BB_SYM_GROUP_INSTANTIATE(double, 17) BB_SYM_GROUP_INSTANTIATE(double, 33)
}  // namespace bb
