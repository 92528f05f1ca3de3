// float group kernels of the symmetric chase (reflector lengths up to 9, 17
// and 33).
#include "bb_sym_group.cuh"

namespace bb {
BB_SYM_GROUP_INSTANTIATE(float, 9) BB_SYM_GROUP_INSTANTIATE(float, 17) BB_SYM_GROUP_INSTANTIATE(float, 33)
}  // namespace bb
