// double: pass dispatch, fill-row zeroing and d/e extraction; the pass kernels
// themselves are instantiated in bb_kernels_f64_narrow.cu / _wide.cu.
#include "bb_launch.cuh"

namespace bb {
BB_EXTERN_W(double, 8) BB_EXTERN_W(double, 9) BB_EXTERN_W(double, 16) BB_EXTERN_W(double, 17)
BB_EXTERN_W(double, 32) BB_EXTERN_W(double, 33) BB_EXTERN_W(double, 65)
BB_INSTANTIATE(double)
}  // namespace bb
