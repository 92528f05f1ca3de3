// float: pass dispatch, fill-row zeroing and d/e extraction; the pass kernels
// themselves are instantiated in bb_kernels_f32_narrow.cu / _wide.cu.
#include "bb_launch.cuh"

namespace bb {
BB_EXTERN_W(float, 8) BB_EXTERN_W(float, 9) BB_EXTERN_W(float, 16) BB_EXTERN_W(float, 17)
BB_EXTERN_W(float, 32) BB_EXTERN_W(float, 33) BB_EXTERN_W(float, 65)
BB_INSTANTIATE(float)
}  // namespace bb
