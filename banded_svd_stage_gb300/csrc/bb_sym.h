// Symmetric variant (bb_sym.cu): launch state and the whole reduction of a
// symmetric lower band to tridiagonal form (zero fill, passes, extraction).
#pragma once

#include <cuda_runtime.h>

namespace bb {

struct SymLaunch {
    int num_sms = 0, max_ctas = 0, stall_sweep = -1;
    unsigned long long wait_budget = 0;
    int* progress = nullptr;  // n per-sweep step counters
    int* status = nullptr;    // device status word
};
int sym_pass_lag(int b, int t);
template <typename T>
cudaError_t run_sym(T* band, long long n, long long ldab, int bw, int tw, T* d, T* e, const SymLaunch& L,
                    cudaStream_t s, long long* launches);

}  // namespace bb
