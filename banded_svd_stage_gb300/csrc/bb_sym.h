// Symmetric variant (bb_sym.cu): launch state and the whole reduction of a
// symmetric lower band to tridiagonal form (zero fill, passes, extraction).
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "bb_internal.h"

namespace bb {

struct SymLaunch {
    int num_sms = 0, max_ctas = 0, stall_sweep = -1;
    // 0: automatic (the group kernel where at least kAutoGroupMin sweeps fit
    // shared memory, else the flag kernel); 3: the group kernel wherever a
    // group fits, else the flag kernel; any other value: the flag kernel
    int scheduler = 0;
    int group_size = 0;  // sweeps per group (0: the largest that fits)
    unsigned long long wait_budget = 0;
    int* progress = nullptr;  // n per-sweep step counters (or per-group watermarks)
    int* status = nullptr;    // device status word
};
// Per pass of the last run: 2 flag kernel, 3 group kernel; group size (0 for
// the flag kernel).
struct SymPassStats {
    std::vector<int> kernel, group;
};
int sym_pass_lag(int b, int t);
// Reflector lengths the symmetric group kernel is compiled for (0: none,
// the flag kernel takes the pass).
inline int sym_group_wmax(int w) { return w <= 9 ? 9 : (w <= 17 ? 17 : (w <= 33 ? 33 : 0)); }
// Whether pass (b, t) of the symmetric chase goes to the group kernel, and
// its plan.
bool sym_choose_group(const PassArgs& P, int scheduler, int group_size, size_t elem, GroupArgs* out);
// Whether any pass of an n x n reduction from bandwidth bw goes to the group
// kernel (whose bulk copies need a 16-byte aligned band and column stride).
bool sym_any_group(long long n, int bw, int tw, const SymLaunch& L, size_t elem);
template <typename T>
cudaError_t run_sym(T* band, long long n, long long ldab, int bw, int tw, T* d, T* e, const SymLaunch& L,
                    cudaStream_t s, long long* launches, SymPassStats* stats);

}  // namespace bb
