// Launches of the half-precision storage path (bb_half.cu), called by the
// C-ABI layer for handles of element type BB_F16.
#pragma once

#include <cuda_runtime.h>

#include "bb_internal.h"

namespace bb {

struct HalfLaunch {
    int num_sms = 0;
    int max_ctas = 0;
    int scheduler = 0;        // 0 automatic, 3 group kernel where a group fits, else the flag kernel
    int group_size = 0;       // sweeps per group (0: the largest that fits)
    int* progress = nullptr;  // the handle's per-sweep counters (or per-group watermarks)
    int* status = nullptr;    // the handle's status word
};

// Whether pass P on binary16 storage goes to the group kernel (under the
// scheduler rule of bb_reduce: 0 where at least kAutoGroupMin sweeps fit, 3
// where one fits; reflectors of up to 33 elements), and its plan.  The band
// must also suit bulk copies (group_layout_ok with 2-byte elements).
bool half_choose_group(const PassArgs& P, int scheduler, int group_size, GroupArgs* out);

// One pass (b, t) of P on a binary16 band: the group kernel with plan *GA
// when GA is not null, else the flag kernel (persistent, cooperative
// launch).
cudaError_t run_half_pass(void* band, const PassArgs& P, const HalfLaunch& L, const GroupArgs* GA,
                          cudaStream_t s);
// Zero the fill rows 0..tw-1 and ku+1..ku+tw of every column.
cudaError_t run_half_zero_fill(void* band, long long n, long long ldab, int tw, int ku, int num_sms,
                               cudaStream_t s);
// d_i = A(i, i), e_i = A(i, i+1), binary16.
cudaError_t run_half_extract(const void* band, long long n, long long ldab, int ku, void* d, void* e, int num_sms,
                             cudaStream_t s);

}  // namespace bb
