// Launches of the half-precision storage path (bb_half.cu), called by the
// C-ABI layer for handles of element type BB_F16.
#pragma once

#include <cuda_runtime.h>

#include "bb_device.cuh"

namespace bb {

struct HalfLaunch {
    int num_sms = 0;
    int max_ctas = 0;
    int* progress = nullptr;  // the handle's per-sweep counters
    int* status = nullptr;    // the handle's status word
};

// One pass (b, t) of P on a binary16 band (persistent kernel, cooperative launch).
cudaError_t run_half_pass(void* band, const PassArgs& P, const HalfLaunch& L, cudaStream_t s);
// Zero the fill rows 0..tw-1 and ku+1..ku+tw of every column.
cudaError_t run_half_zero_fill(void* band, long long n, long long ldab, int tw, int ku, int num_sms,
                               cudaStream_t s);
// d_i = A(i, i), e_i = A(i, i+1), binary16.
cudaError_t run_half_extract(const void* band, long long n, long long ldab, int ku, void* d, void* e, int num_sms,
                             cudaStream_t s);

}  // namespace bb
