// Internal interface between the C-ABI layer (bb_api.cu) and the
// per-precision kernel translation units (bb_kernels_f32.cu, bb_kernels_f64.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bb_device.cuh"

namespace bb {

// Largest reflector length the kernels are instantiated for (tw <= 64).
constexpr int kMaxW = 65;

struct LaunchCfg {
    int tpb;       // threads per block
    int max_ctas;  // cap on the persistent grid (0: co-resident maximum)
    int num_sms;
};

struct LaunchStats {
    int64_t launches = 0;  // kernel launches issued
    int grid = 0;          // persistent grid of the last pass
};

// One pass of the reduction on `stream`.  scheduler 0: persistent kernel
// (cooperative launch); 1: one launch per cycle.
template <typename T>
cudaError_t run_pass(T* band, const PassArgs& P, int scheduler, const LaunchCfg& cfg,
                     int* progress, int* status, cudaStream_t stream, LaunchStats* stats);

template <typename T>
cudaError_t run_zero_fill(T* band, long long n, long long ldab, int tw, int ku, cudaStream_t s);

template <typename T>
cudaError_t run_extract(const T* band, long long n, long long ldab, int ku, T* d, T* e,
                        cudaStream_t s);

// Threads per block the launcher uses for a pass when none is requested.
int auto_tpb(int b, int t);

// Set the message bb_last_error() returns on the calling thread.
void set_last_error(const char* msg);

}  // namespace bb
