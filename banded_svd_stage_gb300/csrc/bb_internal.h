// Internal interface between the C-ABI layer (bb_api.cu) and the
// per-precision kernel translation units (bb_kernels_f32.cu, bb_kernels_f64.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bb_device.cuh"
#include "bb_group.cuh"

namespace bb {

// Largest reflector length the kernels are instantiated for (tw <= 64).
constexpr int kMaxW = 65;

struct LaunchCfg {
    int tpb = 0;         // threads per block (flag and per-cycle kernels)
    int max_ctas = 0;    // cap on the persistent grid (0: co-resident maximum)
    int num_sms = 0;
    int group_size = 0;  // requested sweeps per group (0: largest that fits, <= 16)
    GroupArgs group{};   // filled by plan_group
};

struct LaunchStats {
    int64_t launches = 0;  // kernel launches issued
    int grid = 0;          // persistent grid of the last pass
    int kernel = 0;        // 1 per-cycle, 2 flag kernel, 3 group kernel
    int group = 0;         // sweeps per group (group kernel)
};

// Shared memory of the group kernel: per-sweep reflectors and scalars, then
// the circular column buffer.
inline size_t group_smem_bytes(const GroupArgs& GA, int wmax, size_t elem) {
    return elem * ((size_t)GA.g * wmax + (size_t)((GA.g + 1) & ~1) + (size_t)GA.nslot * GA.lds);
}

// Largest group (<= requested, or <= 16 when requested == 0) whose column
// buffer fits in shared memory; false if not even one sweep fits.
bool plan_group(const PassArgs& P, int wmax, size_t elem, int requested, GroupArgs* out);

// Largest group size the group kernel is compiled for (GroupMaxWarps, minus
// the loader and the storer warps).
inline int group_max_warps(int wmax, size_t elem) { return ((wmax * (int)elem <= 17 * 4) ? 16 : 8) - 2; }

// Ticks the group kernel's loader runs ahead of its storer.
constexpr int kGroupAhead = 3;

// Columns the group starting at sweep 0 holds at most when its loader runs
// `ahead` ticks ahead (the buffer size the group kernel needs; groups further
// down the matrix hold no more).
int group_footprint(const PassArgs& P, int g, int ahead);

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
