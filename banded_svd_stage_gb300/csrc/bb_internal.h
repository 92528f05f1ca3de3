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

// Reflector lengths the kernels are compiled for: the exact t + 1 of common
// tile widths (interior steps then run without predicates) and buckets for
// the rest (predicated on the run-time length).
inline int wmax_bucket(int w) {
    for (int c : {8, 9, 16, 17, 32, 33, 65})
        if (w <= c) return c;
    return 0;
}

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
    int kernel = 0;        // 1 per-cycle, 2 flag kernel, 3 group kernel, 4 per-cycle graph
    int group = 0;         // sweeps per group (group kernel)
};

// The chase a group kernel runs: the bidiagonal one (BidiagChase, two
// half-steps per step) or the symmetric one (SymChase in bb_sym_group.cuh,
// one two-sided step; lower band storage).
enum class ChaseKind { kBidiag = 0, kSym = 1 };
// Reflector-sized vectors of shared scratch per sweep (Chase::kVecs).
inline int chase_vecs(ChaseKind kind) { return kind == ChaseKind::kSym ? 2 : 1; }

// Shared memory of the group kernel: per-sweep scratch and scalars (elem:
// the arithmetic type's size), then the circular column buffer (selem: the
// storage type's size; 0 = elem).
inline size_t group_smem_bytes(const GroupArgs& GA, int wmax, size_t elem, int nvec = 1, size_t selem = 0) {
    return group_cols_offset(GA.g, wmax, elem, nvec) + (selem ? selem : elem) * (size_t)GA.nslot * GA.lds;
}

// Cooperative launch of the group kernel (arithmetic T, storage ST, chase
// Chase) for one pass: as many CTAs as can be co-resident, at most max_ctas
// (when > 0) and at most one per group; the groups' watermarks wm zeroed
// first, on the same stream.  *grid_out (if given) receives the grid.
template <typename T, int WMAX, class Chase, typename ST>
cudaError_t launch_group_pass(ST* band, const PassArgs& P, const GroupArgs& GA, int num_sms, int max_ctas, int* wm,
                              int* status, cudaStream_t s, int* grid_out = nullptr) {
    auto kern = pass_group_kernel<T, WMAX, Chase, ST>;
    const size_t smem = group_smem_bytes(GA, WMAX, sizeof(T), Chase::kVecs, sizeof(ST));
    // always raise the dynamic limit: static shared memory counts against 48 KB too
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (GA.g + 3), smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)per_sm * num_sms;
    if (grid > GA.ngroups) grid = GA.ngroups;
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    err = cudaMemsetAsync(wm, 0, sizeof(int) * (size_t)GA.ngroups, s);
    if (err != cudaSuccess) return err;
    ST* band_arg = band;
    PassArgs p_arg = P;
    GroupArgs g_arg = GA;
    int* wm_arg = wm;
    int* stat_arg = status;
    void* args[] = {&band_arg, &p_arg, &g_arg, &wm_arg, &stat_arg};
    if (grid_out) *grid_out = (int)grid;
    return cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(32 * (GA.g + 3)), args, smem,
                                       s);
}

// Largest group (<= requested, or the most the kernel is compiled for when
// requested == 0) whose column buffer fits in shared memory; false if not
// even one sweep fits.  elem: the arithmetic type's size; selem: the
// storage type's size (0 = elem; 2 for binary16 storage).  The kernel then
// needs the band and ldab * selem 16-byte aligned (group_layout_ok).
bool plan_group(const PassArgs& P, int wmax, size_t elem, int requested, GroupArgs* out,
                ChaseKind kind = ChaseKind::kBidiag, size_t selem = 0);

// Whether the group kernel's bulk copies can address this band storage.
inline bool group_layout_ok(const void* band, long long ldab, size_t elem) {
    return ((uintptr_t)band & 15) == 0 && ((size_t)ldab * elem) % 16 == 0;
}

// Orders the group kernel handles (its step geometry is 32-bit).
constexpr long long kGroupMaxN = 1LL << 30;

// Largest group size the group kernel is compiled for (GroupMaxWarps, minus
// the loader, storer and publisher warps).
inline int group_max_warps(int wmax, size_t elem) {
    const int b = wmax * (int)elem;
    return (b <= 17 * 4 ? 16 : 8) - 3;
}

// Fewest sweeps per group for which the automatic scheduler prefers the
// group kernel: with fewer, the per-group hand-over (a few ticks) is shared
// by too few sweeps and the flag kernel is faster (measured on the
// workloads' passes: the group kernel wins from 5 sweeps per group on).
constexpr int kAutoGroupMin = 5;

// Whether a pass goes to the group kernel, and its group plan: scheduler 3
// always when a group fits, scheduler 0 (automatic) when at least
// kAutoGroupMin sweeps fit (given a storage that suits bulk copies).
inline bool choose_group(const PassArgs& P, int scheduler, int group_size, size_t elem, GroupArgs* out) {
    if (scheduler != 0 && scheduler != 3) return false;
    if (P.nsweeps <= 0 || P.n >= kGroupMaxN) return false;
    GroupArgs ga;
    if (!plan_group(P, wmax_bucket(P.t + 1), elem, group_size, &ga)) return false;
    if (scheduler == 0 && ga.g < kAutoGroupMin) return false;
    if (out) *out = ga;
    return true;
}

// Ticks the group kernel's loader runs ahead of its storer.
constexpr int kGroupAhead = 3;

// Columns the group starting at sweep 0 holds at most when its loader runs
// `ahead` ticks ahead (the buffer size the group kernel needs; groups further
// down the matrix hold no more).
int group_footprint(const PassArgs& P, int g, int ahead, ChaseKind kind = ChaseKind::kBidiag);

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
// Half-step lag of the persistent schedulers and cycle lag of the per-cycle
// scheduler for pass (b, t) (bb_plan.cu).
int pass_lag_half(int b, int t);
int pass_lag_cycle(int b, int t);

// Set the message bb_last_error() returns on the calling thread.
void set_last_error(const char* msg);

}  // namespace bb
