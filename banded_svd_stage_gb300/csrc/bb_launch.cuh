// Launch logic shared by the per-precision translation units.
#pragma once

#include <algorithm>

#include "bb_group.cuh"
#include "bb_internal.h"

namespace bb {

template <typename T, int WMAX>
size_t smem_bytes(const PassArgs& P) {
    const int wp = WMAX | 1;
    const size_t ncol = (size_t)P.b + P.t + 1;
    return sizeof(T) * ((size_t)WMAX + 2 + (2 * ncol - 1) * wp);
}

template <typename T, int WMAX>
cudaError_t run_pass_w(T* band, const PassArgs& P, int scheduler, const LaunchCfg& cfg,
                       int* progress, int* status, cudaStream_t stream, LaunchStats* stats) {
    const size_t smem = smem_bytes<T, WMAX>(P);
    const int tpb = std::min(cfg.tpb, MaxThreads<T, WMAX>::value);
    cudaError_t err;
    if (scheduler == 3) {
        if (P.nsweeps <= 0) return cudaSuccess;
        const GroupArgs& GA = cfg.group;
        int grid = 0;
        err = launch_group_pass<T, WMAX, BidiagChase, T>(band, P, GA, cfg.num_sms, cfg.max_ctas, progress, status,
                                                         stream, &grid);
        if (stats) {
            stats->launches += 1;
            stats->grid = grid;
            stats->kernel = 3;
            stats->group = GA.g;
        }
        return err;
    }
    if (stats) stats->kernel = (scheduler == 1) ? 1 : 2;
    if (scheduler != 1) {
        auto kern = pass_persistent_kernel<T, WMAX>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, tpb, smem);
        if (err != cudaSuccess) return err;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        long long grid = (long long)per_sm * cfg.num_sms;
        // Sweeps in flight at once: sweep 0 has about 2n/b half-steps and each
        // later sweep starts lagh half-steps after its predecessor.  CTAs
        // beyond that only spin on their first flag.
        const long long in_flight = (2 * (P.n - P.bp)) / ((long long)P.b * P.lagh) + 2;
        grid = std::min<long long>(grid, in_flight + in_flight / 4 + 8);
        if (cfg.max_ctas > 0) grid = std::min<long long>(grid, cfg.max_ctas);
        grid = std::min<long long>(grid, P.nsweeps);
        if (grid < 1) return cudaSuccess;
        err = cudaMemsetAsync(progress, 0, sizeof(int) * (size_t)P.nsweeps, stream);
        if (err != cudaSuccess) return err;
        T* band_arg = band;
        PassArgs p_arg = P;
        int* prog_arg = progress;
        int* stat_arg = status;
        void* args[] = {&band_arg, &p_arg, &prog_arg, &stat_arg};
        err = cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(tpb), args,
                                          smem, stream);
        if (stats) {
            stats->launches += 1;
            stats->grid = (int)grid;
        }
        return err;
    }
    // Per-cycle scheduler.
    auto kern = pass_cycle_kernel<T, WMAX>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const long long S = P.nsweeps;
    if (S <= 0) return cudaSuccess;
    auto steps = [&](long long r) -> long long {
        long long last = P.n - 2 - r - P.bp;
        return last < 0 ? 0 : last / P.b + 1;
    };
    long long tmax = 0;
    for (long long r = 0; r < S; ++r) tmax = std::max(tmax, P.lag * r + steps(r) - 1);
    long long r_lo = 0;
    for (long long T0 = 0; T0 <= tmax; ++T0) {
        // active sweeps: 0 <= T0 - lag r <= K_r - 1
        while (r_lo < S && T0 - P.lag * r_lo > steps(r_lo) - 1) ++r_lo;
        long long r_hi = std::min(S - 1, T0 / P.lag);
        if (r_hi < r_lo) continue;
        kern<<<(unsigned)(r_hi - r_lo + 1), tpb, smem, stream>>>(band, P, (int)T0, (int)r_lo);
        if (stats) stats->launches += 1;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_pass(T* band, const PassArgs& P, int scheduler, const LaunchCfg& cfg_in,
                     int* progress, int* status, cudaStream_t stream, LaunchStats* stats) {
    LaunchCfg cfg = cfg_in;
    const int wmax = wmax_bucket(P.t + 1);
    if (scheduler == 0 || scheduler == 3) {
        // group kernel where enough sweeps' columns fit shared memory and the
        // storage suits bulk copies; the flag kernel otherwise
        const bool ok = group_layout_ok(band, P.ldab, sizeof(T)) &&
                        choose_group(P, scheduler, cfg.group_size, sizeof(T), &cfg.group);
        scheduler = ok ? 3 : 2;
    }
    switch (wmax) {
#define BB_CASE(W) \
        case W: return run_pass_w<T, W>(band, P, scheduler, cfg, progress, status, stream, stats);
        BB_CASE(8) BB_CASE(9) BB_CASE(16) BB_CASE(17) BB_CASE(32) BB_CASE(33) BB_CASE(65)
#undef BB_CASE
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t run_zero_fill(T* band, long long n, long long ldab, int tw, int ku, cudaStream_t s) {
    long long total = n * 2LL * tw;
    if (total <= 0) return cudaSuccess;
    int blocks = (int)std::min<long long>((total + 255) / 256, 4096);
    zero_fill_kernel<T><<<blocks, 256, 0, s>>>(band, n, ldab, tw, ku);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_extract(const T* band, long long n, long long ldab, int ku, T* d, T* e,
                        cudaStream_t s) {
    int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
    extract_kernel<T><<<blocks, 256, 0, s>>>(band, n, ldab, ku, d, e);
    return cudaGetLastError();
}

// Explicit instantiation: one translation unit per (type, width group) so
// that the build compiles them in parallel.
#define BB_INSTANTIATE_W(T, W)                                                                     \
    template cudaError_t run_pass_w<T, W>(T*, const PassArgs&, int, const LaunchCfg&, int*, int*,  \
                                          cudaStream_t, LaunchStats*);
#define BB_EXTERN_W(T, W)                                                                          \
    extern template cudaError_t run_pass_w<T, W>(T*, const PassArgs&, int, const LaunchCfg&, int*, \
                                                 int*, cudaStream_t, LaunchStats*);
#define BB_INSTANTIATE(T)                                                                          \
    template cudaError_t run_pass<T>(T*, const PassArgs&, int, const LaunchCfg&, int*, int*,       \
                                     cudaStream_t, LaunchStats*);                                  \
    template cudaError_t run_zero_fill<T>(T*, long long, long long, int, int, cudaStream_t);       \
    template cudaError_t run_extract<T>(const T*, long long, long long, int, T*, T*, cudaStream_t);

}  // namespace bb
