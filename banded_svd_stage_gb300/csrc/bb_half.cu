// Half-precision storage: the band, d and e in IEEE binary16, every step's
// arithmetic in float.
//
// "Accelerating Bidiagonalization of Banded Matrices through Memory-Aware
// Bulge-Chasing on GPUs" (arXiv 2510.12705), Section V, runs the reduction
// in FP16 as well as FP32/FP64.  Here each half-step reads the entries it
// touches into float, builds and applies the reflector in float (LAPACK
// xLARFG convention, warp 0), and writes every entry it changes back rounded
// to binary16 (round to nearest even); the reflector itself stays in float.
// Entries of one half-step are therefore rounded exactly once per write, as
// in a run on binary16 storage.
//
// Schedulers, per pass:
// - the flag kernel here: the flag kernel's progress protocol (one CTA per
//   sweep, persistent, cooperative launch): half-step h of sweep r starts
//   once sweep r-1 has completed min(h + lagh, H_{r-1}) half-steps, and a
//   sweep reports its last half-step only after its predecessor reported all
//   of its own.  Every half-step reads its whole window after its wait,
//   through L2 (ld.global.cg), so the data a neighbouring CTA wrote is never
//   read from a stale L1 line;
// - the group kernel (bb_group.cuh) with binary16 storage: the columns are
//   buffered in shared memory as stored, and each half-step converts the
//   entries it reads to float and rounds the ones it writes, exactly as
//   here.  Both kernels give bitwise equal results.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "bb_device.cuh"
#include "bb_group.cuh"
#include "bb_half.h"

namespace bb {

constexpr int kHalfThreads = 256;

__device__ __forceinline__ float h_ld(const __half* p) { return __half2float(__ldcg(p)); }
__device__ __forceinline__ void h_st(__half* p, float v) { *p = __float2half_rn(v); }

// Right half-step: reflector from row p over columns c..ce, applied from the
// right to rows p+1..ce.  A(i, j) = base[i + j * stride].
template <int WMAX>
__device__ __forceinline__ void half_right(__half* __restrict__ base, long long stride, const StepGeom& g,
                                           float* s_v, float* s_tau) {
    constexpr int NPL = (WMAX + 31) / 32;
    const int W = g.w;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float x[NPL];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            x[q] = (m < W) ? h_ld(base + g.p + (g.c + m) * stride) : 0.f;
        }
        const float beta = warp_larfg<float, NPL>(x, W, lane, s_v, s_tau);
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            if (m < W) h_st(base + g.p + (g.c + m) * stride, (m == 0) ? beta : 0.f);
        }
    }
    __syncthreads();
    const float tau = *s_tau;
    if (tau == 0.f) return;  // the same value in every thread
    for (int i = 1 + (int)threadIdx.x; i <= g.nrows; i += blockDim.x) {
        __half* row = base + g.p + i + g.c * stride;
        float x[WMAX];
        float y = 0.f;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) {
                x[m] = h_ld(row + m * stride);
                y = fmaf(x[m], s_v[m], y);
            }
        const float s = tau * y;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) h_st(row + m * stride, fmaf(-s, s_v[m], x[m]));
    }
}

// Left half-step: reflector from column c over rows c..ce, applied from the
// left to columns c+1..cend.
template <int WMAX>
__device__ __forceinline__ void half_left(__half* __restrict__ base, long long stride, const StepGeom& g,
                                          float* s_v, float* s_tau) {
    constexpr int NPL = (WMAX + 31) / 32;
    const int W = g.w;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        __half* colc = base + g.c + g.c * stride;  // colc[m] = A(c + m, c)
        float x[NPL];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            x[q] = (m < W) ? h_ld(colc + m) : 0.f;
        }
        const float beta = warp_larfg<float, NPL>(x, W, lane, s_v, s_tau);
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            if (m < W) h_st(colc + m, (m == 0) ? beta : 0.f);
        }
    }
    __syncthreads();
    const float tau = *s_tau;
    if (tau == 0.f) return;
    for (int dj = 1 + (int)threadIdx.x; dj < g.ncol; dj += blockDim.x) {
        __half* col = base + g.c + (g.c + dj) * stride;  // col[m] = A(c + m, c + dj)
        float x[WMAX];
        float y = 0.f;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) {
                x[m] = h_ld(col + m);
                y = fmaf(s_v[m], x[m], y);
            }
        const float s = tau * y;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) h_st(col + m, fmaf(-s, s_v[m], x[m]));
    }
}

template <int WMAX>
__global__ void __launch_bounds__(kHalfThreads)
pass_half_kernel(__half* __restrict__ band, PassArgs P, int* __restrict__ progress, int* __restrict__ status) {
    __shared__ float s_v[WMAX];
    __shared__ float s_tau;
    __shared__ int s_flag;
    if (threadIdx.x == 0) s_flag = ld_relaxed_gpu(status);
    __syncthreads();
    if (s_flag != kStatusOk) return;
    const long long stride = P.ldab - 1;
    __half* base = band + P.ku;
    for (int r = blockIdx.x; r < P.nsweeps; r += gridDim.x) {
        const int K = sweep_steps(P, r);
        const int Hprev = (r > 0) ? 2 * sweep_steps(P, r - 1) : 0;
        const bool publish = (r != P.stall_sweep);
        for (int k = 0; k < K; ++k) {
            const StepGeom g = step_geom(P, r, k);
            if (r > 0) {
                if (!block_wait(progress + r - 1, min(2 * k + P.lagh, Hprev), status, P, &s_flag)) return;
            } else {
                __syncthreads();  // s_v of the previous half-step is no longer read
            }
            half_right<WMAX>(base, stride, g, s_v, &s_tau);
            block_publish_if(progress + r, 2 * k + 1, publish);
            if (r > 0 && !block_wait(progress + r - 1, min(2 * k + 1 + P.lagh, Hprev), status, P, &s_flag))
                return;
            half_left<WMAX>(base, stride, g, s_v, &s_tau);
            if (k == K - 1 && r > 0 && !block_wait(progress + r - 1, Hprev, status, P, &s_flag)) return;
            block_publish_if(progress + r, 2 * k + 2, publish);
        }
    }
}

__global__ void half_zero_fill_kernel(__half* __restrict__ band, long long n, long long ldab, int tw, int ku) {
    const long long total = n * (2LL * tw);
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long j = e / (2 * tw);
        const int q = (int)(e % (2 * tw));
        const int row = (q < tw) ? q : ku + 1 + (q - tw);
        band[row + j * ldab] = __float2half_rn(0.f);
    }
}

// d_i = A(i, i), e_i = A(i, i+1).
__global__ void half_extract_kernel(const __half* __restrict__ band, long long n, long long ldab, int ku,
                                    __half* __restrict__ d, __half* __restrict__ e) {
    const long long stride = ldab - 1;
    const __half* base = band + ku;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        d[i] = base[i + i * stride];
        if (i + 1 < n) e[i] = base[i + (i + 1) * stride];
    }
}

template <int WMAX>
static cudaError_t run_half_pass_w(__half* band, const PassArgs& P, const HalfLaunch& L, cudaStream_t s,
                                   int* grid_out) {
    auto kern = pass_half_kernel<WMAX>;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kHalfThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = std::min<long long>((long long)per_sm * L.num_sms, P.nsweeps);
    if (L.max_ctas > 0) grid = std::min<long long>(grid, L.max_ctas);
    err = cudaMemsetAsync(L.progress, 0, sizeof(int) * (size_t)P.nsweeps, s);
    if (err != cudaSuccess) return err;
    __half* band_arg = band;
    PassArgs p_arg = P;
    int* prog_arg = L.progress;
    int* stat_arg = L.status;
    void* args[] = {&band_arg, &p_arg, &prog_arg, &stat_arg};
    if (grid_out) *grid_out = (int)grid;
    return cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(kHalfThreads), args, 0, s);
}

// Reflector lengths the binary16 group kernel is compiled for (0: none).
static int half_group_wmax(int w) { return w <= 9 ? 9 : (w <= 17 ? 17 : (w <= 33 ? 33 : 0)); }

bool half_choose_group(const PassArgs& P, int scheduler, int group_size, GroupArgs* out) {
    if (scheduler != 0 && scheduler != 3) return false;
    if (P.nsweeps <= 0 || P.n >= kGroupMaxN) return false;
    const int wmax = half_group_wmax(P.t + 1);
    if (wmax == 0) return false;
    GroupArgs ga;
    if (!plan_group(P, wmax, sizeof(float), group_size, &ga, ChaseKind::kBidiag, sizeof(__half))) return false;
    if (scheduler == 0 && ga.g < kAutoGroupMin) return false;
    if (out) *out = ga;
    return true;
}

template <int WMAX>
static cudaError_t run_half_group_w(__half* band, const PassArgs& P, const GroupArgs& GA, const HalfLaunch& L,
                                    cudaStream_t s) {
    return launch_group_pass<float, WMAX, BidiagChase, __half>(band, P, GA, L.num_sms, L.max_ctas, L.progress,
                                                                L.status, s);
}

cudaError_t run_half_pass(void* band, const PassArgs& P, const HalfLaunch& L, const GroupArgs* GA,
                          cudaStream_t s) {
    if (P.nsweeps <= 0) return cudaSuccess;
    __half* b = static_cast<__half*>(band);
    const int w = P.t + 1;
    if (GA) {
        const int wmax = half_group_wmax(w);
        if (wmax == 9) return run_half_group_w<9>(b, P, *GA, L, s);
        if (wmax == 17) return run_half_group_w<17>(b, P, *GA, L, s);
        if (wmax == 33) return run_half_group_w<33>(b, P, *GA, L, s);
        return cudaErrorInvalidValue;
    }
    if (w <= 9) return run_half_pass_w<9>(b, P, L, s, nullptr);
    if (w <= 17) return run_half_pass_w<17>(b, P, L, s, nullptr);
    if (w <= 33) return run_half_pass_w<33>(b, P, L, s, nullptr);
    return run_half_pass_w<65>(b, P, L, s, nullptr);
}

cudaError_t run_half_zero_fill(void* band, long long n, long long ldab, int tw, int ku, int num_sms, cudaStream_t s) {
    const long long total = n * 2LL * tw;
    if (total <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)std::min<long long>((total + 255) / 256, 4LL * num_sms);
    half_zero_fill_kernel<<<grid, 256, 0, s>>>(static_cast<__half*>(band), n, ldab, tw, ku);
    return cudaGetLastError();
}

cudaError_t run_half_extract(const void* band, long long n, long long ldab, int ku, void* d, void* e, int num_sms,
                             cudaStream_t s) {
    const unsigned grid = (unsigned)std::max<long long>(1, std::min<long long>((n + 255) / 256, 4LL * num_sms));
    half_extract_kernel<<<grid, 256, 0, s>>>(static_cast<const __half*>(band), n, ldab, ku, static_cast<__half*>(d),
                                             static_cast<__half*>(e));
    return cudaGetLastError();
}

}  // namespace bb
