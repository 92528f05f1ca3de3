// Singular values of an upper bidiagonal matrix (d, e) on the GPU:
// multisection on Sturm counts of the 2n x 2n Golub-Kahan tridiagonal, a
// group of lanes per singular value.
//
// The Golub-Kahan matrix T has a zero diagonal and off-diagonal
// a = (d_0, e_0, d_1, e_1, ..., e_{n-2}, d_{n-1}); its eigenvalues are the
// +- sigma_i.  The number of eigenvalues of T below x is the number of
// negative pivots of T - x I: q_0 = -x, q_i = -x - a_{i-1}^2 / q_{i-1}
// (LAPACK xSTEBZ's count, with its pivmin guard: |q_i| < pivmin becomes
// -pivmin).  For x > 0, #{sigma < x} = count(x) - n.  This is the step the
// two-stage SVD takes right after the band -> bidiagonal reduction ("A
// two-stage reduction on an Apple M5 Pro", Section 7, bisection for the
// bidiagonal singular values); the GPU layout is this library's.
//
// Every thread runs the same number of steps, so a block walks the squared
// off-diagonal in shared-memory chunks in lockstep.  The entries are
// first scaled by a power of two that brings the largest near 1.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "../../include/bb.h"

namespace bb {

void set_last_error(const char* msg);  // bb_api.cu

template <typename T> struct SvLim;
template <> struct SvLim<float> {
    static __device__ __forceinline__ float safmin() { return 1.17549435e-38f; }
};
template <> struct SvLim<double> {
    static __device__ __forceinline__ double safmin() { return 2.2250738585072014e-308; }
};

constexpr int kSvThreads = 128;
constexpr int kSvChunk = 2048;  // squared off-diagonal entries per shared-memory chunk

// sigma[k] = the k-th largest singular value (k = 0 .. n-1).  A group of P
// consecutive lanes of a warp (P a power of two, 1 .. 32) works on one value:
// each step, lane l of the group counts at lo + (hi - lo) (l + 1) / (P + 1)
// and the group keeps the subinterval where the count passes j (the counts
// grow with l, so the lanes at or below j form a prefix: a ballot finds it).
// P = 1 is plain bisection; larger P trades more counts for fewer steps.
template <typename T>
__global__ void __launch_bounds__(kSvThreads)
bidiag_svals_kernel(const T* __restrict__ d, const T* __restrict__ e, int n, int P, int steps,
                    T* __restrict__ sigma) {
    __shared__ T s_a2[kSvChunk];
    __shared__ T s_red[kSvThreads / 32];
    const int m = 2 * n - 1;  // off-diagonal entries of T
    // The largest |a_i|, each block on its own (one pass; the bisection
    // makes tens of them).  The counts run on a * sc, sc the power of two
    // that brings it near 1, so that the squares neither under- nor overflow
    // (as LAPACK scales before bisecting); sigma = result / sc exactly.
    T amax = 0;
    for (int i = threadIdx.x; i < m; i += blockDim.x) amax = fmax(amax, fabs(i & 1 ? e[i >> 1] : d[i >> 1]));
    for (int o = 16; o > 0; o >>= 1) amax = fmax(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0;
    for (int w = 0; w < kSvThreads / 32; ++w) amax = fmax(amax, s_red[w]);
    const T sc = (amax > T(0) && isfinite(amax)) ? ldexp(T(1), -ilogb(amax)) : T(1);
    // Gershgorin bound of the scaled T: max over rows of |a_{i-1}| + |a_i|
    T bound = 0;
    for (int i = threadIdx.x; i <= m; i += blockDim.x) {
        const T left = (i > 0) ? fabs((i - 1) & 1 ? e[(i - 1) >> 1] : d[(i - 1) >> 1]) : T(0);
        const T right = (i < m) ? fabs(i & 1 ? e[i >> 1] : d[i >> 1]) : T(0);
        bound = fmax(bound, (left + right) * sc);
    }
    for (int o = 16; o > 0; o >>= 1) bound = fmax(bound, __shfl_xor_sync(0xffffffffu, bound, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = bound;
    __syncthreads();
    bound = 0;
    for (int w = 0; w < kSvThreads / 32; ++w) bound = fmax(bound, s_red[w]);
    const T amax_s = amax * sc;
    const T pivmin = SvLim<T>::safmin() * fmax(T(1), amax_s * amax_s);

    const int lane = threadIdx.x & 31;
    const int l = lane & (P - 1);                     // lane within the group
    const int gbase = lane & ~(P - 1);                // first lane of the group
    const unsigned gmask = (P == 32) ? 0xffffffffu : (((1u << P) - 1u) << gbase);
    const int k = (blockIdx.x * blockDim.x + threadIdx.x) / P;  // k-th largest
    const int j = n - 1 - k;                                     // j-th smallest
    T lo = 0, hi = bound * T(1.0000001) + pivmin;
    for (int it = 0; it < steps; ++it) {
        const T x = lo + (hi - lo) * T(l + 1) / T(P + 1);
        T q = -x;
        int cnt = (q < T(0)) ? 1 : 0;
        for (int c0 = 0; c0 < m; c0 += kSvChunk) {
            const int len = min(kSvChunk, m - c0);
            __syncthreads();
            for (int i = threadIdx.x; i < len; i += blockDim.x) {
                const int g = c0 + i;
                const T a = ((g & 1) ? e[g >> 1] : d[g >> 1]) * sc;
                s_a2[i] = a * a;
            }
            __syncthreads();
            for (int i = 0; i < len; ++i) {
                q = -x - s_a2[i] / q;
                if (fabs(q) < pivmin) q = -pivmin;
                cnt += (q < T(0)) ? 1 : 0;
            }
        }
        // lanes whose point has at most j singular values below it: a prefix
        const unsigned below = __ballot_sync(0xffffffffu, cnt - n <= j) & gmask;
        const int lstar = __popc(below) - 1;  // last such lane of the group, or -1
        const T xlo = __shfl_sync(0xffffffffu, x, gbase + max(lstar, 0));
        const T xhi = __shfl_sync(0xffffffffu, x, gbase + min(lstar + 1, P - 1));
        if (lstar >= 0) lo = xlo;
        if (lstar < P - 1) hi = xhi;
    }
    if (l == 0 && k < n) sigma[k] = T(0.5) * (lo + hi) / sc;
}

}  // namespace bb

namespace {

// Steps of multisection with P lanes per value: each step keeps one of the
// P + 1 equal parts of the interval, so the least s with (P + 1)^s >= 2^bits
// brings it down to 2^-bits of the starting bound.
int multisection_steps(int P, int bits) {
    const unsigned long long target = 1ull << bits;
    unsigned long long acc = 1;
    int s = 0;
    while (acc < target) {
        acc = (acc > target / (unsigned long long)(P + 1)) ? target : acc * (unsigned long long)(P + 1);
        ++s;
    }
    return s;
}

bb_status launch_svals(bb_dtype dtype, int64_t n, const void* d, const void* e, void* sigma_out, int64_t lanes,
                       bb_stream_t stream) {
    if (n < 1 || n > (int64_t)1 << 29) {
        bb::set_last_error("bb_singular_values: n must be in [1, 2^29]");
        return BB_ERR_INVALID_ARG;
    }
    if (!d || !sigma_out || (n > 1 && !e)) {
        bb::set_last_error("bb_singular_values: null d, e or sigma_out");
        return BB_ERR_INVALID_ARG;
    }
    if (dtype != BB_F32 && dtype != BB_F64) {
        bb::set_last_error("bb_singular_values: unknown dtype");
        return BB_ERR_DTYPE;
    }
    if (lanes != 0 && (lanes < 1 || lanes > 32 || (lanes & (lanes - 1)) != 0)) {
        bb::set_last_error("bb_singular_values: lanes must be 0 or a power of two in [1, 32]");
        return BB_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    // lanes per value: about enough threads to fill the GPU (152 SMs x 2048),
    // a power of two; at most 32 in float, where a count is cheap, and 8 in
    // double, where the division sequence of each count is the bound and
    // extra lanes cost more counts than the steps they save
    int P = (int)lanes;
    if (P == 0) {
        const int cap = (dtype == BB_F32) ? 32 : 8;
        P = 1;
        while (P < cap && (int64_t)P * 2 * n <= (int64_t)152 * 2048) P *= 2;
    }
    // the interval shrinks by P + 1 per step, down to 2^-27 (float) or 2^-56
    // (double) of the bound
    const int steps = multisection_steps(P, (dtype == BB_F32) ? 27 : 56);
    const unsigned grid = (unsigned)((n * P + bb::kSvThreads - 1) / bb::kSvThreads);
    // e may be null for n == 1: the kernel never reads it then (m = 1)
    if (dtype == BB_F32)
        bb::bidiag_svals_kernel<float><<<grid, bb::kSvThreads, 0, s>>>(
            (const float*)d, (const float*)e, (int)n, P, steps, (float*)sigma_out);
    else
        bb::bidiag_svals_kernel<double><<<grid, bb::kSvThreads, 0, s>>>(
            (const double*)d, (const double*)e, (int)n, P, steps, (double*)sigma_out);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) {
        bb::set_last_error(cudaGetErrorString(err));
        return BB_ERR_CUDA;
    }
    return BB_OK;
}

}  // namespace

extern "C" bb_status bb_singular_values(bb_dtype dtype, int64_t n, const void* d, const void* e, void* sigma_out,
                                        bb_stream_t stream) {
    return launch_svals(dtype, n, d, e, sigma_out, 0, stream);
}

extern "C" bb_status bb_singular_values_lanes(bb_dtype dtype, int64_t n, const void* d, const void* e,
                                              void* sigma_out, int64_t lanes, bb_stream_t stream) {
    return launch_svals(dtype, n, d, e, sigma_out, lanes, stream);
}
