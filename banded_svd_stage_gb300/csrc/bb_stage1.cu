// Stage 1 of the two-stage SVD on the GPU: a dense n x n matrix reduced to
// upper band form of bandwidth bw by orthogonal transformations (the first
// stage of "Accelerating Bidiagonalization of Banded Matrices through
// Memory-Aware Bulge-Chasing on GPUs", Section V, the "classical block
// Householder reduction" its accuracy protocol runs before the band stage;
// the GPU stage 1 of "A two-stage reduction on an Apple M5 Pro" uses the same
// panels).
//
// For each panel of bw columns k .. k+bw-1:
//   QR of the panel, column by column: the reflector of A(j.., j) (LAPACK
//   xLARFG convention) is applied from the left to every later column;
//   LQ of the panel's rows right of the band, row by row: the reflector of
//   A(i, i+bw ..) is applied from the right to every later row.
// Annihilated entries are set to exactly zero.  One reflector is built by one
// block (block-wide scaled norm) and applied as a rank-one update: one block
// per trailing column for a left reflector (its column is contiguous), a
// row-parallel product then a rank-one update for a right reflector.  The
// arithmetic is in the matrix's own precision; these are SIMT kernels (the
// tensor cores of this GPU have no float64 rate worth using, and TF32 would
// lose float32 accuracy).
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/bb.h"
#include "bb_device.cuh"
#include "bb_internal.h"

namespace bb {

constexpr int kS1Threads = 256;

template <typename T>
__device__ __forceinline__ T block_reduce_sum(T v, T* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    T s = 0;
    if (threadIdx.x < 32) {
        s = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : T(0);
        s = warp_sum(s);
        if (threadIdx.x == 0) red[32] = s;
    }
    __syncthreads();
    return red[32];
}
template <typename T>
__device__ __forceinline__ T block_reduce_max(T v, T* red) {
    v = warp_max(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    T s = 0;
    if (threadIdx.x < 32) {
        s = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : T(0);
        s = warp_max(s);
        if (threadIdx.x == 0) red[32] = s;
    }
    __syncthreads();
    return red[32];
}

// Reflector of x[0], x[inc], ..., x[(m-1) inc] (m >= 2), one block: on
// return v[0 .. m-1] holds v (v[0] = 1), *tau_out tau, x[0] = beta and the
// other entries of x are exactly zero.  Norm of the tail: the largest
// magnitude first, then the sum of squares of the scaled entries; tiny
// results are rescaled by safmin as LAPACK does.
template <typename T>
__global__ void __launch_bounds__(kS1Threads) s1_larfg_kernel(T* __restrict__ x, long long inc, int m,
                                                               T* __restrict__ v, T* __restrict__ tau_out) {
    __shared__ T red[33];
    T amax = 0;
    for (int i = 1 + threadIdx.x; i < m; i += blockDim.x) amax = fmax(amax, fabs(x[(long long)i * inc]));
    const T scale = block_reduce_max(amax, red);
    T alpha = x[0];
    if (scale == T(0)) {
        for (int i = threadIdx.x; i < m; i += blockDim.x) v[i] = (i == 0) ? T(1) : T(0);
        if (threadIdx.x == 0) *tau_out = T(0);
        return;
    }
    T ss = 0;
    for (int i = 1 + threadIdx.x; i < m; i += blockDim.x) {
        const T u = x[(long long)i * inc] / scale;
        ss = fma(u, u, ss);
    }
    ss = block_reduce_sum(ss, red);
    T xnorm = scale * dev_sqrt(ss);
    T beta = (alpha >= T(0)) ? -dev_hypot(alpha, xnorm) : dev_hypot(alpha, xnorm);
    const T safmin = Lim<T>::safmin();
    int knt = 0;
    T mult = T(1);  // the scaling applied to x's tail
    if (fabs(beta) < safmin) {
        const T rsafmn = T(1) / safmin;
        do {
            ++knt;
            mult = mult * rsafmn;
            beta = beta * rsafmn;
            alpha = alpha * rsafmn;
        } while (fabs(beta) < safmin && knt < 20);
        xnorm = xnorm * mult;
        beta = (alpha >= T(0)) ? -dev_hypot(alpha, xnorm) : dev_hypot(alpha, xnorm);
    }
    const T tau = (beta - alpha) / beta;
    const T scal = T(1) / (alpha - beta);
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
        if (i == 0) {
            v[0] = T(1);
        } else {
            T* xi = x + (long long)i * inc;
            v[i] = (*xi * mult) * scal;
            *xi = T(0);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int j = 0; j < knt; ++j) beta = beta * safmin;
        x[0] = beta;
        *tau_out = tau;
    }
}

// Left application: columns c0 + blockIdx.x (+ gridDim.x ...), rows r0 ..
// r0+m-1 of the column-major matrix: y = v^T A(r0.., c), A(r0.., c) -= tau v y.
template <typename T>
__global__ void __launch_bounds__(kS1Threads) s1_apply_left_kernel(T* __restrict__ a, long long lda, int r0,
                                                                    int m, int c0, int c1,
                                                                    const T* __restrict__ v,
                                                                    const T* __restrict__ tau_p) {
    __shared__ T red[33];
    const T tau = *tau_p;
    if (tau == T(0)) return;
    for (int c = c0 + blockIdx.x; c < c1; c += gridDim.x) {
        T* col = a + (long long)c * lda + r0;
        T y = 0;
        for (int i = threadIdx.x; i < m; i += blockDim.x) y = fma(v[i], col[i], y);
        y = block_reduce_sum(y, red);
        const T s = tau * y;
        for (int i = threadIdx.x; i < m; i += blockDim.x) col[i] = fma(-s, v[i], col[i]);
        __syncthreads();
    }
}

// Right application, part one: y[r] = sum_c A(r0 + r, c0 + c) u[c], one
// thread per row (consecutive threads, consecutive rows of a column).
template <typename T>
__global__ void s1_gemv_rows_kernel(const T* __restrict__ a, long long lda, int r0, int mr, int c0, int mc,
                                    const T* __restrict__ u, T* __restrict__ y, const T* __restrict__ tau_p) {
    if (*tau_p == T(0)) return;
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < mr; r += gridDim.x * blockDim.x) {
        const T* row = a + (long long)c0 * lda + r0 + r;
        T s = 0;
        for (int c = 0; c < mc; ++c) s = fma(row[(long long)c * lda], u[c], s);
        y[r] = s;
    }
}

// Right application, part two: A(r0 + r, c0 + c) -= tau y[r] u[c].
template <typename T>
__global__ void s1_rank1_kernel(T* __restrict__ a, long long lda, int r0, int mr, int c0, int mc,
                                const T* __restrict__ u, const T* __restrict__ y, const T* __restrict__ tau_p) {
    const T tau = *tau_p;
    if (tau == T(0)) return;
    for (int c = blockIdx.y; c < mc; c += gridDim.y) {
        T* col = a + (long long)(c0 + c) * lda + r0;
        const T tu = tau * u[c];
        for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < mr; r += gridDim.x * blockDim.x)
            col[r] = fma(-y[r], tu, col[r]);
    }
}

// Band storage from the dense band: band[(ku + i - j) + j ldab] = A(i, j) for
// 0 <= j - i <= bw, every other stored entry of the column zero.
template <typename T>
__global__ void s1_pack_kernel(const T* __restrict__ a, long long lda, long long n, int bw, int ku,
                               T* __restrict__ band, long long ldab) {
    const long long total = n * ldab;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long j = e / ldab, q = e % ldab;
        const long long i = j + q - ku;
        const bool in = (i >= 0) && (i <= j) && (j - i <= bw);
        band[e] = in ? a[i + j * lda] : T(0);
    }
}

template <typename T>
static cudaError_t run_stage1(T* a, long long n, long long lda, int bw, T* ws, int num_sms, cudaStream_t s) {
    T* v = ws;          // n entries
    T* y = ws + n;      // n entries
    T* tau = ws + 2 * n;  // 1 entry
    const int apply_grid = std::max(1, 4 * num_sms);
    cudaError_t err = cudaSuccess;
    for (long long k = 0; k < n && err == cudaSuccess; k += bw) {
        const long long kb = std::min(k + bw, n);
        for (long long j = k; j < kb && err == cudaSuccess; ++j) {
            if (j + 1 >= n) break;
            const int m = (int)(n - j);
            s1_larfg_kernel<T><<<1, kS1Threads, 0, s>>>(a + j + j * lda, 1, m, v, tau);
            const int ncols = (int)(n - j - 1);
            s1_apply_left_kernel<T><<<std::min(ncols, apply_grid), kS1Threads, 0, s>>>(
                a, lda, (int)j, m, (int)(j + 1), (int)n, v, tau);
            err = cudaGetLastError();
        }
        for (long long i = k; i < kb && err == cudaSuccess; ++i) {
            const long long c0 = i + bw;
            if (c0 + 1 >= n) break;
            const int mc = (int)(n - c0);
            s1_larfg_kernel<T><<<1, kS1Threads, 0, s>>>(a + i + c0 * lda, lda, mc, v, tau);
            const int mr = (int)(n - i - 1);
            if (mr > 0) {
                const unsigned gx = (unsigned)std::max(1, std::min((mr + 255) / 256, apply_grid));
                s1_gemv_rows_kernel<T><<<gx, 256, 0, s>>>(a, lda, (int)(i + 1), mr, (int)c0, mc, v, y, tau);
                const unsigned gy = (unsigned)std::max(1, std::min(mc, 2 * apply_grid));
                s1_rank1_kernel<T><<<dim3(gx, gy), 256, 0, s>>>(a, lda, (int)(i + 1), mr, (int)c0, mc, v, y, tau);
            }
            err = cudaGetLastError();
        }
    }
    return err;
}

}  // namespace bb

namespace {
bool device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}
bb_status s1_fail(bb_status st, const char* msg) {
    bb::set_last_error(msg);
    return st;
}
}  // namespace

extern "C" int64_t bb_dense_to_band_workspace(int64_t n, bb_dtype dtype) {
    if (n < 1 || (dtype != BB_F32 && dtype != BB_F64)) return -1;
    return (2 * n + 16) * (dtype == BB_F64 ? 8 : 4);
}

extern "C" bb_status bb_dense_to_band(bb_dtype dtype, int64_t n, int64_t bw, void* a, int64_t lda, void* workspace,
                                      int64_t workspace_bytes, bb_stream_t stream) {
    if (dtype != BB_F32 && dtype != BB_F64) return s1_fail(BB_ERR_DTYPE, "bb_dense_to_band: float32 or float64 only");
    if (n < 1 || n >= (int64_t)1 << 30 || bw < 1 || lda < n)
        return s1_fail(BB_ERR_INVALID_ARG, "bb_dense_to_band: need 1 <= n < 2^30, bw >= 1, lda >= n");
    if (workspace_bytes < bb_dense_to_band_workspace(n, dtype))
        return s1_fail(BB_ERR_INVALID_ARG, "bb_dense_to_band: workspace smaller than bb_dense_to_band_workspace");
    if (!a || !workspace || !device_ptr(a) || !device_ptr(workspace))
        return s1_fail(BB_ERR_INVALID_ARG, "bb_dense_to_band: a and workspace must be device pointers");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) {
        cudaStream_t s = (cudaStream_t)stream;
        if (dtype == BB_F32)
            e = bb::run_stage1<float>((float*)a, n, lda, (int)std::min<int64_t>(bw, n), (float*)workspace, sms, s);
        else
            e = bb::run_stage1<double>((double*)a, n, lda, (int)std::min<int64_t>(bw, n), (double*)workspace, sms, s);
    }
    if (e != cudaSuccess) return s1_fail(BB_ERR_CUDA, cudaGetErrorString(e));
    return BB_OK;
}

extern "C" bb_status bb_pack_band(bb_dtype dtype, int64_t n, int64_t bw, int64_t tw, const void* a, int64_t lda,
                                  void* band, int64_t ldab, bb_stream_t stream) {
    if (dtype != BB_F32 && dtype != BB_F64) return s1_fail(BB_ERR_DTYPE, "bb_pack_band: float32 or float64 only");
    if (n < 1 || bw < 0 || bw >= n || tw < 0 || lda < n) return s1_fail(BB_ERR_INVALID_ARG, "bb_pack_band: bad sizes");
    if (ldab < bw + 2 * tw + 1) return s1_fail(BB_ERR_LDAB, "bb_pack_band: ldab < bw + 2*tw + 1");
    if (!a || !band || !device_ptr(a) || !device_ptr(band))
        return s1_fail(BB_ERR_INVALID_ARG, "bb_pack_band: a and band must be device pointers");
    const long long total = n * ldab;
    const unsigned grid = (unsigned)std::min<long long>((total + 255) / 256, 8192);
    cudaStream_t s = (cudaStream_t)stream;
    const int ku = (int)(bw + tw);
    if (dtype == BB_F32)
        bb::s1_pack_kernel<float><<<grid, 256, 0, s>>>((const float*)a, lda, n, (int)bw, ku, (float*)band, ldab);
    else
        bb::s1_pack_kernel<double><<<grid, 256, 0, s>>>((const double*)a, lda, n, (int)bw, ku, (double*)band, ldab);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return s1_fail(BB_ERR_CUDA, cudaGetErrorString(e));
    return BB_OK;
}
