// Back-transformation: the singular vectors' transforms U and V of the band
// -> bidiagonal reduction, from the reflectors the flag kernel recorded.
//
// The reduction applies left reflectors L_i and right reflectors R_i in the
// order pass -> sweep -> step (right, then left), so A = U B V^T with
// U = L_1 L_2 ... and V = R_1 R_2 ...  ("Accelerating Bidiagonalization of
// Banded Matrices through Memory-Aware Bulge-Chasing on GPUs", Section III,
// keeps the reflector vectors for this).  Both products are formed from the
// identity by multiplying on the right, reflector by reflector in that
// order.  The reflectors of one sweep act on disjoint column ranges
// (c_k = r + b' + k b, width t + 1 < b), so they commute and one launch
// applies all of them at once; consecutive sweeps overlap and run in order.
#include <cuda_runtime.h>

#include <algorithm>

#include "bb_vectors.h"

namespace bb {

template <typename T>
__global__ void identity_kernel(T* __restrict__ M, long long n, long long ld) {
    const long long total = n * n;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long j = idx / n, i = idx % n;
        M[i + j * ld] = (i == j) ? T(1) : T(0);
    }
}

// M <- M H_k for every reflector k of one sweep (one side): H_k acts on
// columns c_k .. c_k + w_k - 1.  blockIdx.y walks the reflectors, threads the
// rows (column-major M: consecutive threads, consecutive addresses).
template <typename T>
__global__ void apply_sweep_kernel(T* __restrict__ M, long long ld, long long n, const T* __restrict__ rec_v,
                                   const T* __restrict__ rec_tau, long long idx0, int K, long long r, int b, int t,
                                   int bp, int stride) {
    for (int k = blockIdx.y; k < K; k += gridDim.y) {
        const long long idx = idx0 + 2LL * k;
        const T tau = rec_tau[idx];
        if (tau == T(0)) continue;
        const long long c = r + bp + (long long)k * b;
        const long long ce = min(c + (long long)t, n - 1);
        const int w = (int)(ce - c + 1);
        const T* v = rec_v + idx * stride;
        T* col = M + c * ld;
        for (long long row = blockIdx.x * (long long)blockDim.x + threadIdx.x; row < n;
             row += (long long)gridDim.x * blockDim.x) {
            T y = 0;
            for (int m = 0; m < w; ++m) y = fma(col[row + m * ld], v[m], y);
            const T s = tau * y;
            for (int m = 0; m < w; ++m) col[row + m * ld] = fma(-s, v[m], col[row + m * ld]);
        }
    }
}

template <typename T>
cudaError_t run_back_transform(long long n, int bw, int tw, const T* rec_v, const T* rec_tau, int stride, T* U,
                               long long ldu, T* V, long long ldv, int num_sms, cudaStream_t s,
                               long long* launches) {
    long long nl = 0;
    const unsigned ig = (unsigned)std::max<long long>(1, std::min<long long>((n * n + 255) / 256, 8LL * num_sms));
    if (U) identity_kernel<T><<<ig, 256, 0, s>>>(U, n, ldu);
    if (V) identity_kernel<T><<<ig, 256, 0, s>>>(V, n, ldv);
    nl += (U != nullptr) + (V != nullptr);
    cudaError_t err = cudaGetLastError();
    const unsigned gx = (unsigned)std::max<long long>(1, std::min<long long>((n + 255) / 256, 16));
    long long base = 0;  // index of the first reflector of the pass
    int b = bw;
    while (err == cudaSuccess && b > 1) {
        const int t = std::min(tw, b - 1);
        const int bp = b - t;
        long long prefix = 0;  // steps of the sweeps before r
        for (long long r = 0; r + bp + 1 <= n - 1 && err == cudaSuccess; ++r) {
            const long long last = n - 2 - r - bp;
            const int K = last < 0 ? 0 : (int)(last / b + 1);
            if (K > 0) {
                const unsigned gy = (unsigned)std::min(K, 65535);
                const long long idx_r = base + 2 * prefix;
                if (V) {
                    apply_sweep_kernel<T><<<dim3(gx, gy), 256, 0, s>>>(V, ldv, n, rec_v, rec_tau, idx_r, K, r, b, t,
                                                                       bp, stride);
                    ++nl;
                }
                if (U) {
                    apply_sweep_kernel<T><<<dim3(gx, gy), 256, 0, s>>>(U, ldu, n, rec_v, rec_tau, idx_r + 1, K, r, b,
                                                                       t, bp, stride);
                    ++nl;
                }
                err = cudaGetLastError();
            }
            prefix += K;
        }
        base += 2 * prefix;
        b -= t;
    }
    if (launches) *launches = nl;
    return err;
}

template cudaError_t run_back_transform<float>(long long, int, int, const float*, const float*, int, float*,
                                               long long, float*, long long, int, cudaStream_t, long long*);
template cudaError_t run_back_transform<double>(long long, int, int, const double*, const double*, int, double*,
                                                long long, double*, long long, int, cudaStream_t, long long*);

}  // namespace bb
