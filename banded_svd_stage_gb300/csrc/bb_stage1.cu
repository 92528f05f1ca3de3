// Stage 1 of the two-stage SVD on the GPU: a dense n x n matrix reduced to
// upper band form of bandwidth bw by orthogonal transformations (the first
// stage of "Accelerating Bidiagonalization of Banded Matrices through
// Memory-Aware Bulge-Chasing on GPUs", Section V, the "classical block
// Householder reduction" its accuracy protocol runs before the band stage;
// the GPU stage 1 of "A two-stage reduction on an Apple M5 Pro" uses the same
// panels, with the trailing updates as matrix products).
//
// For each panel of bw columns k .. kb-1 (kb = min(k + bw, n)):
//   QR of the panel, column by column: the reflector of A(j.., j) (LAPACK
//   xLARFG convention) is applied from the left to every later column;
//   LQ of the panel's rows right of the band, row by row: the reflector of
//   A(i, i+bw ..) is applied from the right to every later row.
// Annihilated entries are set to exactly zero.
//
// Blocked (compact WY) form of that sequence, kInner reflectors at a time,
// or fewer where the block would not fit shared memory (the QR reflectors
// of a panel in order, then its LQ reflectors in order):
//   1. s1_panel_kernel (one CTA) factorizes a block of kInner columns:
//      reflector j is built from P(j.., j) and applied to the block's later
//      columns only; it writes V (unit lower trapezoidal), tau and the upper
//      triangular T with H_0 H_1 ... = I - V T V^T (LAPACK xLARFT, forward,
//      columnwise);
//   2. the rest of the matrix is updated with matrix products:
//        QR: rows of the block's reflectors, later columns:  A -= V T^T (V^T A);
//        LQ: rows below the block's rows, their columns:     A -= (A U) T U^T;
//      the long inner products (V^T A, A U) are split over several CTAs and
//      their partial sums added in a fixed order (s1_reduce_tri_kernel, which
//      also applies T).
// The LQ panel is the QR panel kernel on the transposed view of the rows
// (P(i, c) = A(k + c, k + bw + i)).  The products are SIMT tiled GEMMs in
// the matrix's own precision (the tensor cores of this GPU have no float64
// rate worth using, and TF32 would lose float32 accuracy).  The arithmetic
// differs from the reflector-by-reflector sequence only in rounding order.
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/bb.h"
#include "bb_device.cuh"
#include "bb_internal.h"

namespace bb {

// Inner block: reflectors per panel-kernel call; the rest of the matrix is
// updated after every kInner reflectors.
constexpr int kInner = 16;
// Most partial products of a split inner dimension.
constexpr int kMaxSplit = 16;
constexpr int kPanelThreads = 512;
constexpr int kPanelWarps = kPanelThreads / 32;
constexpr int kDotChunk = 16;  // dot products are reduced kDotChunk at a time

// Sum over the block of one value per thread; every thread gets the result.
template <typename T>
__device__ __forceinline__ T s1_block_sum(T v, T* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    T s = 0;
#pragma unroll
    for (int w = 0; w < kPanelWarps; ++w) s += red[w];
    return s;
}
template <typename T>
__device__ __forceinline__ T s1_block_max(T v, T* red) {
    v = warp_max(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    T s = 0;
#pragma unroll
    for (int w = 0; w < kPanelWarps; ++w) s = fmax(s, red[w]);
    return s;
}

// Panel factorization, one CTA.  The panel P (m x nc) is P(i, c) =
// p[i * si + c * sc]; reflectors j = 0 .. nq-1 (nq <= nc, nq <= m - 1), the
// reflector of P(j .. m-1, j) applied to columns j+1 .. nc-1.  Outputs:
//   P(j, j) = beta, P(j+1.., j) = 0;
//   V (m x nq, column-major, ld m): column j is v_j (zeros above row j, 1 at
//   row j);  tau[j];  Tm (nq x nq, column-major): T(l, j) for l <= j;
//   dots (nc entries): scratch.
// Norm as the oracle: the plain sum of squares of the tail; when it under-
// or overflows, the largest magnitude first and the sum of squares of the
// scaled entries; then LAPACK's safmin rescaling for a tiny beta.
template <typename T>
__global__ void __launch_bounds__(kPanelThreads)
s1_panel_kernel(T* __restrict__ p, long long si, long long sc, int m, int nc, int nq, T* __restrict__ V,
                T* __restrict__ tau_out, T* __restrict__ Tm, T* __restrict__ dots) {
    __shared__ T red[kPanelWarps];
    __shared__ T part[kPanelWarps][kDotChunk];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    auto P = [&](int i, int c) -> T& { return p[(long long)i * si + (long long)c * sc]; };
    for (int j = 0; j < nq; ++j) {
        T* vj = V + (long long)j * m;
        const T alpha = P(j, j);
        T ss = 0;
        for (int i = j + 1 + tid; i < m; i += kPanelThreads) {
            const T x = P(i, j);
            ss = fma(x, x, ss);
        }
        ss = s1_block_sum(ss, red);
        T beta, tau, scal, mult = T(1);
        int knt = 0;
        bool identity = false;
        if (isfinite(ss) && ss >= Lim<T>::min_normal()) {
            const T nrm = dev_sqrt(fma(alpha, alpha, ss));
            beta = (alpha >= T(0)) ? -nrm : nrm;
        } else {
            T amax = 0;
            for (int i = j + 1 + tid; i < m; i += kPanelThreads) amax = fmax(amax, fabs(P(i, j)));
            const T scale = s1_block_max(amax, red);
            if (scale == T(0)) {
                identity = true;
                beta = alpha;
            } else {
                T s2 = 0;
                for (int i = j + 1 + tid; i < m; i += kPanelThreads) {
                    const T u = P(i, j) / scale;
                    s2 = fma(u, u, s2);
                }
                s2 = s1_block_sum(s2, red);
                const T xnorm = scale * dev_sqrt(s2);
                beta = (alpha >= T(0)) ? -dev_hypot(alpha, xnorm) : dev_hypot(alpha, xnorm);
                const T safmin = Lim<T>::safmin();
                if (fabs(beta) < safmin) {
                    const T rsafmn = T(1) / safmin;
                    T a2 = alpha;
                    do {
                        ++knt;
                        mult = mult * rsafmn;
                        beta = beta * rsafmn;
                        a2 = a2 * rsafmn;
                    } while (fabs(beta) < safmin && knt < 20);
                    const T xn2 = xnorm * mult;
                    beta = (a2 >= T(0)) ? -dev_hypot(a2, xn2) : dev_hypot(a2, xn2);
                    tau = (beta - a2) / beta;
                    scal = T(1) / (a2 - beta);
                }
            }
        }
        if (!identity && knt == 0) {
            tau = (beta - alpha) / beta;
            scal = T(1) / (alpha - beta);
        }
        if (identity) {
            tau = T(0);
            scal = T(0);
        }
        // v_j, the annihilated entries, beta
        for (int i = tid; i < m; i += kPanelThreads) {
            if (i < j) {
                vj[i] = T(0);
            } else if (i == j) {
                vj[i] = T(1);
            } else {
                T& x = P(i, j);
                vj[i] = identity ? T(0) : (x * mult) * scal;
                x = T(0);
            }
        }
        if (tid == 0) {
            T b = beta;
            for (int q = 0; q < knt; ++q) b = b * Lim<T>::safmin();
            P(j, j) = b;
            tau_out[j] = tau;
        }
        __syncthreads();
        // dot products of v_j (rows j..m-1) with the panel's later columns
        // (dots[c], c > j) and with the earlier reflectors (dots[l], l < j),
        // kDotChunk values at a time: each thread walks its rows once per
        // chunk with the partial sums in registers
        const int R = (tau != T(0)) ? nc - 1 : j;  // values c != j, c < nc
        for (int c0 = 0; c0 < R; c0 += kDotChunk) {
            const int cn = min(kDotChunk, R - c0);
            T d[kDotChunk];
#pragma unroll
            for (int q = 0; q < kDotChunk; ++q) d[q] = T(0);
            if (tau != T(0)) {
                for (int i = j + tid; i < m; i += kPanelThreads) {
                    const T vi = vj[i];
#pragma unroll
                    for (int q = 0; q < kDotChunk; ++q) {
                        if (q < cn) {
                            const int c = (c0 + q < j) ? c0 + q : c0 + q + 1;
                            const T x = (c > j) ? P(i, c) : V[(long long)c * m + i];
                            d[q] = fma(vi, x, d[q]);
                        }
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kDotChunk; ++q) {
                const T w = warp_sum(d[q]);
                if (lane == 0) part[warp][q] = w;
            }
            __syncthreads();
            for (int q = tid; q < cn; q += kPanelThreads) {
                T sum = 0;
#pragma unroll
                for (int w = 0; w < kPanelWarps; ++w) sum += part[w][q];
                dots[(c0 + q < j) ? c0 + q : c0 + q + 1] = sum;
            }
            __syncthreads();
        }
        // P(i, c) -= (tau (v_j . P(:, c))) v_j(i), c > j
        if (tau != T(0)) {
            for (int i = j + tid; i < m; i += kPanelThreads) {
                const T vi = vj[i];
                for (int c = j + 1; c < nc; ++c) P(i, c) = fma(-(tau * dots[c]), vi, P(i, c));
            }
        }
        // T(j, j) = tau_j; T(l, j) = -tau_j sum_{q = l}^{j-1} T(l, q) (v_q . v_j)
        for (int l = tid; l <= j; l += kPanelThreads) {
            T t = tau;
            if (l < j) {
                T s = 0;
                for (int q = l; q < j; ++q) s = fma(Tm[l + (long long)q * nq], dots[q], s);
                t = -tau * s;
            }
            Tm[l + (long long)j * nq] = t;
        }
        __syncthreads();
    }
}

// Panel factorization as s1_panel_kernel, with the panel staged in shared
// memory (m x nc, column-major, ld m) when it fits: one copy in, the steps
// on shared memory, one copy out.  v_j is kept below the diagonal of
// column j (LAPACK's storage) and beta aside until the copy out, which
// writes beta and the zeros to the matrix and v (1 on the diagonal) to V.
// The operations and their order per entry are those of s1_panel_kernel.
constexpr size_t kPanelSmemMax = 200 * 1024;
template <typename T>
__global__ void __launch_bounds__(kPanelThreads)
s1_panel_smem_kernel(T* __restrict__ p, long long si, long long sc, int m, int nc, int nq, T* __restrict__ V,
                     T* __restrict__ tau_out, T* __restrict__ Tm_out) {
    extern __shared__ __align__(16) unsigned char s1_smem[];
    T* Ps = reinterpret_cast<T*>(s1_smem);  // m x nc
    __shared__ T red[kPanelWarps];
    __shared__ T part[kPanelWarps][kDotChunk];
    __shared__ T sdots[kInner];
    __shared__ T sbeta[kInner], stau[kInner];
    __shared__ T sT[kInner * kInner];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    // copy in, consecutive threads on the matrix's contiguous index (32-bit
    // indices: the panel has at most kPanelSmemMax / sizeof(T) entries)
    if (sc == 1) {  // rows of the matrix: lane group c = tid % kInner of row i
        const int c = tid % kInner;
        for (int i = tid / kInner; i < m; i += kPanelThreads / kInner)
            if (c < nc) Ps[i + c * m] = p[(long long)i * si + c];
    } else {
        for (int c = 0; c < nc; ++c)
            for (int i = tid; i < m; i += kPanelThreads) Ps[i + c * m] = p[i + (long long)c * sc];
    }
    __syncthreads();
    auto P = [&](int i, int c) -> T& { return Ps[i + c * m]; };
    for (int j = 0; j < nq; ++j) {
        const T alpha = P(j, j);
        T ss = 0;
        for (int i = j + 1 + tid; i < m; i += kPanelThreads) {
            const T x = P(i, j);
            ss = fma(x, x, ss);
        }
        ss = s1_block_sum(ss, red);
        T beta, tau, scal, mult = T(1);
        int knt = 0;
        bool identity = false;
        if (isfinite(ss) && ss >= Lim<T>::min_normal()) {
            const T nrm = dev_sqrt(fma(alpha, alpha, ss));
            beta = (alpha >= T(0)) ? -nrm : nrm;
        } else {
            T amax = 0;
            for (int i = j + 1 + tid; i < m; i += kPanelThreads) amax = fmax(amax, fabs(P(i, j)));
            const T scale = s1_block_max(amax, red);
            if (scale == T(0)) {
                identity = true;
                beta = alpha;
            } else {
                T s2 = 0;
                for (int i = j + 1 + tid; i < m; i += kPanelThreads) {
                    const T u = P(i, j) / scale;
                    s2 = fma(u, u, s2);
                }
                s2 = s1_block_sum(s2, red);
                const T xnorm = scale * dev_sqrt(s2);
                beta = (alpha >= T(0)) ? -dev_hypot(alpha, xnorm) : dev_hypot(alpha, xnorm);
                const T safmin = Lim<T>::safmin();
                if (fabs(beta) < safmin) {
                    const T rsafmn = T(1) / safmin;
                    T a2 = alpha;
                    do {
                        ++knt;
                        mult = mult * rsafmn;
                        beta = beta * rsafmn;
                        a2 = a2 * rsafmn;
                    } while (fabs(beta) < safmin && knt < 20);
                    const T xn2 = xnorm * mult;
                    beta = (a2 >= T(0)) ? -dev_hypot(a2, xn2) : dev_hypot(a2, xn2);
                    tau = (beta - a2) / beta;
                    scal = T(1) / (a2 - beta);
                }
            }
        }
        if (!identity && knt == 0) {
            tau = (beta - alpha) / beta;
            scal = T(1) / (alpha - beta);
        }
        if (identity) {
            tau = T(0);
            scal = T(0);
        }
        // v_j below the diagonal (each thread its own rows: the rows it reads
        // next), 1 on the diagonal
        for (int i = j + 1 + tid; i < m; i += kPanelThreads) {
            T& x = P(i, j);
            x = identity ? T(0) : (x * mult) * scal;
        }
        if (tid == 0) {
            T b = beta;
            for (int q = 0; q < knt; ++q) b = b * Lim<T>::safmin();
            sbeta[j] = b;
            stau[j] = tau;
            P(j, j) = T(1);
        }
        __syncthreads();
        const int R = (tau != T(0)) ? nc - 1 : j;
        for (int c0 = 0; c0 < R; c0 += kDotChunk) {
            const int cn = min(kDotChunk, R - c0);
            T d[kDotChunk];
#pragma unroll
            for (int q = 0; q < kDotChunk; ++q) d[q] = T(0);
            if (tau != T(0)) {
                for (int i = j + tid; i < m; i += kPanelThreads) {
                    const T vi = P(i, j);
#pragma unroll
                    for (int q = 0; q < kDotChunk; ++q) {
                        if (q < cn) {
                            const int c = (c0 + q < j) ? c0 + q : c0 + q + 1;
                            // v_c(i) for an earlier reflector (i >= j > c: below its diagonal)
                            d[q] = fma(vi, P(i, c), d[q]);
                        }
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kDotChunk; ++q) {
                const T w = warp_sum(d[q]);
                if (lane == 0) part[warp][q] = w;
            }
            __syncthreads();
            for (int q = tid; q < cn; q += kPanelThreads) {
                T sum = 0;
#pragma unroll
                for (int w = 0; w < kPanelWarps; ++w) sum += part[w][q];
                sdots[(c0 + q < j) ? c0 + q : c0 + q + 1] = sum;
            }
            __syncthreads();
        }
        if (tau != T(0)) {
            for (int i = j + tid; i < m; i += kPanelThreads) {
                const T vi = P(i, j);
                for (int c = j + 1; c < nc; ++c) P(i, c) = fma(-(tau * sdots[c]), vi, P(i, c));
            }
        }
        for (int l = tid; l <= j; l += kPanelThreads) {
            T t = tau;
            if (l < j) {
                T sum = 0;
                for (int q = l; q < j; ++q) sum = fma(sT[l + q * nq], sdots[q], sum);
                t = -tau * sum;
            }
            sT[l + j * nq] = t;
        }
        __syncthreads();
    }
    // copy out: R and the zeros to the matrix, v to V, tau and T
    auto out_of = [&](int i, int c) -> T {
        if (c < nq) {
            if (i > c) return T(0);
            if (i == c) return sbeta[c];
        }
        return P(i, c);
    };
    if (sc == 1) {
        const int c = tid % kInner;
        for (int i = tid / kInner; i < m; i += kPanelThreads / kInner)
            if (c < nc) p[(long long)i * si + c] = out_of(i, c);
    } else {
        for (int c = 0; c < nc; ++c)
            for (int i = tid; i < m; i += kPanelThreads) p[i + (long long)c * sc] = out_of(i, c);
    }
    for (int c = 0; c < nq; ++c)
        for (int i = tid; i < m; i += kPanelThreads)
            V[i + (long long)c * m] = (i < c) ? T(0) : (i == c) ? T(1) : P(i, c);
    for (int e = tid; e < nq * nq; e += kPanelThreads) Tm_out[e] = sT[e];
    for (int e = tid; e < nq; e += kPanelThreads) tau_out[e] = stau[e];
}

// Launch of one panel factorization: shared memory when the panel fits.
template <typename T>
static cudaError_t s1_panel(T* p, long long si, long long sc, int m, int nc, int nq, T* V, T* tau, T* Tm, T* dots,
                            cudaStream_t s) {
    const size_t bytes = sizeof(T) * (size_t)m * (size_t)nc;
    if (bytes <= kPanelSmemMax) {  // (run_stage1 raised the kernel's dynamic shared memory limit)
        s1_panel_smem_kernel<T><<<1, kPanelThreads, bytes, s>>>(p, si, sc, m, nc, nq, V, tau, Tm);
    } else {
        s1_panel_kernel<T><<<1, kPanelThreads, 0, s>>>(p, si, sc, m, nc, nq, V, tau, Tm, dots);
    }
    return cudaGetLastError();
}

// C = alpha op(A) op(B) + beta C, column-major (M x N, inner dimension K):
// op(A)(i, l) = TA ? A[l + i lda] : A[i + l lda], op(B)(l, j) = TB ?
// B[j + l ldb] : B[l + j ldb].  A CTA of 16 x 16 threads computes a
// (16 PM) x (16 PN) tile of C, each thread PM x PN entries (rows tx + 16 p,
// columns ty + 16 q), the inner dimension in steps of 16 through shared
// memory with the next step's tiles fetched into registers meanwhile.
// PM = PN = 4 for the square products; 1 x 16 and 16 x 1 for the skinny
// ones (16 rows or columns of output).  beta is 0 (C is not read) or 1.
// Split inner dimension: CTA z sums l in [z kchunk, (z + 1) kchunk) into
// C + z cz (partial products, reduced by the caller).
constexpr int kGemmBK = 16;
template <typename T, bool TA, bool TB, int PM, int PN>
__global__ void __launch_bounds__(256)
s1_gemm_kernel(int M, int N, int K, T alpha, const T* __restrict__ A, long long lda, const T* __restrict__ B,
               long long ldb, T beta, T* __restrict__ C, long long ldc, int kchunk, long long cz) {
    constexpr int BM = 16 * PM, BN = 16 * PN;
    __shared__ T As[kGemmBK][BM + 1];
    __shared__ T Bs[kGemmBK][BN + 1];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int i0 = blockIdx.x * BM, j0 = blockIdx.y * BN;
    const int lbeg = blockIdx.z * kchunk, lend = min(K, lbeg + kchunk);
    C += blockIdx.z * cz;
    T acc[PM][PN];
#pragma unroll
    for (int a = 0; a < PM; ++a)
#pragma unroll
        for (int b = 0; b < PN; ++b) acc[a][b] = T(0);
    // tile loads: element e of the 16 x BM (16 x BN) tile, consecutive
    // threads on the contiguous index of A (B)
    constexpr int kPerA = kGemmBK * BM / 256, kPerB = kGemmBK * BN / 256;
    T ra[kPerA], rb[kPerB];
    auto fetch = [&](int l0) {
#pragma unroll
        for (int u = 0; u < kPerA; ++u) {
            const int e = tid + 256 * u;
            const int ii = TA ? e / kGemmBK : e % BM;
            const int ll = TA ? e % kGemmBK : e / BM;
            const int gi = i0 + ii, gl = l0 + ll;
            ra[u] = (gi < M && gl < lend) ? (TA ? A[gl + (long long)gi * lda] : A[gi + (long long)gl * lda]) : T(0);
        }
#pragma unroll
        for (int u = 0; u < kPerB; ++u) {
            const int e = tid + 256 * u;
            const int jj = TB ? e % BN : e / kGemmBK;
            const int ll = TB ? e / BN : e % kGemmBK;
            const int gj = j0 + jj, gl = l0 + ll;
            rb[u] = (gj < N && gl < lend) ? (TB ? B[gj + (long long)gl * ldb] : B[gl + (long long)gj * ldb]) : T(0);
        }
    };
    auto stash = [&]() {
#pragma unroll
        for (int u = 0; u < kPerA; ++u) {
            const int e = tid + 256 * u;
            As[TA ? e % kGemmBK : e / BM][TA ? e / kGemmBK : e % BM] = ra[u];
        }
#pragma unroll
        for (int u = 0; u < kPerB; ++u) {
            const int e = tid + 256 * u;
            Bs[TB ? e / BN : e % kGemmBK][TB ? e % BN : e / kGemmBK] = rb[u];
        }
    };
    if (lbeg < lend) fetch(lbeg);
    for (int l0 = lbeg; l0 < lend; l0 += kGemmBK) {
        stash();
        __syncthreads();
        if (l0 + kGemmBK < lend) fetch(l0 + kGemmBK);
#pragma unroll
        for (int l = 0; l < kGemmBK; ++l) {
            T a[PM], b[PN];
#pragma unroll
            for (int q = 0; q < PM; ++q) a[q] = As[l][tx + 16 * q];
#pragma unroll
            for (int q = 0; q < PN; ++q) b[q] = Bs[l][ty + 16 * q];
#pragma unroll
            for (int pa = 0; pa < PM; ++pa)
#pragma unroll
                for (int pb = 0; pb < PN; ++pb) acc[pa][pb] = fma(a[pa], b[pb], acc[pa][pb]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int pb = 0; pb < PN; ++pb) {
        const int gj = j0 + ty + 16 * pb;
        if (gj >= N) continue;
#pragma unroll
        for (int pa = 0; pa < PM; ++pa) {
            const int gi = i0 + tx + 16 * pa;
            if (gi >= M) continue;
            T* c = C + gi + (long long)gj * ldc;
            *c = (beta == T(0)) ? alpha * acc[pa][pb] : fma(alpha, acc[pa][pb], *c);
        }
    }
}

// nsplit > 1: nsplit partial products of the inner dimension into C + z cz
// (beta must be 0).  The output shape picks the tile: 16 x 256 when M <= 16,
// 256 x 16 when N <= 16, else 64 x 64.
template <typename T, bool TA, bool TB>
static cudaError_t s1_gemm(int M, int N, int K, T alpha, const T* A, long long lda, const T* B, long long ldb,
                           T beta, T* C, long long ldc, cudaStream_t s, int nsplit = 1, long long cz = 0) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    const int kchunk = (nsplit > 1) ? ((K + nsplit - 1) / nsplit + kGemmBK - 1) / kGemmBK * kGemmBK : K;
    const int pm = (M <= 16) ? 1 : (N <= 16 ? 16 : 4);
    const int pn = (M <= 16) ? 16 : (N <= 16 ? 1 : 4);
    const int bm = 16 * pm, bn = 16 * pn;
    // column blocks of C within the grid's y limit
    const int nmax = 65535 * bn;
    for (int j0 = 0; j0 < N; j0 += nmax) {
        const int nb = std::min(nmax, N - j0);
        const T* Bj = TB ? B + j0 : B + (long long)j0 * ldb;
        T* Cj = C + (long long)j0 * ldc;
        const dim3 grid((unsigned)((M + bm - 1) / bm), (unsigned)((nb + bn - 1) / bn), (unsigned)std::max(1, nsplit));
        if (pm == 1)
            s1_gemm_kernel<T, TA, TB, 1, 16><<<grid, 256, 0, s>>>(M, nb, K, alpha, A, lda, Bj, ldb, beta, Cj, ldc,
                                                                  kchunk, cz);
        else if (pm == 16)
            s1_gemm_kernel<T, TA, TB, 16, 1><<<grid, 256, 0, s>>>(M, nb, K, alpha, A, lda, Bj, ldb, beta, Cj, ldc,
                                                                  kchunk, cz);
        else
            s1_gemm_kernel<T, TA, TB, 4, 4><<<grid, 256, 0, s>>>(M, nb, K, alpha, A, lda, Bj, ldb, beta, Cj, ldc,
                                                                 kchunk, cz);
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// W[q qs + j ls] = sum_{l <= j} T(l, j) w_l, w_l = sum_z Wp[z zs + q qs + l ls]
// (z ascending), for the nvec vectors q of nb <= kInner entries: with
// columns of W this is T^T W, with rows W T.  A block takes kInner vectors,
// one thread per entry: the partial sums are added with consecutive threads
// on the contiguous index (l when ls == 1, else q), the vectors staged in
// shared memory, then each thread forms one output entry.
template <typename T>
__global__ void __launch_bounds__(kInner * kInner)
s1_reduce_tri_kernel(const T* __restrict__ Wp, int nsplit, long long zs, T* __restrict__ W, int nvec,
                     long long qs, long long ls, int nb, const T* __restrict__ Tm) {
    __shared__ T w[kInner][kInner + 1];  // [vector][entry]
    __shared__ T t[kInner * kInner];
    const int tid = threadIdx.x;
    const bool l_fast = (ls == 1);
    const int a = tid % kInner, b2 = tid / kInner;
    const int l = l_fast ? a : b2, qq = l_fast ? b2 : a;  // entry l of vector qq of the block
    if (tid < nb * nb) t[tid] = Tm[tid];
    for (int q0 = blockIdx.x * kInner; q0 < nvec; q0 += gridDim.x * kInner) {
        const int q = q0 + qq;
        T sum = 0;
        if (q < nvec && l < nb) {
            const long long off = (long long)q * qs + (long long)l * ls;
            for (int z = 0; z < nsplit; ++z) sum += Wp[z * zs + off];
        }
        w[qq][l] = sum;
        __syncthreads();
        if (q < nvec && l < nb) {
            T out = 0;
            for (int k = 0; k <= l; ++k) out = fma(t[k + l * nb], w[qq][k], out);
            W[(long long)q * qs + (long long)l * ls] = out;
        }
        __syncthreads();
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

// Workspace (elements), b = min(bw, kInner): V or U (n x b), W (n x b), the
// partial products (kMaxSplit x n x b), T (b x b), tau and dots (b each).
static long long s1_workspace_elems(long long n, long long bw) {
    const long long b = std::min<long long>(std::min(bw, n), kInner);
    return (2 + kMaxSplit) * n * b + b * b + 2 * b + 64;
}

// Partial products for a product of nvec x nb outputs with a long inner
// dimension K: enough for several CTAs per SM, at least 256 of K each.
static int s1_splits(long long tiles, long long K, int num_sms) {
    long long z = (8LL * num_sms + tiles - 1) / std::max(1LL, tiles);
    z = std::min<long long>(z, std::max(1LL, K / 256));
    return (int)std::max(1LL, std::min<long long>(z, kMaxSplit));
}

// Reflectors per block for a panel of m rows: kInner, or fewer so that the
// block fits the shared-memory panel kernel; below the narrowest width
// worth its extra passes over the trailing matrix (1 in float; 8 in double,
// whose products are bound by the FP64 rate) the global-memory panel kernel
// takes kInner.  Measured on a dense 4096 x 4096, bw 16: float 174 -> 105
// ms with narrowing down to 1; double 917 ms without narrowing, 1425 ms
// narrowing down to 6.
template <typename T>
static int s1_block_width(long long m, long long nb) {
    const long long fit = (long long)(kPanelSmemMax / sizeof(T)) / std::max(1LL, m);
    const long long narrowest = std::min<long long>(nb, sizeof(T) == 8 ? 8 : 1);
    return (int)(fit >= narrowest ? std::min(nb, fit) : nb);
}

template <typename T>
static cudaError_t run_stage1(T* a, long long n, long long lda, int bw, T* ws, int num_sms, cudaStream_t s) {
    const long long nb = std::min(kInner, bw);
    T* V = ws;                   // m x nq (QR) or m x nl (LQ), ld m
    T* W = V + n * nb;           // nq x N (QR, ld nq) or M x nl (LQ, ld M)
    T* Wp = W + n * nb;          // kMaxSplit partial products of W
    T* Tm = Wp + kMaxSplit * n * nb;  // nq x nq
    T* tau = Tm + nb * nb;
    T* dots = tau + nb;
    const long long zs = n * nb;
    const unsigned vec_grid = (unsigned)std::max(1, 4 * num_sms);
    cudaError_t err = cudaFuncSetAttribute(s1_panel_smem_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kPanelSmemMax);
    for (long long k = 0; k < n && err == cudaSuccess; k += bw) {
        const long long kb = std::min(k + bw, n);
        // QR of columns k .. kb-1, kInner reflectors at a time: reflectors
        // j = cs .. cs+nq-1 (j < min(kb, n-1)) on the sub-panel of columns
        // cs .. cs+nc-1, then columns cs+nc .. n-1 of rows cs .. updated
        const long long qend = std::min(kb, n - 1);
        for (long long cs = k, nbs = 0; cs < qend && err == cudaSuccess; cs += nbs) {
            nbs = s1_block_width<T>(n - cs, nb);
            const int nq = (int)std::min<long long>(nbs, qend - cs);
            const int nc = (int)std::min<long long>(nbs, kb - cs);
            const int m = (int)(n - cs);
            err = s1_panel<T>(a + cs + cs * lda, 1, lda, m, nc, nq, V, tau, Tm, dots, s);
            const int N = (int)(n - cs - nc);
            if (err == cudaSuccess && N > 0) {
                T* At = a + cs + (cs + nc) * lda;  // rows cs .., columns cs + nc ..
                const long long tiles = (N + 255) / 256;  // 16 x 256 tiles of W (nq <= 16 rows)
                const int z = s1_splits(tiles, m, num_sms);
                // W = T^T (V^T At)
                err = s1_gemm<T, true, false>(nq, N, m, T(1), V, m, At, lda, T(0), Wp, nq, s, z, zs);
                if (err == cudaSuccess) {
                    s1_reduce_tri_kernel<T><<<std::min<unsigned>(vec_grid, (unsigned)((N + kInner - 1) / kInner)),
                                              kInner * kInner, 0, s>>>(Wp, z, zs, W, N, nq, 1, nq, Tm);
                    err = cudaGetLastError();
                }
                // At -= V W
                if (err == cudaSuccess) err = s1_gemm<T, false, false>(m, N, nq, T(-1), V, m, W, nq, T(1), At, lda, s);
            }
        }
        // LQ of rows k .. kb-1 right of the band, kInner rows at a time:
        // reflectors i = rs .. rs+nl-1 (i + bw + 1 < n) on the block rows
        // rs .., columns rs + bw ..; then rows rs+nl .. n-1 of those columns
        const long long lend = std::min(kb, n - 1 - bw);
        for (long long rs = k, nbs = 0; rs < lend && err == cudaSuccess; rs += nbs) {
            nbs = s1_block_width<T>(n - rs - bw, nb);
            const int nl = (int)std::min<long long>(nbs, lend - rs);
            const int m = (int)(n - rs - bw);  // columns rs + bw .. n-1
            T* B = a + rs + (rs + bw) * lda;   // B(r, c) = A(rs + r, rs + bw + c)
            err = s1_panel<T>(B, lda, 1, m, nl, nl, V, tau, Tm, dots, s);
            const int M = (int)(n - rs - nl);  // rows rs + nl .. n-1
            if (err == cudaSuccess && M > 0) {
                T* At = a + (rs + nl) + (rs + bw) * lda;
                const long long tiles = (M + 255) / 256;  // 256 x 16 tiles of W (nl <= 16 columns)
                const int z = s1_splits(tiles, m, num_sms);
                // W = (At U) T
                err = s1_gemm<T, false, false>(M, nl, m, T(1), At, lda, V, m, T(0), Wp, M, s, z, zs);
                if (err == cudaSuccess) {
                    s1_reduce_tri_kernel<T><<<std::min<unsigned>(vec_grid, (unsigned)((M + kInner - 1) / kInner)),
                                              kInner * kInner, 0, s>>>(Wp, z, zs, W, M, 1, M, nl, Tm);
                    err = cudaGetLastError();
                }
                // At -= W U^T
                if (err == cudaSuccess) err = s1_gemm<T, false, true>(M, m, nl, T(-1), W, M, V, m, T(1), At, lda, s);
            }
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

extern "C" int64_t bb_dense_to_band_workspace(int64_t n, int64_t bw, bb_dtype dtype) {
    if (n < 1 || n >= (int64_t)1 << 30 || bw < 1 || (dtype != BB_F32 && dtype != BB_F64)) return -1;
    return bb::s1_workspace_elems(n, bw) * (dtype == BB_F64 ? 8 : 4);
}

extern "C" bb_status bb_dense_to_band(bb_dtype dtype, int64_t n, int64_t bw, void* a, int64_t lda, void* workspace,
                                      int64_t workspace_bytes, bb_stream_t stream) {
    if (dtype != BB_F32 && dtype != BB_F64) return s1_fail(BB_ERR_DTYPE, "bb_dense_to_band: float32 or float64 only");
    if (n < 1 || n >= (int64_t)1 << 30 || bw < 1 || lda < n)
        return s1_fail(BB_ERR_INVALID_ARG, "bb_dense_to_band: need 1 <= n < 2^30, bw >= 1, lda >= n");
    if (workspace_bytes < bb_dense_to_band_workspace(n, bw, dtype))
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
