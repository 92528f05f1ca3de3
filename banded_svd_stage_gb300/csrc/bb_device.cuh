// Device code of the band -> bidiagonal bulge-chasing reduction (sm_103a).
//
// Method: "Accelerating Bidiagonalization of Banded Matrices through
// Memory-Aware Bulge-Chasing on GPUs" (arXiv 2510.12705), Section III:
//   - one sweep per row R; each cycle of a sweep annihilates one horizontal
//     group (TW entries of a row, plus the entry to their left as the
//     reflector's first element) and then one vertical group (the leftmost
//     column of the bulge that the horizontal reflector created);
//   - Algorithm 2 text: the entries to annihilate are staged cooperatively,
//     the reflector is computed jointly, written back, and then the threads
//     loop over the rows (columns) of the block holding rows of width TW+1 in
//     registers;
//   - the three-cycle separation between consecutive sweeps is what makes
//     concurrent sweeps safe; here it is refined to half-step granularity
//     (see pass_lag_half in bb_api.cu).
// The Householder reflector uses the LAPACK xLARFG convention.
//
// Band storage: A(i, j) = band[(ku + i - j) + j * ldab], so with
// base = band + ku and stride = ldab - 1, A(i, j) = base[i + j * stride]:
// a row of the matrix is strided by ldab - 1, a column is contiguous.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bb {

enum : int { kStatusOk = 0, kStatusTimeout = 5 };

struct PassArgs {
    long long n;          // matrix order
    long long ldab;       // leading dimension of the band storage
    int b;                // bandwidth at the start of the pass
    int t;                // entries annihilated per reflector (tile width)
    int bp;               // b - t, bandwidth after the pass
    int ku;               // band row holding the main diagonal (= BW + TW)
    int nsweeps;          // sweeps r = 0 .. nsweeps-1 (n - bp - 1, or 0)
    int lag;              // cycle lag of the per-cycle scheduler (2 or 3)
    int lagh;             // half-step lag of the persistent scheduler (2, 3 or 4)
    int stall_sweep;      // fault injection: this sweep never publishes (-1: none)
    unsigned long long wait_budget;  // SM clock cycles a flag wait may spin
};

// Number of steps of sweep r: k runs while c_k + 1 <= n - 1.
__device__ __forceinline__ int sweep_steps(const PassArgs& P, long long r) {
    long long last = P.n - 2 - r - P.bp;
    return last < 0 ? 0 : (int)(last / P.b) + 1;
}

template <typename T> struct Lim;
template <> struct Lim<float> {
    static __device__ __forceinline__ float min_normal() { return 1.17549435e-38f; }
    // tiny / (eps/2), the threshold below which LAPACK rescales beta
    static __device__ __forceinline__ float safmin() { return 1.17549435e-38f / 5.96046448e-08f; }
};
template <> struct Lim<double> {
    static __device__ __forceinline__ double min_normal() { return 2.2250738585072014e-308; }
    static __device__ __forceinline__ double safmin() {
        return 2.2250738585072014e-308 / 1.1102230246251565e-16;
    }
};

__device__ __forceinline__ float dev_hypot(float a, float b) { return hypotf(a, b); }
__device__ __forceinline__ double dev_hypot(double a, double b) { return hypot(a, b); }
__device__ __forceinline__ float dev_sqrt(float a) { return sqrtf(a); }
__device__ __forceinline__ double dev_sqrt(double a) { return sqrt(a); }

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
template <typename T>
__device__ __forceinline__ T warp_max(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Euclidean norm of the entries m = 1 .. w-1 held by a warp (entry m in lane
// m % 32, slot m / 32).  Plain sum of squares; if it under- or overflows while
// some entry is nonzero, the sum is retaken on entries divided by the largest
// magnitude, so a zero norm means every entry is zero.
template <typename T, int NPL>
__device__ __forceinline__ T warp_tail_norm(const T (&x)[NPL], int w, int lane) {
    T ss = 0;
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        int m = lane + 32 * q;
        if (m >= 1 && m < w) ss = fma(x[q], x[q], ss);
    }
    ss = warp_sum(ss);
    if (isfinite(ss) && ss >= Lim<T>::min_normal()) return dev_sqrt(ss);
    T scale = 0;
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        int m = lane + 32 * q;
        if (m >= 1 && m < w) scale = fmax(scale, fabs(x[q]));
    }
    scale = warp_max(scale);
    if (scale == T(0)) return T(0);
    T s2 = 0;
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        int m = lane + 32 * q;
        if (m >= 1 && m < w) {
            T u = x[q] / scale;
            s2 = fma(u, u, s2);
        }
    }
    s2 = warp_sum(s2);
    return scale * dev_sqrt(s2);
}

// Householder reflector of the w entries held by one warp (LAPACK xLARFG
// convention): on return s_v[0..w-1] = v (v_0 = 1), *s_tau = tau, and the
// function returns beta (all lanes).  tau == 0 means H = I and beta = alpha.
template <typename T, int NPL>
__device__ __forceinline__ T warp_larfg(T (&x)[NPL], int w, int lane, T* s_v, T* s_tau) {
    T alpha = __shfl_sync(0xffffffffu, x[0], 0);
    T xnorm = (w > 1) ? warp_tail_norm<T, NPL>(x, w, lane) : T(0);
    if (xnorm == T(0)) {
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            int m = lane + 32 * q;
            if (m < w) s_v[m] = (m == 0) ? T(1) : T(0);
        }
        if (lane == 0) *s_tau = T(0);
        return alpha;
    }
    T beta = (alpha >= T(0)) ? -dev_hypot(alpha, xnorm) : dev_hypot(alpha, xnorm);
    const T safmin = Lim<T>::safmin();
    int knt = 0;
    if (fabs(beta) < safmin) {
        const T rsafmn = T(1) / safmin;
        do {
            ++knt;
#pragma unroll
            for (int q = 0; q < NPL; ++q) x[q] = x[q] * rsafmn;
            beta = beta * rsafmn;
            alpha = alpha * rsafmn;
        } while (fabs(beta) < safmin && knt < 20);
        xnorm = warp_tail_norm<T, NPL>(x, w, lane);
        beta = (alpha >= T(0)) ? -dev_hypot(alpha, xnorm) : dev_hypot(alpha, xnorm);
    }
    const T tau = (beta - alpha) / beta;
    const T scal = T(1) / (alpha - beta);
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        int m = lane + 32 * q;
        if (m < w) s_v[m] = (m == 0) ? T(1) : x[q] * scal;
    }
    if (lane == 0) *s_tau = tau;
    for (int j = 0; j < knt; ++j) beta = beta * safmin;
    return beta;
}

// Shared-memory layout of one CTA.
//   v[WMAX]          reflector of the current half-step
//   tau              its scalar
//   tile[ncol][WP]   the column block of the left half-step: rows c..ce of
//                    columns c..cend, column-major with odd column stride WP
template <typename T>
struct Smem {
    T* v;
    T* tau;
    T* tile;
    int wp;
};

template <typename T, int WMAX>
__device__ __forceinline__ Smem<T> carve_smem(unsigned char* raw) {
    Smem<T> s;
    T* p = reinterpret_cast<T*>(raw);
    s.v = p;
    s.tau = p + WMAX;
    s.tile = p + WMAX + 2;
    s.wp = WMAX | 1;
    return s;
}

// ---------------------------------------------------------------------------
// Right (horizontal) half-step of sweep r, step k: reflector from row p over
// columns c..ce, applied from the right to rows p+1..ce.  Rows c..ce of the
// result (the part the left half-step needs) are also left in the tile.
// ---------------------------------------------------------------------------
template <typename T, int WMAX>
__device__ __forceinline__ void right_half(T* __restrict__ band, const PassArgs& P, int r, int k,
                                           const Smem<T>& sm) {
    constexpr int NPL = (WMAX + 31) / 32;
    const long long stride = P.ldab - 1;
    T* __restrict__ base = band + P.ku;
    const long long c = (long long)r + P.bp + (long long)k * P.b;
    const long long p = (k == 0) ? (long long)r : c - P.b;
    const long long ce = min(c + (long long)P.t, P.n - 1);
    const int w = (int)(ce - c + 1);
    const int nrows = (int)(ce - p);  // rows p+1 .. ce
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31;

    // Stage: warp 0 holds row p (entries m = lane + 32 q); every thread loads
    // the first chunk of its rows before the reflector is known.
    T xp[NPL];
    if (tid < 32) {
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            int m = lane + 32 * q;
            xp[q] = (m < w) ? __ldcg(base + p + (c + m) * stride) : T(0);
        }
    }
    T x[WMAX];
    int i_loc = tid;  // row p + 1 + i_loc
    if (i_loc < nrows) {
        const T* src = base + (p + 1 + i_loc) + c * stride;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < w) x[m] = __ldcg(src + m * stride);
    }
    if (tid < 32) {
        T beta = warp_larfg<T, NPL>(xp, w, lane, sm.v, sm.tau);
        // row p becomes (beta, 0, ..., 0)
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            int m = lane + 32 * q;
            if (m < w) base[p + (c + m) * stride] = (m == 0) ? beta : T(0);
        }
    }
    __syncthreads();
    const T tau = *sm.tau;
    const long long row_c = c - p - 1;  // local index of row c
    for (; i_loc < nrows; i_loc += nthr) {
        if (i_loc >= nthr) {  // later chunks: load now
            const T* src = base + (p + 1 + i_loc) + c * stride;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) x[m] = __ldcg(src + m * stride);
        }
        if (tau != T(0)) {
            T y = 0;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) y = fma(x[m], sm.v[m], y);
            const T s = tau * y;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) x[m] = fma(-s, sm.v[m], x[m]);
        }
        T* dst = base + (p + 1 + i_loc) + c * stride;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < w) dst[m * stride] = x[m];
        const long long rr = i_loc - row_c;  // row c + rr
        if (rr >= 0) {
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) sm.tile[m * sm.wp + rr] = x[m];
        }
    }
}

// ---------------------------------------------------------------------------
// Left (vertical) half-step of sweep r, step k: reflector from column c over
// rows c..ce, applied from the left to columns c+1..cend.  Expects the tile's
// first w columns to hold rows c..ce of columns c..ce (left there by the
// right half-step of the same step, which this CTA ran just before).
// ---------------------------------------------------------------------------
template <typename T, int WMAX>
__device__ __forceinline__ void left_half(T* __restrict__ band, const PassArgs& P, int r, int k,
                                          const Smem<T>& sm) {
    constexpr int NPL = (WMAX + 31) / 32;
    const long long stride = P.ldab - 1;
    T* __restrict__ base = band + P.ku;
    const long long c = (long long)r + P.bp + (long long)k * P.b;
    const long long ce = min(c + (long long)P.t, P.n - 1);
    const long long cend = min(ce + (long long)P.b, P.n - 1);
    const int w = (int)(ce - c + 1);
    const int ncol = (int)(cend - c + 1);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarp = nthr >> 5;
    const int wp = sm.wp;

    // Stage the columns ce+1 .. cend (a warp per column, lanes over rows).
    for (int jl = w + warp; jl < ncol; jl += nwarp) {
        const T* src = base + c + (c + jl) * stride;
        for (int m = lane; m < w; m += 32) sm.tile[jl * wp + m] = __ldcg(src + m);
    }
    __syncthreads();
    if (tid < 32) {
        T xc[NPL];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            int m = lane + 32 * q;
            xc[q] = (m < w) ? sm.tile[m] : T(0);
        }
        T beta = warp_larfg<T, NPL>(xc, w, lane, sm.v, sm.tau);
        __syncwarp();
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            int m = lane + 32 * q;
            if (m < w) sm.tile[m] = (m == 0) ? beta : T(0);
        }
    }
    __syncthreads();
    const T tau = *sm.tau;
    if (tau != T(0)) {
        for (int jl = 1 + tid; jl < ncol; jl += nthr) {
            T x[WMAX];
            T* col = sm.tile + jl * wp;
            T y = 0;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) {
                    x[m] = col[m];
                    y = fma(sm.v[m], x[m], y);
                }
            const T s = tau * y;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) col[m] = fma(-s, sm.v[m], x[m]);
        }
    }
    __syncthreads();
    // Write the whole block back (columns c .. cend, rows c .. ce).
    for (int jl = warp; jl < ncol; jl += nwarp) {
        T* dst = base + c + (c + jl) * stride;
        for (int m = lane; m < w; m += 32) dst[m] = sm.tile[jl * wp + m];
    }
}

// ---------------------------------------------------------------------------
// Cross-CTA progress flags (persistent scheduler).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Block-wide wait until *flag >= target.  Thread 0 spins with acquire loads;
// the wait is bounded by P.wait_budget SM clock cycles and by an iteration
// cap, and gives up early if another CTA has already latched an error.  On
// giving up it latches kStatusTimeout and the block returns false.
__device__ __forceinline__ bool block_wait(const int* flag, int target, int* status,
                                           const PassArgs& P, int* s_flag) {
    if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire_gpu(flag) < target) {
            const long long t0 = clock64();
            unsigned int it = 0;
            for (;;) {
                if (ld_acquire_gpu(flag) >= target) break;
                ++it;
                if ((it & 255u) == 0u) {
                    if (ld_relaxed_gpu(status) != kStatusOk) { ok = 0; break; }
                    if ((unsigned long long)(clock64() - t0) > P.wait_budget || it > (1u << 30)) {
                        atomicCAS(status, kStatusOk, kStatusTimeout);
                        ok = 0;
                        break;
                    }
                }
            }
        }
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

// Publish "this sweep has completed `value` half-steps": every thread's
// stores are ordered before the flag by the barrier and a gpu-scope fence.
__device__ __forceinline__ void block_publish(int* flag, int value) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        st_release_gpu(flag, value);
    }
}

// Persistent scheduler: CTAs take sweeps r = blockIdx.x, blockIdx.x + grid,
// ... in order.  Half-step h (right: 2k, left: 2k+1) of sweep r starts once
// sweep r-1 has completed min(h + lagh, H_{r-1}) half-steps; a sweep reports
// its last half-step only after its predecessor reported all of its own, so
// "sweep r complete" implies every earlier sweep is complete.  Requires all
// CTAs to be co-resident (cooperative launch).
// Register budget: a thread holds one row (or column) of WMAX entries plus
// addressing state, so the block size is capped to leave it the registers.
template <typename T, int WMAX>
struct MaxThreads {
    static constexpr int value = (WMAX * sizeof(T) <= 33 * 4) ? 512 : 256;
};

template <typename T, int WMAX>
__global__ void __launch_bounds__(MaxThreads<T, WMAX>::value)
pass_persistent_kernel(T* __restrict__ band, PassArgs P, int* __restrict__ progress,
                       int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_flag;
    const Smem<T> sm = carve_smem<T, WMAX>(smem_raw);
    if (ld_relaxed_gpu(status) != kStatusOk) return;
    for (int r = blockIdx.x; r < P.nsweeps; r += gridDim.x) {
        const int K = sweep_steps(P, r);
        const int Hprev = (r > 0) ? 2 * sweep_steps(P, r - 1) : 0;
        const bool publish = (r != P.stall_sweep);
        for (int k = 0; k < K; ++k) {
            if (r > 0 && !block_wait(progress + r - 1, min(2 * k + P.lagh, Hprev), status, P, &s_flag))
                return;
            right_half<T, WMAX>(band, P, r, k, sm);
            if (publish) block_publish(progress + r, 2 * k + 1);
            else __syncthreads();
            if (r > 0 && !block_wait(progress + r - 1, min(2 * k + 1 + P.lagh, Hprev), status, P, &s_flag))
                return;
            left_half<T, WMAX>(band, P, r, k, sm);
            if (k == K - 1 && r > 0 && !block_wait(progress + r - 1, Hprev, status, P, &s_flag)) return;
            if (publish) block_publish(progress + r, 2 * k + 2);
            else __syncthreads();
        }
    }
}

// Per-cycle scheduler (one launch per cycle): block b runs step
// k = cycle - lag * r of sweep r = r_first + b.  Steps in one cycle touch
// disjoint windows, and the launch boundary orders consecutive cycles.
template <typename T, int WMAX>
__global__ void __launch_bounds__(MaxThreads<T, WMAX>::value)
pass_cycle_kernel(T* __restrict__ band, PassArgs P, int cycle, int r_first) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const Smem<T> sm = carve_smem<T, WMAX>(smem_raw);
    const int r = r_first + blockIdx.x;
    const int k = cycle - P.lag * r;
    right_half<T, WMAX>(band, P, r, k, sm);
    __syncthreads();
    left_half<T, WMAX>(band, P, r, k, sm);
}

// Zero the fill rows 0..tw-1 and ku+1..ku+tw of every column.
template <typename T>
__global__ void zero_fill_kernel(T* __restrict__ band, long long n, long long ldab, int tw, int ku) {
    const long long total = n * (2LL * tw);
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        long long j = e / (2 * tw);
        int q = (int)(e % (2 * tw));
        int row = (q < tw) ? q : ku + 1 + (q - tw);
        band[row + j * ldab] = T(0);
    }
}

// d_i = A(i, i), e_i = A(i, i+1).
template <typename T>
__global__ void extract_kernel(const T* __restrict__ band, long long n, long long ldab, int ku,
                               T* __restrict__ d, T* __restrict__ e) {
    const long long stride = ldab - 1;
    const T* base = band + ku;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        d[i] = base[i + i * stride];
        if (i + 1 < n) e[i] = base[i + (i + 1) * stride];
    }
}

}  // namespace bb
