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
//     (see pass_lag_half in bb_plan.cu).
// The Householder reflector uses the LAPACK xLARFG convention.
//
// Band storage: A(i, j) = band[(ku + i - j) + j * ldab], so with
// base = band + ku and stride = ldab - 1, A(i, j) = base[i + j * stride]:
// a row of the matrix is strided by ldab - 1, a column is contiguous.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bb {

enum : int { kStatusOk = 0, kStatusTimeout = 5, kStatusInternal = 7 };

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
    // Reflector record for the back-transformation (rec_v == nullptr: none).
    // Reflector (sweep r, step k, side 0 right / 1 left) of this pass goes to
    // index rec_base + 2 (rec_prefix[r] + k) + side: v in rec_v[index *
    // rec_stride ..] (v_0 = 1), tau in rec_tau[index].  rec_prefix[r] = the
    // steps of the sweeps before r in this pass.
    void* rec_v = nullptr;
    void* rec_tau = nullptr;
    const long long* rec_prefix = nullptr;
    long long rec_base = 0;
    int rec_stride = 0;
};

// Records the reflector warp_larfg just built (s_v, s_tau) when the pass
// keeps a record; called by the warp that built it.  Lane m wrote s_v[m]
// itself and lane 0 the scalar, so no synchronisation is needed.
template <typename T>
__device__ __forceinline__ void record_reflector(const PassArgs& P, long long r, int k, int side, int W,
                                                 const T* s_v, const T* s_tau, int lane) {
    if (P.rec_v == nullptr) return;
    const long long idx = P.rec_base + 2 * (P.rec_prefix[r] + k) + side;
    T* v = static_cast<T*>(P.rec_v) + idx * P.rec_stride;
    for (int m = lane; m < W; m += 32) v[m] = s_v[m];
    if (lane == 0) static_cast<T*>(P.rec_tau)[idx] = *s_tau;
}

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

// Explicit shared-memory accesses by shared-window address.  A pointer into
// dynamic shared memory that travels through a struct or a function argument
// may compile to generic loads and stores; these always compile to
// ld/st.shared and use 32-bit addresses.  They are volatile so that they keep
// their program order with respect to each other and to the barriers around
// them.
__device__ __forceinline__ unsigned sh_addr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
template <typename T>
__device__ __forceinline__ T sh_ld(unsigned a);
template <>
__device__ __forceinline__ float sh_ld<float>(unsigned a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
template <>
__device__ __forceinline__ double sh_ld<double>(unsigned a) {
    double v;
    asm volatile("ld.shared.f64 %0, [%1];" : "=d"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sh_st(unsigned a, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void sh_st(unsigned a, double v) {
    asm volatile("st.shared.f64 [%0], %1;" ::"r"(a), "d"(v) : "memory");
}
// 16 bytes from a 16-byte aligned shared address
__device__ __forceinline__ void sh_ld16(unsigned a, float (&v)[4]) {
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(a));
}
__device__ __forceinline__ void sh_ld16(unsigned a, double (&v)[2]) {
    asm volatile("ld.shared.v2.f64 {%0, %1}, [%2];" : "=d"(v[0]), "=d"(v[1]) : "r"(a));
}

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
    // Fast path: the plain sum of squares is in range, so
    // beta = -sign(alpha) sqrt(alpha^2 + ||x||^2) with one square root (the
    // same norm as below up to rounding; beta then exceeds safmin).
    {
        T ss = 0;
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            if (m >= 1 && m < w) ss = fma(x[q], x[q], ss);
        }
        ss = warp_sum(ss);
        const T s2 = fma(alpha, alpha, ss);
        if (w > 1 && isfinite(s2) && ss >= Lim<T>::min_normal()) {
            const T nrm = dev_sqrt(s2);
            const T beta = (alpha >= T(0)) ? -nrm : nrm;
            const T tau = (beta - alpha) / beta;
            const T scal = T(1) / (alpha - beta);
#pragma unroll
            for (int q = 0; q < NPL; ++q) {
                const int m = lane + 32 * q;
                if (m < w) s_v[m] = (m == 0) ? T(1) : x[q] * scal;
            }
            if (lane == 0) *s_tau = tau;
            return beta;
        }
    }
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

// Applies that stream each row (column) through shared memory twice (dot
// product, then update) instead of holding it in registers: the kernels
// with reflectors of 256 bytes or more (32 and 33 doubles), which otherwise
// run out of registers and spill the row to local memory.  The arithmetic
// and its order are the same either way.
template <typename T, int WMAX>
constexpr bool kStreamApply = WMAX * sizeof(T) >= 256;

// Shared-memory layout of one CTA (ncolmax = b + t + 1 of the pass).
//   v[WMAX]              reflector of the current half-step
//   tau                  its scalar
//   tile[ncolmax][WP]    the column block of the left half-step: rows c..ce of
//                        columns c..cend, column-major with odd column stride WP
//   rtile[ncolmax-1][WP] the row block of the right half-step: rows p+1..ce of
//                        columns c..ce, row-major with odd row stride WP
template <typename T>
struct Smem {
    T* v;
    T* tau;
    T* tile;
    T* rtile;
    int wp;
};

template <typename T, int WMAX>
__device__ __forceinline__ Smem<T> carve_smem(unsigned char* raw, int ncolmax) {
    Smem<T> s;
    T* p = reinterpret_cast<T*>(raw);
    s.wp = WMAX | 1;
    s.v = p;
    s.tau = p + WMAX;
    s.tile = p + WMAX + 2;
    s.rtile = s.tile + (size_t)ncolmax * s.wp;
    return s;
}

// Asynchronous 4- or 8-byte copy global -> shared (no register staging); the
// copies a thread issued are complete after cp_async_wait_all().
template <typename T>
__device__ __forceinline__ void cp_async_elem(T* smem_dst, const T* gsrc) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(d), "l"(gsrc), "n"(sizeof(T))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Geometry of step k of sweep r (pass (b, t), b' = b - t):
//   c = r + b' + k b, p = r (k = 0) or c - b, ce = min(c + t, n-1),
//   cend = min(ce + b, n-1); right block rows p..ce x cols c..ce, left block
//   rows c..ce x cols c..cend.
struct StepGeom {
    long long c, p, ce, cend;
    int w;      // ce - c + 1: reflector length
    int nrows;  // ce - p: rows p+1..ce of the right apply
    int ncol;   // cend - c + 1: columns of the left block
};

__device__ __forceinline__ StepGeom step_geom(const PassArgs& P, int r, int k) {
    StepGeom g;
    g.c = (long long)r + P.bp + (long long)k * P.b;
    g.p = (k == 0) ? (long long)r : g.c - P.b;
    g.ce = min(g.c + (long long)P.t, P.n - 1);
    g.cend = min(g.ce + (long long)P.b, P.n - 1);
    g.w = (int)(g.ce - g.c + 1);
    g.nrows = (int)(g.ce - g.p);
    g.ncol = (int)(g.cend - g.c + 1);
    return g;
}

// Rows of the right block (from row c - 1, or c + 1 on the last pass) and
// columns of the left block (from column c + b - 1, or c + b + 1) that the
// half-step awaited by the progress wait may still write.  Everything before
// them was last written by half-steps already known to be complete when the
// previous wait of the same sweep returned, so it may be read before the
// wait.  (Exhaustive check over all (n, b, t) with b < 26 of the half-step
// protocol; for b - t == 2 nothing is late and the rule is conservative.)
__device__ __forceinline__ long long late_row(const PassArgs& P, long long c) {
    return (P.lagh == 4) ? c + 1 : c - 1;
}
__device__ __forceinline__ long long late_col(const PassArgs& P, long long c) {
    return (P.lagh == 4) ? c + P.b + 1 : c + P.b - 1;
}

// ---------------------------------------------------------------------------
// Right (horizontal) half-step of sweep r, step k: reflector from row p over
// columns c..ce, applied from the right to rows p+1..ce.  Rows p+1..c-1 are
// stored; rows c..ce (the square the left half-step starts from) are left in
// the tile only and reach memory with the left half-step's block.  That is
// safe for the progress protocol: any later half-step that touches the square
// also touches the left half-step's block, so it already waits for the left
// half-step.
//
// Split in two around the progress wait.  right_pre (k >= 1): the reflector
// input, row p = c - b, is row 0 of the previous left block, still in the
// tile, so the reflector is built before the wait, and rows before late_row
// start copying into rtile.  right_post copies the late rows (or, for k = 0,
// everything after building the reflector from memory) and applies.
// ---------------------------------------------------------------------------

// Copy rows [i0, i1) (local: row p + 1 + i) of the right block into rtile.
// Row i is always copied by thread i mod blockDim.x, the thread that applies
// the reflector to it, so a thread needs only its own copies to be complete.
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void copy_rows(const T* __restrict__ base, long long stride, const StepGeom& g,
                                          int i0, int i1, const Smem<T>& sm) {
    const int W = FULL ? WMAX : g.w;
    const int nthr = blockDim.x;
    const int first = i0 + (((int)threadIdx.x - i0 % nthr) + nthr) % nthr;
    for (int i = first; i < i1; i += nthr) {
        const T* src = base + (g.p + 1 + i) + g.c * stride;
        T* dst = sm.rtile + i * sm.wp;
#pragma unroll
        for (int m = 0; m < WMAX; ++m) {
            if (m < W) cp_async_elem<T>(dst + m, src);
            src += stride;
        }
    }
}

template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ bool right_pre(T* __restrict__ band, const PassArgs& P, int r, int k,
                                          const Smem<T>& sm) {
    constexpr int NPL = (WMAX + 31) / 32;
    if (k == 0) return false;
    const StepGeom g = step_geom(P, r, k);
    const int W = FULL ? WMAX : g.w;
    const int lane = threadIdx.x & 31;
    const long long stride = P.ldab - 1;
    T* __restrict__ base = band + P.ku;
    const int i_late = (int)min((long long)g.nrows, max(0LL, late_row(P, g.c) - g.p - 1));
    copy_rows<T, WMAX, FULL>(base, stride, g, 0, i_late, sm);
    cp_async_commit();
    if (threadIdx.x < 32) {
        T xp[NPL];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            xp[q] = (m < W) ? sm.tile[(P.b + m) * sm.wp] : T(0);
        }
        T beta = warp_larfg<T, NPL>(xp, W, lane, sm.v, sm.tau);
        record_reflector<T>(P, r, k, 0, W, sm.v, sm.tau, lane);
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            if (m < W) base[g.p + (g.c + m) * stride] = (m == 0) ? beta : T(0);
        }
    }
    return true;
}

template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void right_post(T* __restrict__ band, const PassArgs& P, int r, int k,
                                           const Smem<T>& sm, bool pre) {
    constexpr int NPL = (WMAX + 31) / 32;
    const StepGeom g = step_geom(P, r, k);
    const int W = FULL ? WMAX : g.w;
    const long long stride = P.ldab - 1;
    T* __restrict__ base = band + P.ku;
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
    if (pre) {
        const int i_late = (int)min((long long)g.nrows, max(0LL, late_row(P, g.c) - g.p - 1));
        copy_rows<T, WMAX, FULL>(base, stride, g, i_late, g.nrows, sm);
    } else {
        copy_rows<T, WMAX, FULL>(base, stride, g, 0, g.nrows, sm);
        if (tid < 32) {
            T xp[NPL];
#pragma unroll
            for (int q = 0; q < NPL; ++q) {
                const int m = lane + 32 * q;
                xp[q] = (m < W) ? __ldcg(base + g.p + (g.c + m) * stride) : T(0);
            }
            T beta = warp_larfg<T, NPL>(xp, W, lane, sm.v, sm.tau);
            record_reflector<T>(P, r, k, 0, W, sm.v, sm.tau, lane);
#pragma unroll
            for (int q = 0; q < NPL; ++q) {
                const int m = lane + 32 * q;
                if (m < W) base[g.p + (g.c + m) * stride] = (m == 0) ? beta : T(0);
            }
        }
    }
    cp_async_commit();
    cp_async_wait_all();
    // With the reflector built before the wait (pre), every thread applies it
    // to the rows it copied itself: no barrier.  Otherwise warp 0 has just
    // built it.
    if (!pre) __syncthreads();
    const T tau = *sm.tau;
    const int row_c = (int)(g.c - g.p - 1);  // local index of row c
    for (int i = tid; i < g.nrows; i += nthr) {
        T x[WMAX];
        const T* src = sm.rtile + i * sm.wp;
        if constexpr (kStreamApply<T, WMAX>) {
            // dot product from shared memory, then each entry read again and
            // updated: the row is never held whole in registers
            T s = 0;
            if (tau != T(0)) {
                T y = 0;
#pragma unroll
                for (int m = 0; m < WMAX; ++m)
                    if (m < W) y = fma(src[m], sm.v[m], y);
                s = tau * y;
            }
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < W) x[m] = (tau != T(0)) ? fma(-s, sm.v[m], src[m]) : src[m];
        } else {
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < W) x[m] = src[m];
            if (tau != T(0)) {
                T y = 0;
#pragma unroll
                for (int m = 0; m < WMAX; ++m)
                    if (m < W) y = fma(x[m], sm.v[m], y);
                const T s = tau * y;
#pragma unroll
                for (int m = 0; m < WMAX; ++m)
                    if (m < W) x[m] = fma(-s, sm.v[m], x[m]);
            }
        }
        const int rr = i - row_c;  // row c + rr
        if (rr < 0) {
            T* dst = base + (g.p + 1 + i) + g.c * stride;
#pragma unroll
            for (int m = 0; m < WMAX; ++m) {
                if (m < W) *dst = x[m];
                dst += stride;
            }
        } else {
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < W) sm.tile[m * sm.wp + rr] = x[m];
        }
    }
}

// ---------------------------------------------------------------------------
// Left (vertical) half-step of sweep r, step k: reflector from column c over
// rows c..ce, applied from the left to columns c+1..cend.  The tile's first w
// columns hold rows c..ce of columns c..ce (left there by the right half-step
// of the same step).  left_pre builds the reflector from the tile and starts
// copying the columns before late_col; left_post copies the rest, applies and
// stores the whole block (columns c..cend, rows c..ce).
// ---------------------------------------------------------------------------

// Copy columns [j0, j1) (local indices) of rows c..ce of the left block from
// memory into the tile.  Thread t takes row m = t % w of columns
// j0 + t / w, + nct / w, ... (consecutive threads read consecutive
// addresses of a column), walking its column pointer by a fixed increment.
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void copy_columns(const T* __restrict__ base, long long stride, const StepGeom& g,
                                             int j0, int j1, const Smem<T>& sm) {
    const int w = FULL ? WMAX : g.w;
    if (j1 <= j0) return;
    const int nthr = blockDim.x;
    const int per = nthr / w;  // columns per round
    const int t = threadIdx.x;
    if (t >= per * w) return;
    const int m = t % w;
    int jl = j0 + t / w;
    const T* src = base + (g.c + m) + (g.c + jl) * stride;
    T* dst = sm.tile + jl * sm.wp + m;
    const long long sstep = (long long)per * stride;
    const int dstep = per * sm.wp;
    for (; jl < j1; jl += per) {
        cp_async_elem<T>(dst, src);
        src += sstep;
        dst += dstep;
    }
}

// after_barrier: a block barrier has followed right_post (the publication
// of the right half-step), so the square is in the tile already; the threads
// not busy with the fence start the column copies at once.
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void left_pre(T* __restrict__ band, const PassArgs& P, int r, int k,
                                         const Smem<T>& sm, bool after_barrier = false) {
    constexpr int NPL = (WMAX + 31) / 32;
    const StepGeom g = step_geom(P, r, k);
    const int W = FULL ? WMAX : g.w;
    const int lane = threadIdx.x & 31;
    const long long stride = P.ldab - 1;
    T* __restrict__ base = band + P.ku;
    if (!after_barrier) __syncthreads();  // the right half-step's rows are in the tile
    const int jlate = (int)min((long long)g.ncol, max((long long)W, late_col(P, g.c) - g.c));
    copy_columns<T, WMAX, FULL>(base, stride, g, W, jlate, sm);
    cp_async_commit();
    if (threadIdx.x < 32) {
        T xc[NPL];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            xc[q] = (m < W) ? sm.tile[m] : T(0);
        }
        T beta = warp_larfg<T, NPL>(xc, W, lane, sm.v, sm.tau);
        record_reflector<T>(P, r, k, 1, W, sm.v, sm.tau, lane);
        __syncwarp();
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            if (m < W) sm.tile[m] = (m == 0) ? beta : T(0);
        }
    }
}

template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void left_post(T* __restrict__ band, const PassArgs& P, int r, int k,
                                          const Smem<T>& sm) {
    const StepGeom g = step_geom(P, r, k);
    const int W = FULL ? WMAX : g.w;
    const int tid = threadIdx.x, nthr = blockDim.x;
    const long long stride = P.ldab - 1;
    T* __restrict__ base = band + P.ku;
    const int wp = sm.wp, w = W, ncol = g.ncol;
    const long long c = g.c;
    const int jlate = (int)min((long long)ncol, max((long long)w, late_col(P, c) - c));
    copy_columns<T, WMAX, FULL>(base, stride, g, jlate, ncol, sm);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    const T tau = *sm.tau;
    if (tau != T(0)) {
        for (int jl = 1 + tid; jl < ncol; jl += nthr) {
            T* col = sm.tile + jl * wp;
            if constexpr (kStreamApply<T, WMAX>) {
                T y = 0;
#pragma unroll
                for (int m = 0; m < WMAX; ++m)
                    if (m < w) y = fma(sm.v[m], col[m], y);
                const T s = tau * y;
#pragma unroll
                for (int m = 0; m < WMAX; ++m)
                    if (m < w) col[m] = fma(-s, sm.v[m], col[m]);
            } else {
                T x[WMAX];
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
    }
    __syncthreads();
    // Write the whole block back (columns c .. cend, rows c .. ce); thread t
    // takes row t % w of columns t / w, + nthr / w, ...
    const int per = nthr / w;
    if (tid < per * w) {
        const int m = tid % w;
        int jl = tid / w;
        T* dst = base + (c + m) + (c + jl) * stride;
        const T* src = sm.tile + jl * wp + m;
        const long long gstep = (long long)per * stride;
        const int sstep = per * wp;
        for (; jl < ncol; jl += per) {
            *dst = *src;
            dst += gstep;
            src += sstep;
        }
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
        // every poll is an acquire load, so the one that sees the target
        // already orders this block's later reads after the producer's writes
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
// stores are ordered before the flag by the barrier and the release store,
// which is cumulative over what the barrier ordered before it.  The first
// thread of the last warp releases, so warp 0 (which builds the next
// reflector) goes on at once.
__device__ __forceinline__ void block_publish(int* flag, int value) {
    __syncthreads();
    if (threadIdx.x == blockDim.x - 32) st_release_gpu(flag, value);
}

__device__ __forceinline__ void block_publish_if(int* flag, int value, bool publish) {
    if (publish) block_publish(flag, value);
    else __syncthreads();
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
    static constexpr int value = (WMAX * sizeof(T) <= 17 * 4) ? 512 : 256;
};

// One step (right then left half-step) of sweep r under the persistent
// scheduler; false if a wait gave up.
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ bool persistent_step(T* __restrict__ band, const PassArgs& P, int r, int k,
                                                int K, int Hprev, bool publish, int* __restrict__ progress,
                                                int* __restrict__ status, const Smem<T>& sm, int* s_flag) {
    const bool pre = right_pre<T, WMAX, FULL>(band, P, r, k, sm);
    // the wait's barrier (or this one for sweep 0) publishes warp 0's reflector
    if (r > 0) {
        if (!block_wait(progress + r - 1, min(2 * k + P.lagh, Hprev), status, P, s_flag)) return false;
    } else {
        __syncthreads();
    }
    right_post<T, WMAX, FULL>(band, P, r, k, sm, pre);
    block_publish_if(progress + r, 2 * k + 1, publish);
    left_pre<T, WMAX, FULL>(band, P, r, k, sm, true);
    if (r > 0 && !block_wait(progress + r - 1, min(2 * k + 1 + P.lagh, Hprev), status, P, s_flag))
        return false;
    left_post<T, WMAX, FULL>(band, P, r, k, sm);
    if (k == K - 1 && r > 0 && !block_wait(progress + r - 1, Hprev, status, P, s_flag)) return false;
    if (publish) block_publish(progress + r, 2 * k + 2);
    else __syncthreads();
    return true;
}

template <typename T, int WMAX>
__global__ void __launch_bounds__(MaxThreads<T, WMAX>::value)
pass_persistent_kernel(T* __restrict__ band, PassArgs P, int* __restrict__ progress,
                       int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_flag;
    const Smem<T> sm = carve_smem<T, WMAX>(smem_raw, P.b + P.t + 1);
    // one read of the status word for the whole CTA, so that all threads agree
    if (threadIdx.x == 0) s_flag = ld_relaxed_gpu(status);
    __syncthreads();
    if (s_flag != kStatusOk) return;
    for (int r = blockIdx.x; r < P.nsweeps; r += gridDim.x) {
        const int K = sweep_steps(P, r);
        const int Hprev = (r > 0) ? 2 * sweep_steps(P, r - 1) : 0;
        const bool publish = (r != P.stall_sweep);
        for (int k = 0; k < K; ++k) {
            const bool ok = (step_geom(P, r, k).w == WMAX)
                                ? persistent_step<T, WMAX, true>(band, P, r, k, K, Hprev, publish, progress,
                                                                 status, sm, &s_flag)
                                : persistent_step<T, WMAX, false>(band, P, r, k, K, Hprev, publish, progress,
                                                                  status, sm, &s_flag);
            if (!ok) return;
        }
    }
}

// Per-cycle scheduler (one launch per cycle): block b runs step
// k = cycle - lag * r of sweep r = r_first + b.  Steps in one cycle touch
// disjoint windows, and the launch boundary orders consecutive cycles.
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void cycle_step(T* __restrict__ band, const PassArgs& P, int r, int k,
                                           const Smem<T>& sm) {
    right_post<T, WMAX, FULL>(band, P, r, k, sm, false);
    left_pre<T, WMAX, FULL>(band, P, r, k, sm);
    left_post<T, WMAX, FULL>(band, P, r, k, sm);
}

template <typename T, int WMAX>
__global__ void __launch_bounds__(MaxThreads<T, WMAX>::value)
pass_cycle_kernel(T* __restrict__ band, PassArgs P, int cycle, int r_first) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const Smem<T> sm = carve_smem<T, WMAX>(smem_raw, P.b + P.t + 1);
    const int r = r_first + blockIdx.x;
    const int k = cycle - P.lag * r;
    if (step_geom(P, r, k).w == WMAX) cycle_step<T, WMAX, true>(band, P, r, k, sm);
    else cycle_step<T, WMAX, false>(band, P, r, k, sm);
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
