// Group scheduler: one CTA runs g consecutive sweeps of a pass in lockstep,
// with every band column they touch held in shared memory.
//
// Within a group, sweep jj (= r - r0) runs half-step h = tau - L * jj at tick
// tau, L being the same half-step lag as the progress protocol of the
// persistent scheduler (2, 3 or 4).  Half-steps of one tick touch disjoint
// windows and overlapping half-steps of different sweeps run in sweep order
// (exhaustive check of the lockstep schedule), so a tick is one CTA barrier.
// Each sweep of the group is run by one warp.
//
// Between groups, whole columns change hands.  A group keeps the columns
// [A, B] of the band in a circular buffer of shared memory: a column is
// copied in (all b + 2t + 1 rows of the pass) the first time the group needs
// it, and written back once no sweep of the group will touch it again.  A
// group publishes its watermark A, the first column it may still touch; the
// next group copies a column in only when the previous group's watermark is
// beyond it, so at any time each column belongs to at most one group, and
// the groups touch every column in sweep order.  Writing back whole columns
// (rows no sweep of the pass touches included) is therefore safe.
//
// The method is that of "Accelerating Bidiagonalization of Banded Matrices
// through Memory-Aware Bulge-Chasing on GPUs" (arXiv 2510.12705), Section III;
// the grouping of sweeps per CTA and the column hand-over are this library's.
#pragma once

#include "bb_device.cuh"

namespace bb {

struct GroupArgs {
    int g;        // sweeps per group
    int ngroups;  // ceil(nsweeps / g)
    int nslot;    // columns of the circular buffer
    int lds;      // shared-memory stride between buffered columns (even)
};

// Last column touched by half-step h (right: 2k, left: 2k+1) of sweep r.
__device__ __forceinline__ long long half_max_col(const PassArgs& P, int r, int h) {
    const StepGeom g = step_geom(P, r, h >> 1);
    return (h & 1) ? g.cend : g.ce;
}
// First column of the window of half-step h of sweep r.
__device__ __forceinline__ long long half_min_col(const PassArgs& P, int r, int h) {
    return (long long)r + P.bp + (long long)(h >> 1) * P.b;
}

// Accessor of the buffered band: A(i, j) of the pass lives at
// cols[slot(j) * lds + (i - j + b + t)], slot(j) = j mod nslot.
template <typename T>
struct ColBuf {
    T* cols;
    int nslot, lds, off;  // off = b + t
    __device__ __forceinline__ int slot(long long j) const { return (int)j % nslot; }
    __device__ __forceinline__ T* col(long long j) const { return cols + (size_t)slot(j) * lds; }
};

// Copy columns [j0, j1] (rows ku-b-t .. ku+t of the pass) between memory and
// the buffer.  Element e of a chunk of columns -> (column e / ld, row e % ld),
// so consecutive threads touch consecutive rows of a column.
template <typename T, bool LOAD>
__device__ __forceinline__ void move_cols(T* __restrict__ band, const PassArgs& P, const ColBuf<T>& cb,
                                          long long j0, long long j1) {
    if (j1 < j0) return;
    const int ld = P.b + 2 * P.t + 1;
    const long long top = (long long)P.ku - P.b - P.t;
    const unsigned magic = 0xffffffffu / (unsigned)ld + 1u;  // e / ld for e < 2^16
    const int chunk = 65535 / ld;                            // columns per chunk
    for (long long jc = j0; jc <= j1; jc += chunk) {
        const int ncols = (int)min((long long)chunk, j1 - jc + 1);
        const int total = ncols * ld;
        const int s0 = cb.slot(jc);
        const T* gsrc = band + jc * P.ldab + top;
        for (int e = threadIdx.x; e < total; e += blockDim.x) {
            const int jj = (int)__umulhi((unsigned)e, magic);
            const int row = e - jj * ld;
            int sl = s0 + jj;
            if (sl >= cb.nslot) sl -= cb.nslot;
            T* sm = cb.cols + (size_t)sl * cb.lds + row;
            T* gm = const_cast<T*>(gsrc) + (long long)jj * P.ldab + row;
            if (LOAD) cp_async_elem<T>(sm, gm);
            else *gm = *sm;
        }
    }
}

// Right half-step of sweep r, step k on the buffered band, by one warp.
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void group_right(const PassArgs& P, const ColBuf<T>& cb, int r, int k, T* vb,
                                            T* taub) {
    constexpr int NPL = (WMAX + 31) / 32;
    const StepGeom g = step_geom(P, r, k);
    const int W = FULL ? WMAX : g.w;
    const int lane = threadIdx.x & 31;
    const int off = cb.off;
    T xp[NPL];
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        xp[q] = (m < W) ? cb.col(g.c + m)[g.p - (g.c + m) + off] : T(0);
    }
    T beta = warp_larfg<T, NPL>(xp, W, lane, vb, taub);
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        if (m < W) cb.col(g.c + m)[g.p - (g.c + m) + off] = (m == 0) ? beta : T(0);
    }
    __syncwarp();
    const T tau = *taub;
    if (tau == T(0)) return;
    // A(i, c+m) = cb.cols[idx[m] + (i - p)] with idx[m] = slot(c+m) lds + off + p - (c+m)
    int idx[WMAX];
    {
        int s = cb.slot(g.c);
#pragma unroll
        for (int m = 0; m < WMAX; ++m) {
            if (m < W) idx[m] = s * cb.lds + off + (int)(g.p - (g.c + m));
            s = (s + 1 == cb.nslot) ? 0 : s + 1;
        }
    }
    const int nrows = (int)(g.ce - g.p);
    for (int i = 1 + lane; i <= nrows; i += 32) {
        T x[WMAX];
        T y = 0;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) {
                x[m] = cb.cols[idx[m] + i];
                y = fma(x[m], vb[m], y);
            }
        const T s = tau * y;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) cb.cols[idx[m] + i] = fma(-s, vb[m], x[m]);
    }
}

// Left half-step of sweep r, step k on the buffered band, by one warp.
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void group_left(const PassArgs& P, const ColBuf<T>& cb, int r, int k, T* vb,
                                           T* taub) {
    constexpr int NPL = (WMAX + 31) / 32;
    const StepGeom g = step_geom(P, r, k);
    const int W = FULL ? WMAX : g.w;
    const int lane = threadIdx.x & 31;
    const int off = cb.off;
    T* colc = cb.col(g.c) + off;  // colc[m] = A(c + m, c)
    T xc[NPL];
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        xc[q] = (m < W) ? colc[m] : T(0);
    }
    T beta = warp_larfg<T, NPL>(xc, W, lane, vb, taub);
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        if (m < W) colc[m] = (m == 0) ? beta : T(0);
    }
    __syncwarp();
    const T tau = *taub;
    if (tau == T(0)) return;
    for (long long j = g.c + 1 + lane; j <= g.cend; j += 32) {
        T* cj = cb.col(j) + off + (g.c - j);  // cj[m] = A(c + m, j)
        T x[WMAX];
        T y = 0;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) {
                x[m] = cj[m];
                y = fma(vb[m], x[m], y);
            }
        const T s = tau * y;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) cj[m] = fma(-s, vb[m], x[m]);
    }
}

template <typename T, int WMAX>
__device__ __forceinline__ void group_half(const PassArgs& P, const ColBuf<T>& cb, int r, int h, T* vb, T* taub) {
    const int k = h >> 1;
    const bool full = step_geom(P, r, k).w == WMAX;
    if ((h & 1) == 0) {
        if (full) group_right<T, WMAX, true>(P, cb, r, k, vb, taub);
        else group_right<T, WMAX, false>(P, cb, r, k, vb, taub);
    } else {
        if (full) group_left<T, WMAX, true>(P, cb, r, k, vb, taub);
        else group_left<T, WMAX, false>(P, cb, r, k, vb, taub);
    }
}

// Warps (= sweeps per group) a group CTA may have: a lane holds one row or
// column of WMAX entries plus WMAX buffer offsets.
template <typename T, int WMAX>
struct GroupMaxWarps {
    static constexpr int value = (WMAX * sizeof(T) <= 17 * 4) ? 16 : 8;
};

// Persistent group kernel: CTAs take groups G = blockIdx.x, + gridDim.x, ...
// in order; blockDim.x = 32 * g.  wm[G] is group G's watermark.
template <typename T, int WMAX>
__global__ void __launch_bounds__(32 * GroupMaxWarps<T, WMAX>::value)
pass_group_kernel(T* __restrict__ band, PassArgs P, GroupArgs GA, int* __restrict__ wm,
                  int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_flag;
    T* vbuf = reinterpret_cast<T*>(smem_raw);          // [g][WMAX]
    T* taubuf = vbuf + (size_t)GA.g * WMAX;             // [g]
    ColBuf<T> cb;
    cb.cols = taubuf + ((GA.g + 1) & ~1);
    cb.nslot = GA.nslot;
    cb.lds = GA.lds;
    cb.off = P.b + P.t;
    const int warp = threadIdx.x >> 5;
    const int L = P.lagh;
    __shared__ int s_nsteps[32];  // steps of each sweep of the group
    // one read of the status word for the whole CTA, so that all threads agree
    if (threadIdx.x == 0) s_flag = ld_relaxed_gpu(status);
    __syncthreads();
    if (s_flag != kStatusOk) return;
    for (int G = blockIdx.x; G < GA.ngroups; G += gridDim.x) {
        const int r0 = G * GA.g;
        const int ng = min(GA.g, P.nsweeps - r0);
        __syncthreads();
        if ((int)threadIdx.x < ng) s_nsteps[threadIdx.x] = sweep_steps(P, r0 + threadIdx.x);
        __syncthreads();
        int tend = 0;
        for (int jj = 0; jj < ng; ++jj) tend = max(tend, L * jj + 2 * s_nsteps[jj]);
        // fault injection: the group holding the stalled sweep never publishes
        const bool publish = !(P.stall_sweep >= r0 && P.stall_sweep < r0 + ng);
        long long A = (long long)r0 + P.bp;  // first column the group may still touch
        long long B = A - 1;                 // last column in the buffer
        int pending = -1;                    // watermark written back, not yet published
        for (int tau = 0; tau < tend; ++tau) {
            // columns this tick needs
            long long xneed = -1;
            for (int jj = 0; jj < ng; ++jj) {
                const int h = tau - L * jj;
                if (h >= 0 && h < 2 * s_nsteps[jj]) xneed = max(xneed, half_max_col(P, r0 + jj, h));
            }
            if (xneed > B) {
                if (xneed - A + 1 > GA.nslot) {  // buffer too small: host sizing error
                    if (threadIdx.x == 0) atomicCAS(status, kStatusOk, kStatusInternal);
                    return;
                }
                if (G > 0 && !block_wait(wm + G - 1, (int)(xneed + 1), status, P, &s_flag)) return;
                move_cols<T, true>(band, P, cb, B + 1, xneed);
                B = xneed;
            }
            cp_async_commit();
            cp_async_wait_all();
            __syncthreads();
            if (warp < ng) {
                const int h = tau - L * warp;
                if (h >= 0 && h < 2 * s_nsteps[warp])
                    group_half<T, WMAX>(P, cb, r0 + warp, h, vbuf + (size_t)warp * WMAX, taubuf + warp);
            }
            __syncthreads();
            // publish the previous tick's watermark: its columns were stored
            // before this tick's barriers, so the fence finds them done
            if (pending >= 0) {
                if (threadIdx.x == 0 && publish) {
                    __threadfence();
                    st_release_gpu(wm + G, pending);
                }
                pending = -1;
            }
            // new watermark: first column of the next half-step of any unfinished sweep
            long long anew = B + 1;
            if (tau < tend - 1) {
                for (int jj = 0; jj < ng; ++jj) {
                    const int h = tau + 1 - L * jj;
                    if (h < 2 * s_nsteps[jj]) anew = min(anew, half_min_col(P, r0 + jj, max(h, 0)));
                }
            }
            if (anew > A) {
                move_cols<T, false>(band, P, cb, A, anew - 1);
                A = anew;
                pending = (int)min(A, (long long)P.n);
            }
        }
        if (pending >= 0) block_publish_if(wm + G, pending, publish);
        __syncthreads();
    }
}

}  // namespace bb
