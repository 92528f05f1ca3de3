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

constexpr int kPublishEvery = 4;  // ticks between two publications of a group's watermark

struct GroupArgs {
    int g;        // sweeps per group
    int ngroups;  // ceil(nsweeps / g)
    int nslot;    // columns of the circular buffer
    int lds;      // shared-memory stride between buffered columns (even)
    int ahead;    // ticks the loader may run ahead of the storer (1 .. kMaxStages - 2)
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

// Warps a group CTA may have (its sweeps plus the loader and the storer): a
// lane holds one row or column of WMAX entries plus WMAX buffer offsets.
template <typename T, int WMAX>
struct GroupMaxWarps {
    static constexpr int value = (WMAX * sizeof(T) <= 17 * 4) ? 16 : 8;
};

// ---------------------------------------------------------------------------
// Shared-memory synchronisation of the group pipeline.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}
// Arrives once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void mbar_arrive_cp_async(unsigned long long* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of parity `parity` of *bar; false on giving up
// (after `budget` SM clock cycles, or when *abort_tick <= tick).
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity, unsigned long long budget,
                                          const volatile int* abort_tick, int tick) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    for (unsigned it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_tick <= tick) return false;
            if ((unsigned long long)(clock64() - t0) > budget) return false;
        }
    }
}
__device__ __forceinline__ int ld_acquire_cta_shared(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_cta_shared(int* p, int v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warp-wide wait until *flag >= target (lane 0 spins; `seen` caches the
// largest value lane 0 has acquired, so a column range already released
// costs no memory round trip).  Bounded like block_wait; false on timeout or
// when another CTA has latched an error.
__device__ __forceinline__ bool warp_wait(const int* flag, int target, int* status, const PassArgs& P,
                                          int& seen) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0 && seen < target) {
        int v = ld_acquire_gpu(flag);
        if (v < target) {
            const long long t0 = clock64();
            unsigned int it = 0;
            for (;;) {
                v = ld_relaxed_gpu(flag);
                if (v >= target) break;
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
            // the value seen is final (watermarks only grow): one acquire load
            // orders the copies that follow after the producer's stores
            if (ok) v = ld_acquire_gpu(flag);
        }
        if (ok) seen = v;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Columns [j0, j1] between memory and the buffer, by one warp.
template <typename T, bool LOAD>
__device__ __forceinline__ void warp_move_cols(T* __restrict__ band, const PassArgs& P, const ColBuf<T>& cb,
                                               long long j0, long long j1) {
    if (j1 < j0) return;
    const int ld = P.b + 2 * P.t + 1;
    const long long top = (long long)P.ku - P.b - P.t;
    const int lane = threadIdx.x & 31;
    int sl = cb.slot(j0);
    for (long long j = j0; j <= j1; ++j) {
        T* sm = cb.cols + (size_t)sl * cb.lds;
        T* gm = band + j * P.ldab + top;
        for (int row = lane; row < ld; row += 32) {
            if (LOAD) cp_async_elem<T>(sm + row, gm + row);
            else gm[row] = sm[row];
        }
        sl = (sl + 1 == cb.nslot) ? 0 : sl + 1;
    }
}

// Last column ticks <= ... touch, one sweep per lane: max over the group's
// sweeps active at tick u of the last column of their half-step.
__device__ __forceinline__ long long tick_max_col(const PassArgs& P, int r0, int ng, int L, const int* nsteps,
                                                  int u) {
    long long x = -1;
    for (int jj = threadIdx.x & 31; jj < ng; jj += 32) {
        const int h = u - L * jj;
        if (h >= 0 && h < 2 * nsteps[jj]) x = max(x, half_max_col(P, r0 + jj, h));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
// First column any tick >= u touches (n when none does).
__device__ __forceinline__ long long tick_min_col(const PassArgs& P, int r0, int ng, int L, const int* nsteps,
                                                  int u) {
    long long a = P.n;
    for (int jj = threadIdx.x & 31; jj < ng; jj += 32) {
        const int h = u - L * jj;
        if (h < 2 * nsteps[jj]) a = min(a, half_min_col(P, r0 + jj, max(h, 0)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
    return a;
}

constexpr int kMaxStages = 8;

// Persistent group kernel: CTAs take groups G = blockIdx.x, + gridDim.x, ...
// in order; blockDim.x = 32 * (g + 2).  Warp jj < g runs sweep r0 + jj, one
// half-step per tick, the g warps meeting at a named barrier after each
// tick.  Warp g (the loader) copies in the columns tick u first needs, once
// group G - 1's watermark is beyond them and the storer has freed their
// slots, and signals full[u mod S] when the copies have landed.  Warp g + 1
// (the storer) waits for done[v mod S] (tick v computed), writes back the
// columns no later tick touches, frees their slots and, every few ticks,
// publishes the group's watermark (the first column the group may still
// touch) with a gpu-scope fence.  The loader runs at most `ahead` ticks
// ahead of the storer, S = ahead + 2 stages, so no mbarrier phase is
// overtaken.  Copies, write-backs and fences thus overlap the computation.
// Every wait is bounded; on giving up the CTA latches an error and all its
// warps leave at the same tick.
template <typename T, int WMAX>
__global__ void __launch_bounds__(32 * GroupMaxWarps<T, WMAX>::value)
pass_group_kernel(T* __restrict__ band, PassArgs P, GroupArgs GA, int* __restrict__ wm,
                  int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_flag;
    __shared__ int s_nsteps[32];  // steps of each sweep of the group
    __shared__ __align__(8) unsigned long long s_full[kMaxStages], s_done[kMaxStages];
    __shared__ int s_freed;       // storer: columns < s_freed are written back
    __shared__ int s_retired;     // storer: last tick whose columns it retired
    __shared__ volatile int s_abort_tick;  // first tick the CTA does not run
    __shared__ int s_dead;        // a compute warp gave up waiting
    T* vbuf = reinterpret_cast<T*>(smem_raw);  // [g][WMAX]
    T* taubuf = vbuf + (size_t)GA.g * WMAX;    // [g]
    ColBuf<T> cb;
    cb.cols = taubuf + ((GA.g + 1) & ~1);
    cb.nslot = GA.nslot;
    cb.lds = GA.lds;
    cb.off = P.b + P.t;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int L = P.lagh;
    const int S = GA.ahead + 2;
    const unsigned long long inner_budget = 2 * P.wait_budget + (1ull << 24);
    if (threadIdx.x == 0) {
        s_flag = ld_relaxed_gpu(status);
        for (int s = 0; s < S; ++s) {
            mbar_init(&s_full[s], 32);
            mbar_init(&s_done[s], 1);
        }
        s_abort_tick = 0x7fffffff;
        s_dead = 0;
    }
    __syncthreads();
    if (s_flag != kStatusOk) return;
    unsigned T0 = 0;  // ticks of earlier groups (mbarrier phases already used)
    for (int G = blockIdx.x; G < GA.ngroups; G += gridDim.x) {
        const int r0 = G * GA.g;
        const int ng = min(GA.g, P.nsweeps - r0);
        __syncthreads();
        if ((int)threadIdx.x < ng) s_nsteps[threadIdx.x] = sweep_steps(P, r0 + threadIdx.x);
        if (threadIdx.x == 0) {
            s_freed = r0 + P.bp;
            s_retired = -1;
        }
        __syncthreads();
        int tend = 0;
        for (int jj = 0; jj < ng; ++jj) tend = max(tend, L * jj + 2 * s_nsteps[jj]);
        if (warp < GA.g) {
            // ---- compute warps ----
            const int my_h_end = (warp < ng) ? 2 * s_nsteps[warp] : 0;
            for (int tau = 0; tau < tend; ++tau) {
                const unsigned q = T0 + (unsigned)tau;
                if (!mbar_wait(&s_full[q % S], (q / S) & 1u, inner_budget, &s_abort_tick, tau)) {
                    if (s_abort_tick > tau) {  // no abort announced: a lost signal
                        atomicCAS(status, kStatusOk, kStatusInternal);
                        s_dead = 1;
                    }
                }
                if (s_abort_tick <= tau) return;  // same tick for every compute warp
                const int h = tau - L * warp;
                if (!s_dead && h >= 0 && h < my_h_end)
                    group_half<T, WMAX>(P, cb, r0 + warp, h, vbuf + (size_t)warp * WMAX, taubuf + warp);
                named_bar_sync(1, 32 * GA.g);
                if (s_dead) return;
                if (threadIdx.x == 0) mbar_arrive(&s_done[q % S]);
            }
        } else if (warp == GA.g) {
            // ---- loader ----
            long long B = (long long)r0 + P.bp - 1;  // last column copied in
            int seen = (G == 0) ? 0x7fffffff : -1;
            for (int u = 0; u < tend; ++u) {
                const unsigned q = T0 + (unsigned)u;
                bool ok = true;
                // stay within `ahead` ticks of the storer (mbarrier phases)
                if (u - GA.ahead - 1 >= 0) {
                    const long long t0 = clock64();
                    while (ld_acquire_cta_shared(&s_retired) < u - GA.ahead - 1) {
                        if ((unsigned long long)(clock64() - t0) > inner_budget || s_dead) { ok = false; break; }
                    }
                }
                const long long xn = ok ? tick_max_col(P, r0, ng, L, s_nsteps, u) : -1;
                if (ok && xn > B) {
                    // slots of the columns xn - nslot + 1 .. xn must be free
                    const long long t0 = clock64();
                    while ((long long)ld_acquire_cta_shared(&s_freed) < xn - GA.nslot + 1) {
                        if ((unsigned long long)(clock64() - t0) > inner_budget || s_dead) { ok = false; break; }
                    }
                    if (ok && G > 0) ok = warp_wait(wm + G - 1, (int)(xn + 1), status, P, seen);
                    if (ok) {
                        warp_move_cols<T, true>(band, P, cb, B + 1, xn);
                        B = xn;
                    }
                }
                if (!ok) {
                    if (lane == 0) {
                        atomicCAS(status, kStatusOk, kStatusTimeout);
                        s_abort_tick = u;
                    }
                    cp_async_wait_all();
                    __syncwarp();
                    mbar_arrive(&s_full[q % S]);  // every lane: completes the phase
                    return;
                }
                mbar_arrive_cp_async(&s_full[q % S]);
            }
            cp_async_wait_all();
        } else {
            // ---- storer ----
            long long A = (long long)r0 + P.bp;  // first column not yet written back
            long long xr = -1;                   // last column ticks <= v touch
            int published = -1;
            for (int v = 0; v < tend; ++v) {
                const unsigned q = T0 + (unsigned)v;
                if (!mbar_wait(&s_done[q % S], (q / S) & 1u, inner_budget, &s_abort_tick, v)) {
                    if (lane == 0 && s_abort_tick > v) {  // no abort announced: a lost signal
                        atomicCAS(status, kStatusOk, kStatusInternal);
                        s_dead = 1;
                    }
                    return;
                }
                xr = max(xr, tick_max_col(P, r0, ng, L, s_nsteps, v));
                long long an = (v == tend - 1) ? (long long)P.n : tick_min_col(P, r0, ng, L, s_nsteps, v + 1);
                an = min(an, xr + 1);
                if (an > A) {
                    warp_move_cols<T, false>(band, P, cb, A, an - 1);
                    A = an;
                }
                __syncwarp();
                if (lane == 0) {
                    st_release_cta_shared(&s_freed, (int)A);
                    st_release_cta_shared(&s_retired, v);
                    const bool last = v == tend - 1;
                    if ((last || (v % kPublishEvery) == kPublishEvery - 1) && (int)A > published) {
                        published = (int)min(A, (long long)P.n);
                        if (P.stall_sweep < r0 || P.stall_sweep >= r0 + ng) {
                            __threadfence();
                            st_release_gpu(wm + G, published);
                        }
                    }
                }
            }
        }
        T0 += (unsigned)tend;
        __syncthreads();
    }
}

}  // namespace bb
