// Group scheduler: one CTA runs g consecutive sweeps of a pass in lockstep,
// with every band column they touch held in shared memory.
//
// Within a group, sweep jj (= r - r0) runs half-step h = tau - L * jj at tick
// tau, L being the same half-step lag as the progress protocol of the
// persistent scheduler (2, 3 or 4).  Half-steps of one tick touch disjoint
// windows and overlapping half-steps of different sweeps run in sweep order
// (exhaustive check of the lockstep schedule; for b - t = 1 a lag of 4 is
// also the least that works), so a tick is one barrier of the compute warps.
// Each sweep of the group is run by one warp.
//
// Between groups, whole columns change hands.  A group keeps the columns
// [A, B] of the band in a circular buffer of shared memory: a column is
// copied in (rows ku-b-t .. ku+t of the pass, rounded out to 16 bytes) the
// first time the group needs it, and written back once no sweep of the group
// will touch it again.  A
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

#include <cuda_fp16.h>

#include <type_traits>

#include "bb_device.cuh"

namespace bb {


struct GroupArgs {
    int g;        // sweeps per group
    int ngroups;  // ceil(nsweeps / g)
    int nslot;    // columns of the circular buffer
    int top;      // first band row a buffered column holds (a multiple of 16 bytes / element)
    int lds;      // rows a buffered column holds = stride between buffered columns
                  // (a multiple of 16 bytes / element, so lds - 1 is odd)
    int ahead;    // ticks the loader may run ahead of the storer (1 .. kMaxStages - 2)
    int bulk_store;  // 1: the storer writes columns back with bulk copies (wide
                     // columns); 0: with plain 16-byte copies (narrow columns)
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

// Accessor of the buffered band: A(i, j) lives at element
// slot(j) * lds + (i - j + off) of the buffer, slot(j) = j mod nslot,
// off = ku - top: buffered column j is band rows top .. top + lds - 1 of
// column j.  The compute warps address it by shared-window byte address
// (base); the loader and the storer use the generic pointer (cols).
template <typename T>
struct ColBuf {
    T* cols;
    unsigned base;  // shared-window address of cols
    int nslot, lds, off;
    __device__ __forceinline__ int slot(int j) const { return j % nslot; }
    __device__ __forceinline__ T* col(int j) const { return cols + slot(j) * lds; }
    __device__ __forceinline__ unsigned at(int idx) const { return base + (unsigned)idx * (unsigned)sizeof(T); }
};

// A buffered entry of storage type ST read as the arithmetic type T, and a
// T value rounded to ST and stored (ST = T, or binary16 with float
// arithmetic: round to nearest even).
template <typename T, typename ST>
__device__ __forceinline__ T sh_ld_as(unsigned a) {
    if constexpr (std::is_same<T, ST>::value) {
        return sh_ld<T>(a);
    } else {
        static_assert(std::is_same<ST, __half>::value && std::is_same<T, float>::value, "binary16 storage: float");
        unsigned short h;
        asm volatile("ld.shared.b16 %0, [%1];" : "=h"(h) : "r"(a));
        return __half2float(__ushort_as_half(h));
    }
}
template <typename ST, typename T>
__device__ __forceinline__ void sh_st_as(unsigned a, T v) {
    if constexpr (std::is_same<T, ST>::value) {
        sh_st(a, v);
    } else {
        static_assert(std::is_same<ST, __half>::value && std::is_same<T, float>::value, "binary16 storage: float");
        const unsigned short h = __half_as_ushort(__float2half_rn(v));
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(h) : "memory");
    }
}

// Geometry of step k of sweep r in 32-bit arithmetic (the group kernel runs
// only for n < 2^30): c, p, ce, cend and w as in step_geom.
struct GGeom {
    int c, p, ce, cend, w;
};
__device__ __forceinline__ GGeom gstep(const PassArgs& P, int r, int k) {
    GGeom g;
    const int n1 = (int)P.n - 1;
    g.c = r + P.bp + k * P.b;
    g.p = (k == 0) ? r : g.c - P.b;
    g.ce = min(g.c + P.t, n1);
    g.cend = min(g.ce + P.b, n1);
    g.w = g.ce - g.c + 1;
    return g;
}

// Each warp's reflector buffer is padded to a multiple of 16 bytes, so that
// the apply loads v into registers with 16-byte loads once per half-step.
__host__ __device__ constexpr int group_v_stride(int wmax, int elem) {
    return ((wmax * elem + 15) / 16 * 16) / elem;
}
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
    using type = float4;
};
template <>
struct Vec16<double> {
    using type = double2;
};
template <typename T, int WMAX>
__device__ __forceinline__ void load_v(unsigned v, T (&vr)[WMAX]) {
    constexpr int PER = 16 / (int)sizeof(T);
    constexpr int NV = (WMAX + PER - 1) / PER;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        T e[PER];
        sh_ld16(v + 16u * q, e);
#pragma unroll
        for (int u = 0; u < PER; ++u)
            if (q * PER + u < WMAX) vr[q * PER + u] = e[u];
    }
}

// Whether the applies hold v in registers: reflectors of up to 64 bytes, and
// 33 floats (those kernels run 8 warps with up to 255 registers); the others
// read it from shared memory.
template <typename T, int WMAX>
__host__ __device__ constexpr bool group_v_in_registers() {
    return WMAX * sizeof(T) <= 64 || (sizeof(T) == 4 && WMAX > 17 && WMAX <= 33);
}

// Right half-step (rows p..ce of columns c..ce) on the buffered band, by one
// warp: reflector from row p, then lane i applies it to rows p+1+i, +32, ...
// The half-step's columns span fewer than nslot slots, so a slot index past
// the end wraps with one subtraction.  T: arithmetic, ST: storage.
template <typename T, typename ST, int WMAX, bool FULL>
__device__ __forceinline__ void group_right(const ColBuf<ST>& cb, const GGeom& g, int s0, T* vb, T* taub) {
    constexpr int NPL = (WMAX + 31) / 32;
    constexpr unsigned S = sizeof(T), SB = sizeof(ST);
    const int W = FULL ? WMAX : g.w;
    const int lane = threadIdx.x & 31;
    // A(p + i, c + m) is element a0 + i + m (lds - 1) - (m >= mwrap ? nslot lds : 0):
    // column c + m sits in slot s0 + m, wrapped once past the end
    const int a0 = s0 * cb.lds + cb.off + (g.p - g.c);
    const int dm = cb.lds - 1;
    const int mwrap = cb.nslot - s0;
    const int wrap = cb.nslot * cb.lds;
    T xp[NPL];
    unsigned xa[NPL];
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        xa[q] = cb.at(a0 + m * dm - ((m >= mwrap) ? wrap : 0));
        xp[q] = (m < W) ? sh_ld_as<T, ST>(xa[q]) : T(0);
    }
    T beta = warp_larfg<T, NPL>(xp, W, lane, vb, taub);
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        if (m < W) sh_st_as<ST>(xa[q], (m == 0) ? beta : T(0));
    }
    __syncwarp();
    const T tau = sh_ld<T>(sh_addr(taub));
    if (tau == T(0)) return;
    // v in registers (16-byte loads, once per half-step) where the registers
    // allow; otherwise read from shared memory at each use
    constexpr bool kVReg = group_v_in_registers<T, WMAX>();
    const unsigned vaddr = sh_addr(vb);
    T vreg[kVReg ? WMAX : 1];
    if constexpr (kVReg) load_v<T, WMAX>(vaddr, vreg);
    auto v = [&](int m) -> T {
        if constexpr (kVReg) return vreg[m];
        else return sh_ld<T>(vaddr + S * (unsigned)m);
    };
    // byte offset of column c + m from column c, wrap included
    unsigned om[WMAX];
#pragma unroll
    for (int m = 0; m < WMAX; ++m) om[m] = SB * (unsigned)(m * dm - ((m >= mwrap) ? wrap : 0));
    const int nrows = g.ce - g.p;
    for (int i = 1 + lane; i <= nrows; i += 32) {
        const unsigned ra = cb.at(a0 + i);
        T x[WMAX];
        T y = 0;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) {
                x[m] = sh_ld_as<T, ST>(ra + om[m]);
                y = fma(x[m], v(m), y);
            }
        const T s = tau * y;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) sh_st_as<ST>(ra + om[m], fma(-s, v(m), x[m]));
    }
}

// Left half-step (rows c..ce of columns c..cend) on the buffered band, by
// one warp: reflector from column c, then lane i applies it to columns
// c+1+i, +32, ...
template <typename T, typename ST, int WMAX, bool FULL>
__device__ __forceinline__ void group_left(const ColBuf<ST>& cb, const GGeom& g, int s0, T* vb, T* taub) {
    constexpr int NPL = (WMAX + 31) / 32;
    constexpr unsigned S = sizeof(T), SB = sizeof(ST);
    const int W = FULL ? WMAX : g.w;
    const int lane = threadIdx.x & 31;
    const unsigned colc = cb.at(s0 * cb.lds + cb.off);  // colc + SB m = A(c + m, c)
    T xc[NPL];
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        xc[q] = (m < W) ? sh_ld_as<T, ST>(colc + SB * (unsigned)m) : T(0);
    }
    T beta = warp_larfg<T, NPL>(xc, W, lane, vb, taub);
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        if (m < W) sh_st_as<ST>(colc + SB * (unsigned)m, (m == 0) ? beta : T(0));
    }
    __syncwarp();
    const T tau = sh_ld<T>(sh_addr(taub));
    if (tau == T(0)) return;
    constexpr bool kVReg = group_v_in_registers<T, WMAX>();
    const unsigned vaddr = sh_addr(vb);
    T vreg[kVReg ? WMAX : 1];
    if constexpr (kVReg) load_v<T, WMAX>(vaddr, vreg);
    auto v = [&](int m) -> T {
        if constexpr (kVReg) return vreg[m];
        else return sh_ld<T>(vaddr + S * (unsigned)m);
    };
    for (int dj = 1 + lane; dj <= g.cend - g.c; dj += 32) {
        int sl = s0 + dj;
        if (sl >= cb.nslot) sl -= cb.nslot;
        const unsigned cj = cb.at(sl * cb.lds + cb.off - dj);  // cj + SB m = A(c + m, c + dj)
        T x[WMAX];
        T y = 0;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) {
                x[m] = sh_ld_as<T, ST>(cj + SB * (unsigned)m);
                y = fma(v(m), x[m], y);
            }
        const T s = tau * y;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) sh_st_as<ST>(cj + SB * (unsigned)m, fma(-s, v(m), x[m]));
    }
}

// The chase a group kernel runs.  A sweep is a sequence of units, kUnits
// per step; the lockstep lag (PassArgs::lagh) and the loader's and storer's
// column bookkeeping count units.  A chase provides the first and last band
// column unit h of sweep r touches (columns only move right as h grows), the
// unit itself on the buffered band by one warp, and kVecs, the reflector-sized
// vectors of shared scratch each warp needs.
//
// The bidiagonal chase: two units per step, the right half-step (rows p..ce
// of columns c..ce) and the left one (rows c..ce of columns c..cend).
struct BidiagChase {
    static constexpr int kUnits = 2;
    static constexpr int kVecs = 1;
    __device__ static long long max_col(const PassArgs& P, int r, int h) { return half_max_col(P, r, h); }
    __device__ static long long min_col(const PassArgs& P, int r, int h) { return half_min_col(P, r, h); }
    // slot: the buffer slot of column c of this half-step's step (the caller
    // carries it from step to step, sparing a modulo on the critical path).
    template <typename T, typename ST, int WMAX>
    __device__ static void unit(const PassArgs& P, const ColBuf<ST>& cb, int r, int h, int slot, T* vb, T* taub) {
        const GGeom g = gstep(P, r, h >> 1);
        const bool full = g.w == WMAX;
        if ((h & 1) == 0) {
            if (full) group_right<T, ST, WMAX, true>(cb, g, slot, vb, taub);
            else group_right<T, ST, WMAX, false>(cb, g, slot, vb, taub);
        } else {
            if (full) group_left<T, ST, WMAX, true>(cb, g, slot, vb, taub);
            else group_left<T, ST, WMAX, false>(cb, g, slot, vb, taub);
        }
    }
};

// Warps a group CTA may have (its sweeps plus the loader, the storer and the
// publisher): a
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
// (after `budget` SM clock cycles, when *abort_tick <= tick or when *dead).
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity, unsigned long long budget,
                                          const volatile int* abort_tick, int tick, const volatile int* dead) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    for (unsigned it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_tick <= tick || *dead) return false;
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
// Bulk (TMA) copies of one buffered column, 16-byte aligned on both sides.
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, unsigned bytes, unsigned long long* bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(smem_src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have read their shared-memory source
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// this thread's bulk stores but those of the most recent group are complete
__device__ __forceinline__ void bulk_wait_prev() { asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); }
// order this thread's generic-proxy accesses with later async-proxy (bulk
// copy) accesses of shared or global memory, and vice versa
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

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

// Last column ticks <= ... touch, one sweep per lane: max over the group's
// sweeps active at tick u of the last column of their unit.
template <class Chase>
__device__ __forceinline__ long long tick_max_col(const PassArgs& P, int r0, int ng, int L, const int* nsteps,
                                                  int u) {
    long long x = -1;
    for (int jj = threadIdx.x & 31; jj < ng; jj += 32) {
        const int h = u - L * jj;
        if (h >= 0 && h < Chase::kUnits * nsteps[jj]) x = max(x, Chase::max_col(P, r0 + jj, h));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
// First column any tick >= u touches (n when none does).
template <class Chase>
__device__ __forceinline__ long long tick_min_col(const PassArgs& P, int r0, int ng, int L, const int* nsteps,
                                                  int u) {
    long long a = P.n;
    for (int jj = threadIdx.x & 31; jj < ng; jj += 32) {
        const int h = u - L * jj;
        if (h < Chase::kUnits * nsteps[jj]) a = min(a, Chase::min_col(P, r0 + jj, max(h, 0)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
    return a;
}

constexpr int kMaxStages = 10;

// Shared memory of the group kernel: per-sweep scratch (nvec reflector-sized
// vectors) and scalars, then (16-byte aligned) the circular column buffer.
__host__ __device__ inline size_t group_cols_offset(int g, int wmax, size_t elem, int nvec = 1) {
    const size_t head =
        elem * ((size_t)g * nvec * group_v_stride(wmax, (int)elem) + (size_t)((g + 1) & ~1));
    return (head + 15) & ~(size_t)15;
}

// Persistent group kernel: CTAs take groups G = blockIdx.x, + gridDim.x, ...
// in order; blockDim.x = 32 * (g + 3).  Chase: the chase it runs (units,
// their columns and their arithmetic; BidiagChase above).  T: the arithmetic
// type, ST: the band's storage type (T, or binary16 with float arithmetic;
// columns are buffered as stored).
//   Warps jj < g run sweep r0 + jj, one unit per tick, and meet at a named
//   barrier after each tick.
//   Warp g (the loader) copies in the columns tick u first needs, one bulk
//   (TMA) copy per column, once group G - 1's watermark is beyond them and
//   the storer has freed their slots; full[u mod S] completes when the bytes
//   have landed.
//   Warp g + 1 (the storer) waits for done[v mod S] (tick v computed), writes
//   back the columns no later tick touches (bulk copies for wide columns,
//   plain 16-byte copies for narrow ones), frees their slots and reports the
//   written-back range in shared memory (bulk copies one tick later, once
//   they are complete).
//   Warp g + 2 (the publisher) turns that report into the group's watermark
//   (the first column the group may still touch) with a release store, so
//   its latency delays neither the storer nor the loader.
// The loader runs at most `ahead` ticks ahead of the storer and S = ahead + 2
// stages, so no mbarrier phase is overtaken.  Copies, write-backs and
// publication thus overlap the computation.  Every wait is bounded; on
// giving up the CTA latches an error, the compute warps leave their loop at
// the same tick, the other roles leave theirs, and the CTA returns after one
// last barrier.  Requires band, ldab * sizeof(ST) and top * sizeof(ST)
// 16-byte aligned and n < 2^30 (32-bit geometry).
template <typename T, int WMAX, class Chase = BidiagChase, typename ST = T>
__global__ void __launch_bounds__(32 * GroupMaxWarps<T, WMAX>::value)
pass_group_kernel(ST* __restrict__ band, PassArgs P, GroupArgs GA, int* __restrict__ wm,
                  int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_flag;
    __shared__ int s_nsteps[32];  // steps of each sweep of the group
    __shared__ __align__(8) unsigned long long s_full[kMaxStages], s_done[kMaxStages], s_stored[kMaxStages];
    __shared__ int s_freed;       // storer: columns < s_freed are written back
    __shared__ int s_retired;     // storer: last tick whose columns it retired
    __shared__ int s_written;     // storer: columns < s_written are written back and complete
    __shared__ volatile int s_abort_tick;  // first tick the CTA does not run
    __shared__ volatile int s_dead;  // a warp gave up waiting on a signal that never came
    constexpr int U = Chase::kUnits;
    constexpr int VS = Chase::kVecs * group_v_stride(WMAX, (int)sizeof(T));
    T* vbuf = reinterpret_cast<T*>(smem_raw);  // [g][VS], 16-byte aligned rows
    T* taubuf = vbuf + (size_t)GA.g * VS;      // [g]
    ColBuf<ST> cb;
    cb.cols = reinterpret_cast<ST*>(smem_raw + group_cols_offset(GA.g, WMAX, sizeof(T), Chase::kVecs));
    cb.base = sh_addr(cb.cols);
    cb.nslot = GA.nslot;
    cb.lds = GA.lds;
    cb.off = P.ku - GA.top;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int L = P.lagh;
    const int S = GA.ahead + 2;
    const unsigned col_bytes = (unsigned)(GA.lds * sizeof(ST));
    const unsigned long long inner_budget = 2 * P.wait_budget + (1ull << 24);
    if (threadIdx.x == 0) {
        s_flag = ld_relaxed_gpu(status);
        for (int s = 0; s < S; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_done[s], 1);
            mbar_init(&s_stored[s], 1);
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
            s_freed = (int)Chase::min_col(P, r0, 0);  // the group's first column
            s_retired = -1;
            s_written = -1;
        }
        __syncthreads();
        int tend = 0;
        for (int jj = 0; jj < ng; ++jj) tend = max(tend, L * jj + U * s_nsteps[jj]);
        if (warp < GA.g) {
            // ---- compute warps ----
            const int my_h_end = (warp < ng) ? U * s_nsteps[warp] : 0;
            // slot of column c of this warp's current step: one modulo per
            // group, then + b per step (one wrap when nslot > b, as the
            // footprint of a whole step gives; the loop keeps it exact anyway)
            int my_slot = -1;
            int stage = (int)(T0 % (unsigned)S);
            unsigned phase = (T0 / (unsigned)S) & 1u;
            for (int tau = 0; tau < tend; ++tau) {
                if (!mbar_wait(&s_full[stage], phase, inner_budget, &s_abort_tick, tau, &s_dead)) {
                    if (s_abort_tick > tau) {  // no abort announced: a lost signal
                        atomicCAS(status, kStatusOk, kStatusInternal);
                        s_dead = 1;
                    }
                }
                if (s_abort_tick <= tau) break;  // same tick for every compute warp
                const int h = tau - L * warp;
                if (!s_dead && h >= 0 && h < my_h_end) {
                    if (my_slot < 0) {
                        my_slot = cb.slot(r0 + warp + P.bp + (h / U) * P.b);
                    } else if (h % U == 0) {
                        my_slot += P.b;
                        while (my_slot >= cb.nslot) my_slot -= cb.nslot;
                    }
                    Chase::template unit<T, ST, WMAX>(P, cb, r0 + warp, h, my_slot, vbuf + (size_t)warp * VS,
                                                      taubuf + warp);
                    // the storer's bulk copies read these columns through the async proxy
                    if (GA.bulk_store) fence_proxy_async_smem();
                }
                named_bar_sync(1, 32 * GA.g);
                if (s_dead) break;  // read after the barrier: same tick for every compute warp
                // the last compute warp signals, so warp 0 (the front sweep) goes on at once
                if (threadIdx.x == 32 * (GA.g - 1)) mbar_arrive(&s_done[stage]);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        } else if (warp == GA.g) {
            // ---- loader ----
            long long B = Chase::min_col(P, r0, 0) - 1;  // last column copied in
            int seen = (G == 0) ? 0x7fffffff : -1;
            int stage = (int)(T0 % (unsigned)S);
            for (int u = 0; u < tend; ++u) {
                bool ok = true;
                // Storer progress: tick X is retired once s_retired >= X.  The
                // loader sleeps on the storer's per-tick mbarrier rather than
                // polling shared memory.  The storer is never past tick u - 1
                // here (compute has not run tick u), so the phase of tick X < u
                // cannot have been overtaken.
                auto storer_done = [&](int X) -> bool {
                    while (ld_acquire_cta_shared(&s_retired) < X) {
                        const unsigned q = T0 + (unsigned)X;
                        if (!mbar_wait(&s_stored[q % S], (q / S) & 1u, inner_budget, &s_abort_tick, u, &s_dead))
                            return false;
                    }
                    return true;
                };
                // stay within `ahead` ticks of the storer (mbarrier phases)
                if (u - GA.ahead - 1 >= 0) ok = storer_done(u - GA.ahead - 1);
                const long long xn = ok ? tick_max_col<Chase>(P, r0, ng, L, s_nsteps, u) : -1;
                if (ok && xn > B) {
                    // slots of the columns xn - nslot + 1 .. xn must be free: wait
                    // for the storer's next ticks (at most up to tick u - 1)
                    while (ok && (long long)ld_acquire_cta_shared(&s_freed) < xn - GA.nslot + 1) {
                        const int X = ld_acquire_cta_shared(&s_retired) + 1;
                        ok = (X <= u - 1) && storer_done(X);
                    }
                    if (ok && G > 0) ok = warp_wait(wm + G - 1, (int)(xn + 1), status, P, seen);
                }
                if (!ok) {
                    if (lane == 0) {
                        atomicCAS(status, kStatusOk, kStatusTimeout);
                        s_abort_tick = u;
                        mbar_arrive(&s_full[stage]);  // completes the phase: no bytes expected
                    }
                    // let the copies already issued land before the CTA leaves
                    const int never = 0;
                    for (int v = max(0, u - S + 1); v < u; ++v) {
                        const unsigned qv = T0 + (unsigned)v;
                        (void)mbar_wait(&s_full[qv % S], (qv / S) & 1u, inner_budget, &s_abort_tick, 0x7fffffff,
                                        &never);
                    }
                    break;
                }
                if (xn > B) {
                    if (lane == 0) mbar_arrive_expect_tx(&s_full[stage], (unsigned)(xn - B) * col_bytes);
                    __syncwarp();
                    // the copies read what group G - 1 wrote (acquired above)
                    fence_proxy_async_global();
                    for (int j = (int)B + 1 + lane; j <= (int)xn; j += 32)
                        bulk_load(cb.col(j), band + (long long)j * P.ldab + GA.top, col_bytes, &s_full[stage]);
                    B = xn;
                } else if (lane == 0) {
                    mbar_arrive(&s_full[stage]);
                }
                if (++stage == S) stage = 0;
            }
        } else if (warp == GA.g + 1) {
            // ---- storer ----
            long long A = Chase::min_col(P, r0, 0);  // first column not yet written back
            long long xr = -1;                   // last column ticks <= v touch
            int a_prev = (int)A;                 // A before this iteration's write-backs
            bool stopped = false;
            int stage = (int)(T0 % (unsigned)S);
            unsigned phase = (T0 / (unsigned)S) & 1u;
            const int nv = (int)(col_bytes / 16);
            for (int v = 0; v < tend; ++v) {
                if (!mbar_wait(&s_done[stage], phase, inner_budget, &s_abort_tick, v, &s_dead)) {
                    if (lane == 0 && s_abort_tick > v && !s_dead) {  // no abort announced: a lost signal
                        atomicCAS(status, kStatusOk, kStatusInternal);
                        s_dead = 1;
                    }
                    stopped = true;
                    break;
                }
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
                xr = max(xr, tick_max_col<Chase>(P, r0, ng, L, s_nsteps, v));
                long long an =
                    (v == tend - 1) ? (long long)P.n : tick_min_col<Chase>(P, r0, ng, L, s_nsteps, v + 1);
                an = min(an, xr + 1);
                if (GA.bulk_store) {
                    if (an > A) {
                        for (int j = (int)A + lane; j < (int)an; j += 32)
                            bulk_store(band + (long long)j * P.ldab + GA.top, cb.col(j), col_bytes);
                        A = an;
                    }
                    bulk_commit();
                    bulk_wait_read();  // sources read: the slots may be refilled
                    // columns written back in earlier iterations are complete once
                    // only this iteration's group may still be pending: report
                    // them (one iteration late, so the wait rarely stalls)
                    bulk_wait_prev();
                    fence_proxy_async_global();
                } else {
                    if (an > A) {
                        // element e of the range: vector e mod nv of column A + e / nv
                        const int total = (int)(an - A) * nv;
                        const int dq = 32 / nv, dr = 32 % nv;
                        int jc = lane / nv, vq = lane % nv;
                        for (int e = lane; e < total; e += 32) {
                            const int j = (int)A + jc;
                            const int4* src = reinterpret_cast<const int4*>(cb.col(j));
                            int4* dst = reinterpret_cast<int4*>(band + (long long)j * P.ldab + GA.top);
                            dst[vq] = src[vq];
                            jc += dq;
                            vq += dr;
                            if (vq >= nv) {
                                vq -= nv;
                                ++jc;
                            }
                        }
                        A = an;
                    }
                    a_prev = (int)A;  // plain stores: reported at once (the publisher fences)
                    // these reads of the freed slots come before the loader's bulk
                    // writes into them
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    st_release_cta_shared(&s_freed, (int)A);
                    st_release_cta_shared(&s_retired, v);
                    st_release_cta_shared(&s_written, a_prev);
                    mbar_arrive(&s_stored[(T0 + (unsigned)v) % (unsigned)S]);  // release: orders the stores above
                }
                a_prev = (int)A;
            }
            if (GA.bulk_store) {
                bulk_wait_all();
                fence_proxy_async_global();
            }
            __syncwarp();
            if (lane == 0 && !stopped) st_release_cta_shared(&s_written, (int)P.n);
        } else if (warp == GA.g + 2) {
            // ---- publisher: the release's latency stays off the storer's path ----
            if (lane == 0) {
                const bool publish = P.stall_sweep < r0 || P.stall_sweep >= r0 + ng;  // fault injection
                int published = -1;
                long long t0 = clock64();
                for (;;) {
                    const int a = ld_acquire_cta_shared(&s_written);
                    if (a > published) {
                        // release: cumulative over the storer's writes, which the
                        // acquire of s_written ordered before it
                        if (publish) st_release_gpu(wm + G, a);
                        published = a;
                        if (a >= P.n) break;
                        t0 = clock64();
                    } else {
                        if (s_abort_tick != 0x7fffffff || s_dead) break;
                        if ((unsigned long long)(clock64() - t0) > inner_budget) {
                            atomicCAS(status, kStatusOk, kStatusInternal);
                            s_dead = 1;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
            }
        }
        T0 += (unsigned)tend;
        __syncthreads();
        // every warp has left its loop; the flags are final and read alike
        if (s_dead || s_abort_tick != 0x7fffffff) return;
    }
}

}  // namespace bb
