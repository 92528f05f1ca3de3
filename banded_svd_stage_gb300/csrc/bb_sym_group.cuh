// The symmetric chase on the group kernel: g consecutive sweeps of a pass per
// CTA in lockstep, every column they touch held in shared memory (the
// pipeline of bb_group.cuh, with the step below as its unit).
//
// Step k of sweep r of pass (b, t) ("A two-stage reduction on an Apple M5
// Pro", Section 6, with the passes of "Accelerating Bidiagonalization of
// Banded Matrices through Memory-Aware Bulge-Chasing on GPUs", Section III):
// c = r + b' + k b, p = r (k = 0) else c - b, ce = min(c + t, n-1),
// cend = min(ce + b, n-1), w = ce - c + 1, on a symmetric band in lower
// storage, A(i, j) (i >= j).  The reflector H = I - tau v v^T of column p,
// rows c..ce, is applied
//   from the left to columns p+1 .. c-1, rows c..ce;
//   from both sides to the block S = A(c..ce, c..ce) as x = tau S v,
//   x += -(tau/2)(x . v) v, S -= v x^T + x v^T (lower triangle);
//   from the right to rows ce+1 .. cend, columns c..ce.
// A step touches columns p..ce, rows up to b + t below the diagonal.
//
// Lockstep: sweep jj of a group runs step tau - L*jj at tick tau with the
// lag L of the flag scheduler (2, or 3 when b - t = 1).  Step k of sweep r
// and step k - L of sweep r + 1 touch disjoint columns ((L-1) b > t + 1), so
// the steps of one tick are independent and overlapping steps of different
// sweeps run in sweep order.
//
// The arithmetic of each part is that of the flag kernel's step (same
// operations in the same order), so the two schedulers give bitwise equal
// results.
#pragma once

#include <algorithm>

#include "bb_group.cuh"
#include "bb_internal.h"

namespace bb {

// One entry of the rank-2 update S -= v x^T + x v^T: a - v_u x_q - x_u v_q.
template <typename T>
__device__ __forceinline__ T sym_rank2(T a, T vu, T xq, T xu, T vq) {
    return fma(-xu, vq, fma(-vu, xq, a));
}

// Lower-triangle entry e = u (u + 1) / 2 + q of a w x w block: (u, q),
// 0 <= q <= u.
__device__ __forceinline__ void sym_pair(int e, int& u, int& q) {
    int uu = (int)((sqrtf(8.f * (float)e + 1.f) - 1.f) * 0.5f);
    while (uu * (uu + 1) / 2 > e) --uu;
    while ((uu + 1) * (uu + 2) / 2 <= e) ++uu;
    u = uu;
    q = e - uu * (uu + 1) / 2;
}

// Step of the symmetric chase on the buffered band, by one warp.  s0: the
// buffer slot of column c; columns c + d, -b <= d <= t, sit in slot s0 + d,
// wrapped once (the buffer holds more than b + t + 1 columns).  vb: the
// reflector, xb: x, taub: tau (this warp's scratch).
template <typename T, int WMAX, bool FULL>
__device__ __forceinline__ void group_sym_step(const ColBuf<T>& cb, const GGeom& g, int s0, T* vb, T* xb,
                                               T* taub) {
    constexpr int NPL = (WMAX + 31) / 32;
    constexpr unsigned S = sizeof(T);
    const int W = FULL ? WMAX : g.w;
    const int lane = threadIdx.x & 31;
    const int lds = cb.lds, nslot = cb.nslot;
    auto slot_of = [&](int d) -> int {
        int sl = s0 + d;
        if (sl < 0) sl += nslot;
        else if (sl >= nslot) sl -= nslot;
        return sl;
    };
    // A(c + m, p) is element colp + m
    const int dp = g.p - g.c;
    const int colp = slot_of(dp) * lds + cb.off - dp;
    T xp[NPL];
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        xp[q] = (m < W) ? sh_ld<T>(cb.at(colp + m)) : T(0);
    }
    const T beta = warp_larfg<T, NPL>(xp, W, lane, vb, taub);
#pragma unroll
    for (int q = 0; q < NPL; ++q) {
        const int m = lane + 32 * q;
        if (m < W) sh_st(cb.at(colp + m), (m == 0) ? beta : T(0));
    }
    __syncwarp();
    const T tau = sh_ld<T>(sh_addr(taub));
    if (tau == T(0)) return;  // H = I
    constexpr bool kVReg = group_v_in_registers<T, WMAX>();
    const unsigned vaddr = sh_addr(vb);
    const unsigned xaddr = sh_addr(xb);
    T vreg[kVReg ? WMAX : 1];
    if constexpr (kVReg) load_v<T, WMAX>(vaddr, vreg);
    auto v = [&](int m) -> T {
        if constexpr (kVReg) return vreg[m];
        else return sh_ld<T>(vaddr + S * (unsigned)m);
    };
    // om(m): address of A(c, c + m) minus m entries, so that A(c + u, c + m)
    // is at om(m) + S u (column c + m in slot s0 + m, wrapped once)
    const int mwrap = nslot - s0;
    const unsigned om0 = cb.at(s0 * lds + cb.off);
    const unsigned dm = S * (unsigned)(lds - 1), wrapb = S * (unsigned)(nslot * lds);
    auto om = [&](int m) -> unsigned { return om0 + dm * (unsigned)m - ((m >= mwrap) ? wrapb : 0u); };
    // Three parts on disjoint entries, one lane per task: a column left of the
    // block, a row below it, a row u of x = tau S v.
    const int nleft = -dp - 1;
    const int nbelow = g.cend - g.ce;
    // y = v . a, a -= (tau y) v over the task's w entries, entry m at addr(m)
    auto apply = [&](auto addr) {
        T a[WMAX];
        T y = 0;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) {
                a[m] = sh_ld<T>(addr(m));
                y = fma(v(m), a[m], y);
            }
        const T s = tau * y;
#pragma unroll
        for (int m = 0; m < WMAX; ++m)
            if (m < W) sh_st(addr(m), fma(-s, v(m), a[m]));
    };
    for (int idx = lane; idx < nleft + nbelow + W; idx += 32) {
        if (idx < nleft) {
            const int d = dp + 1 + idx;  // column c + d, rows c .. ce
            const unsigned ea = cb.at(slot_of(d) * lds + cb.off - d);
            apply([&](int m) { return ea + S * (unsigned)m; });
        } else if (idx < nleft + nbelow) {
            const unsigned ei = S * (unsigned)(g.ce + 1 + (idx - nleft) - g.c);  // row c + i, columns c .. ce
            apply([&](int m) { return om(m) + ei; });
        } else {
            const int u = idx - nleft - nbelow;
            const unsigned ou = cb.at(slot_of(u) * lds + cb.off - u);  // A(c + q, c + u) at ou + S q
            T y = 0;
#pragma unroll
            for (int q = 0; q < WMAX; ++q)
                if (q < W) {
                    const T sq = (u >= q) ? sh_ld<T>(om(q) + S * (unsigned)u) : sh_ld<T>(ou + S * (unsigned)q);
                    y = fma(sq, v(q), y);
                }
            sh_st(xaddr + S * (unsigned)u, tau * y);
        }
    }
    __syncwarp();
    {
        T dot = 0;
        // v from shared memory: u is not a compile-time index here
        for (int u = lane; u < W; u += 32)
            dot = fma(sh_ld<T>(xaddr + S * (unsigned)u), sh_ld<T>(vaddr + S * (unsigned)u), dot);
        dot = warp_sum(dot);
        const T alpha = -(T(0.5) * tau) * dot;
        for (int u = lane; u < W; u += 32)
            sh_st(xaddr + S * (unsigned)u,
                  fma(alpha, sh_ld<T>(vaddr + S * (unsigned)u), sh_ld<T>(xaddr + S * (unsigned)u)));
    }
    __syncwarp();
    const int npairs = W * (W + 1) / 2;
    for (int e = lane; e < npairs; e += 32) {
        int u, q;
        sym_pair(e, u, q);
        const unsigned aq = cb.at(slot_of(q) * lds + cb.off - q + u);  // A(c + u, c + q)
        const T vu = sh_ld<T>(vaddr + S * (unsigned)u), vq = sh_ld<T>(vaddr + S * (unsigned)q);
        const T xu = sh_ld<T>(xaddr + S * (unsigned)u), xq = sh_ld<T>(xaddr + S * (unsigned)q);
        sh_st(aq, sym_rank2(sh_ld<T>(aq), vu, xq, xu, vq));
    }
}

// The symmetric chase as a group-kernel unit: one step per unit; per warp the
// reflector v and the vector x.
struct SymChase {
    static constexpr int kUnits = 1;
    static constexpr int kVecs = 2;
    // ce of step h
    __device__ static long long max_col(const PassArgs& P, int r, int h) {
        return min((long long)r + P.bp + (long long)h * P.b + P.t, P.n - 1);
    }
    // p of step h
    __device__ static long long min_col(const PassArgs& P, int r, int h) {
        return (h == 0) ? (long long)r : (long long)r + P.bp + (long long)(h - 1) * P.b;
    }
    template <typename T, typename ST, int WMAX>
    __device__ static void unit(const PassArgs& P, const ColBuf<ST>& cb, int r, int h, int slot, T* vb, T* taub) {
        static_assert(std::is_same<T, ST>::value, "the symmetric chase stores its band in its arithmetic type");
        const GGeom g = gstep(P, r, h);
        T* xb = vb + group_v_stride(WMAX, (int)sizeof(T));
        if (g.w == WMAX) group_sym_step<T, WMAX, true>(cb, g, slot, vb, xb, taub);
        else group_sym_step<T, WMAX, false>(cb, g, slot, vb, xb, taub);
    }
};

// One pass of the symmetric chase on the group kernel (cooperative launch of
// up to the co-resident maximum of CTAs; wm: one watermark per group).
template <typename T, int WMAX>
cudaError_t run_sym_group_pass(T* band, const PassArgs& P, const GroupArgs& GA, int num_sms, int max_ctas,
                               int* wm, int* status, cudaStream_t s) {
    if (P.nsweeps <= 0) return cudaSuccess;
    return launch_group_pass<T, WMAX, SymChase, T>(band, P, GA, num_sms, max_ctas, wm, status, s);
}

#define BB_SYM_GROUP_INSTANTIATE(T, W)                                                                         \
    template cudaError_t run_sym_group_pass<T, W>(T*, const PassArgs&, const GroupArgs&, int, int, int*, int*, \
                                                  cudaStream_t);
#define BB_SYM_GROUP_EXTERN(T, W)                                                                             \
    extern template cudaError_t run_sym_group_pass<T, W>(T*, const PassArgs&, const GroupArgs&, int, int, int*, \
                                                         int*, cudaStream_t);

}  // namespace bb
