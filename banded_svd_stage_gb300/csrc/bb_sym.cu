// Symmetric variant: a symmetric band (lower band storage) reduced to
// symmetric tridiagonal form by the same passes BW -> BW - TW, one two-sided
// Householder reflector per step.
//
// The variant: "A two-stage reduction on an Apple M5 Pro", Section 6 (band
// to tridiagonal by bulge chasing, timed against ssytrd_sb2st), with the pass
// structure of "Accelerating Bidiagonalization of Banded Matrices through
// Memory-Aware Bulge-Chasing on GPUs", Section III.  Step geometry of pass
// (b, t), sweep r, step k: c = r + b' + k b, p = r (k = 0) else c - b,
// ce = min(c + t, n-1), cend = min(ce + b, n-1), w = ce - c + 1.  The
// reflector H = I - tau v v^T comes from column p, rows c..ce (A(c, p) = beta,
// A(c+1..ce, p) = 0) and is applied
//   from the left to columns p+1 .. c-1, rows c..ce;
//   from both sides to the diagonal block c..ce, as the symmetric rank-2
//   update x = tau S v, x += -(tau/2)(x . v) v, S -= v x^T + x v^T;
//   from the right to rows ce+1 .. cend, columns c..ce.
// Storage: A(i, j), i >= j, at band[(i - j) + j * ldab], ldab >= bw + tw + 1.
//
// Schedulers, per pass:
// - the flag kernel here: one CTA per sweep (persistent, cooperative
//   launch), sweep r taking step k once sweep r-1 has finished
//   min(k + L, K_{r-1}) steps, the last step once all of sweep r-1 is done;
//   L = 2, or 3 when b - t = 1, the least lag for which overlapping steps of
//   consecutive sweeps stay in sweep order.  Band data another CTA wrote is
//   read through L2 (ld.global.cg);
// - the group kernel (bb_sym_group.cuh): g sweeps per CTA in lockstep with
//   the same lag, their columns in shared memory, whole columns handed from
//   group to group.  Chosen where at least kAutoGroupMin sweeps fit shared
//   memory (or wherever one fits, on request), for reflectors of up to 33
//   elements.
// Both give bitwise equal results.
#include <cuda_runtime.h>

#include <algorithm>

#include "bb_device.cuh"
#include "bb_internal.h"
#include "bb_sym.h"
#include "bb_sym_group.cuh"

namespace bb {

BB_SYM_GROUP_EXTERN(float, 9) BB_SYM_GROUP_EXTERN(float, 17) BB_SYM_GROUP_EXTERN(float, 33)
BB_SYM_GROUP_EXTERN(double, 9) BB_SYM_GROUP_EXTERN(double, 17) BB_SYM_GROUP_EXTERN(double, 33)

constexpr int kSymThreads = 256;

// Step lag of the symmetric variant in pass (b, t).
int sym_pass_lag(int b, int t) { return (b - t >= 2) ? 2 : 3; }

bool sym_choose_group(const PassArgs& P, int scheduler, int group_size, size_t elem, GroupArgs* out) {
    if (scheduler != 0 && scheduler != 3) return false;
    if (P.nsweeps <= 0 || P.n >= kGroupMaxN) return false;
    const int wmax = sym_group_wmax(P.t + 1);
    if (wmax == 0) return false;
    GroupArgs ga;
    if (!plan_group(P, wmax, elem, group_size, &ga, ChaseKind::kSym)) return false;
    // automatic: the group kernel from 3 sweeps per group in float, from
    // kAutoGroupMin in double.  Measured against this file's flag kernel:
    // float, n = 8192, bw 64, pass 0 on the group kernel with g = 4: 414 ->
    // 351 ms for the reduction; float, n = 32768, bw 256, passes with g = 1
    // and 3: 12.3 -> 10.9 s; double, n = 8192, bw 64, passes with g = 1 and
    // 3: 844 -> 1050 ms (the FP64 work of g sweeps shares one SM)
    const int gmin = (elem == 4) ? 3 : kAutoGroupMin;
    if (scheduler == 0 && ga.g < gmin) return false;
    if (out) *out = ga;
    return true;
}

template <typename T>
__device__ __forceinline__ T sym_ld(const T* band, long long ld, long long i, long long j) {
    return __ldcg(band + (i - j) + j * ld);
}
template <typename T>
__device__ __forceinline__ void sym_st(T* band, long long ld, long long i, long long j, T v) {
    band[(i - j) + j * ld] = v;
}

// One step of sweep r by the whole CTA.  s_v, s_x hold WMAX entries.
template <typename T, int WMAX>
__device__ __forceinline__ void sym_step(T* __restrict__ band, const PassArgs& P, long long r, int k, T* s_v,
                                         T* s_x, T* s_tau) {
    constexpr int NPL = (WMAX + 31) / 32;
    const long long n = P.n, ld = P.ldab;
    const long long c = r + P.bp + (long long)k * P.b;
    const long long p = (k == 0) ? r : c - P.b;
    const long long ce = min(c + (long long)P.t, n - 1);
    const long long cend = min(ce + (long long)P.b, n - 1);
    const int w = (int)(ce - c + 1);
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        T x[NPL];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            x[q] = (m < w) ? sym_ld(band, ld, c + m, p) : T(0);
        }
        const T beta = warp_larfg<T, NPL>(x, w, lane, s_v, s_tau);
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            if (m < w) sym_st(band, ld, c + m, p, (m == 0) ? beta : T(0));
        }
    }
    __syncthreads();
    const T tau = *s_tau;
    if (tau == T(0)) return;  // H = I; the value is the same for every thread
    // the three parts touch disjoint entries: one thread per column left of
    // the block, per row below it, and per row u of x = tau S v
    const int nleft = (int)(c - 1 - p);
    const int nbelow = (int)(cend - ce);
    for (int idx = threadIdx.x; idx < nleft + nbelow + w; idx += blockDim.x) {
        if (idx < nleft) {
            const long long j = p + 1 + idx;
            T a[WMAX];
            T y = 0;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) {
                    a[m] = sym_ld(band, ld, c + m, j);
                    y = fma(s_v[m], a[m], y);
                }
            const T s = tau * y;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) sym_st(band, ld, c + m, j, fma(-s, s_v[m], a[m]));
        } else if (idx < nleft + nbelow) {
            const long long i = ce + 1 + (idx - nleft);
            T a[WMAX];
            T y = 0;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) {
                    a[m] = sym_ld(band, ld, i, c + m);
                    y = fma(s_v[m], a[m], y);
                }
            const T s = tau * y;
#pragma unroll
            for (int m = 0; m < WMAX; ++m)
                if (m < w) sym_st(band, ld, i, c + m, fma(-s, s_v[m], a[m]));
        } else {
            // row u of x = tau S v; unrolled over the compiled width so that
            // the row's loads are in flight together
            const int u = idx - nleft - nbelow;
            T y = 0;
#pragma unroll
            for (int q = 0; q < WMAX; ++q)
                if (q < w) {
                    const T sq = (u >= q) ? sym_ld(band, ld, c + u, c + q) : sym_ld(band, ld, c + q, c + u);
                    y = fma(sq, s_v[q], y);
                }
            s_x[u] = tau * y;
        }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        T dot = 0;
        for (int u = threadIdx.x; u < w; u += 32) dot = fma(s_x[u], s_v[u], dot);
        dot = warp_sum(dot);
        const T alpha = -(T(0.5) * tau) * dot;
        for (int u = threadIdx.x; u < w; u += 32) s_x[u] = fma(alpha, s_v[u], s_x[u]);
    }
    __syncthreads();
    // S -= v x^T + x v^T on the lower triangle: one thread per entry (u, q),
    // 0 <= q <= u < w, entry e = u (u + 1) / 2 + q
    const int npairs = w * (w + 1) / 2;
    for (int e = threadIdx.x; e < npairs; e += blockDim.x) {
        int u, q;
        sym_pair(e, u, q);
        const T a = sym_ld(band, ld, c + u, c + q);
        sym_st(band, ld, c + u, c + q, sym_rank2(a, s_v[u], s_x[q], s_x[u], s_v[q]));
    }
}

template <typename T, int WMAX>
__global__ void __launch_bounds__(kSymThreads)
sym_pass_kernel(T* __restrict__ band, PassArgs P, int* __restrict__ progress, int* __restrict__ status) {
    __shared__ T s_v[WMAX];
    __shared__ T s_x[WMAX];
    __shared__ T s_tau;
    __shared__ int s_flag;
    if (threadIdx.x == 0) s_flag = ld_relaxed_gpu(status);
    __syncthreads();
    if (s_flag != kStatusOk) return;
    for (int r = blockIdx.x; r < P.nsweeps; r += gridDim.x) {
        const int K = sweep_steps(P, r);
        const int Kp = (r > 0) ? sweep_steps(P, r - 1) : 0;
        const bool publish = (r != P.stall_sweep);
        for (int k = 0; k < K; ++k) {
            if (r > 0) {
                const int need = (k == K - 1) ? Kp : min(k + P.lag, Kp);
                if (!block_wait(progress + r - 1, need, status, P, &s_flag)) return;
            } else {
                __syncthreads();  // s_v, s_x of the previous step are no longer read
            }
            sym_step<T, WMAX>(band, P, r, k, s_v, s_x, &s_tau);
            if (publish) block_publish(progress + r, k + 1);
            else __syncthreads();
        }
    }
}

// One step of sweep r by the whole CTA on a shared-memory copy of its
// window, with the operations and their order of sym_step (so the two give
// bitwise equal results):
//   Lt: columns p .. c-1, rows c .. ce: Lt[(j - p) ws + m] = A(c + m, j)
//       (ws = WMAX | 1, an odd stride);
//   Rt: columns c .. ce, rows c .. cend: Rt[q rs + i] = A(c + i, c + q),
//       i >= q (rs = b + t + 1).
// The window is read once after the wait and written back once; in between
// the three parts, alpha and the rank-2 update work on shared memory.
template <typename T, int WMAX>
__device__ __forceinline__ void sym_step_smem(T* __restrict__ band, const PassArgs& P, long long r, int k, T* Lt,
                                              T* Rt, T* s_v, T* s_x, T* s_tau) {
    constexpr int NPL = (WMAX + 31) / 32;
    constexpr int ws = WMAX | 1;
    const int rs = P.b + P.t + 1;
    const long long n = P.n, ld = P.ldab;
    const long long c = r + P.bp + (long long)k * P.b;
    const long long p = (k == 0) ? r : c - P.b;
    const long long ce = min(c + (long long)P.t, n - 1);
    const long long cend = min(ce + (long long)P.b, n - 1);
    const int w = (int)(ce - c + 1);
    const int nl = (int)(c - p);        // columns p .. c-1
    const int nr = (int)(cend - c + 1);  // rows c .. cend
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
    // read the window (through L2: other CTAs wrote it), a warp per column
    // of the band, lanes along the column
    for (int jl = warp; jl < nl; jl += nwarps) {
        const T* col = band + (c - (p + jl)) + (p + jl) * ld;  // A(c + m, p + jl) = col[m]
        for (int m = lane; m < w; m += 32) Lt[jl * ws + m] = __ldcg(col + m);
    }
    for (int q = warp; q < w; q += nwarps) {
        const T* col = band + (c + q) * ld - q;  // A(c + i, c + q) = col[i], i >= q
        for (int i = q + lane; i < nr; i += 32) Rt[q * rs + i] = __ldcg(col + i);
    }
    __syncthreads();
    if (tid < 32) {
        T x[NPL];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            x[q] = (m < w) ? Lt[m] : T(0);
        }
        const T beta = warp_larfg<T, NPL>(x, w, lane, s_v, s_tau);
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            const int m = lane + 32 * q;
            if (m < w) Lt[m] = (m == 0) ? beta : T(0);
        }
    }
    __syncthreads();
    const T tau = *s_tau;  // the same value in every thread
    if (tau != T(0)) {
        // the three parts on disjoint entries: a column left of the block, a
        // row below it, a row u of x = tau S v; each task's entries are read
        // for the dot product and again for the update (shared memory)
        const int nleft = nl - 1;
        const int nbelow = nr - w;
        for (int idx = tid; idx < nleft + nbelow + w; idx += nt) {
            if (idx < nleft + nbelow) {
                T* a0;
                int st;
                if (idx < nleft) {
                    a0 = Lt + (idx + 1) * ws;  // column p + 1 + idx
                    st = 1;
                } else {
                    a0 = Rt + w + (idx - nleft);  // row c + w + (idx - nleft)
                    st = rs;
                }
                T y = 0;
#pragma unroll
                for (int m = 0; m < WMAX; ++m)
                    if (m < w) y = fma(s_v[m], a0[m * st], y);
                const T sc = tau * y;
#pragma unroll
                for (int m = 0; m < WMAX; ++m)
                    if (m < w) a0[m * st] = fma(-sc, s_v[m], a0[m * st]);
            } else {
                const int u = idx - nleft - nbelow;
                T y = 0;
#pragma unroll
                for (int q = 0; q < WMAX; ++q)
                    if (q < w) {
                        const T sq = (u >= q) ? Rt[q * rs + u] : Rt[u * rs + q];
                        y = fma(sq, s_v[q], y);
                    }
                s_x[u] = tau * y;
            }
        }
        __syncthreads();
        if (tid < 32) {
            T dot = 0;
            for (int u = tid; u < w; u += 32) dot = fma(s_x[u], s_v[u], dot);
            dot = warp_sum(dot);
            const T alpha = -(T(0.5) * tau) * dot;
            for (int u = tid; u < w; u += 32) s_x[u] = fma(alpha, s_v[u], s_x[u]);
        }
        __syncthreads();
        const int npairs = w * (w + 1) / 2;
        for (int e = tid; e < npairs; e += nt) {
            int u, q;
            sym_pair(e, u, q);
            T& a = Rt[q * rs + u];
            a = sym_rank2(a, s_v[u], s_x[q], s_x[u], s_v[q]);
        }
        __syncthreads();
    }
    // write the window back, as it was read
    for (int jl = warp; jl < nl; jl += nwarps) {
        T* col = band + (c - (p + jl)) + (p + jl) * ld;
        for (int m = lane; m < w; m += 32) col[m] = Lt[jl * ws + m];
    }
    for (int q = warp; q < w; q += nwarps) {
        T* col = band + (c + q) * ld - q;
        for (int i = q + lane; i < nr; i += 32) col[i] = Rt[q * rs + i];
    }
}

// Shared memory of sym_step_smem: the two tiles of pass (b, t).
template <typename T, int WMAX>
__host__ __device__ inline size_t sym_tile_bytes(int b, int t) {
    return sizeof(T) * ((size_t)b * (WMAX | 1) + (size_t)(t + 1) * (size_t)(b + t + 1));
}

// The flag kernel with each step's window in shared memory.
template <typename T, int WMAX, int NT>
__global__ void __launch_bounds__(NT)
sym_pass_smem_kernel(T* __restrict__ band, PassArgs P, int* __restrict__ progress, int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char sym_smem[];
    T* Lt = reinterpret_cast<T*>(sym_smem);
    T* Rt = Lt + (size_t)P.b * (WMAX | 1);
    __shared__ T s_v[WMAX];
    __shared__ T s_x[WMAX];
    __shared__ T s_tau;
    __shared__ int s_flag;
    if (threadIdx.x == 0) s_flag = ld_relaxed_gpu(status);
    __syncthreads();
    if (s_flag != kStatusOk) return;
    for (int r = blockIdx.x; r < P.nsweeps; r += gridDim.x) {
        const int K = sweep_steps(P, r);
        const int Kp = (r > 0) ? sweep_steps(P, r - 1) : 0;
        const bool publish = (r != P.stall_sweep);
        for (int k = 0; k < K; ++k) {
            if (r > 0) {
                const int need = (k == K - 1) ? Kp : min(k + P.lag, Kp);
                if (!block_wait(progress + r - 1, need, status, P, &s_flag)) return;
            } else {
                __syncthreads();  // the tiles and s_v, s_x of the previous step are no longer read
            }
            sym_step_smem<T, WMAX>(band, P, r, k, Lt, Rt, s_v, s_x, &s_tau);
            if (publish) block_publish(progress + r, k + 1);
            else __syncthreads();
        }
    }
}

// Zero the fill rows bw+1 .. bw+tw of every column.
template <typename T>
__global__ void sym_zero_fill_kernel(T* __restrict__ band, long long n, long long ldab, int bw, int tw) {
    const long long total = n * (long long)tw;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long j = idx / tw;
        const long long q = bw + 1 + idx % tw;
        band[q + j * ldab] = T(0);
    }
}

// d_i = A(i, i), e_i = A(i+1, i).
template <typename T>
__global__ void sym_extract_kernel(const T* __restrict__ band, long long n, long long ldab, T* __restrict__ d,
                                   T* __restrict__ e) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        d[i] = band[i * ldab];
        if (i + 1 < n) e[i] = band[1 + i * ldab];
    }
}

// Most shared memory the window copy of sym_pass_smem_kernel may take.
constexpr size_t kSymTileMax = 200 * 1024;

// The flag kernel with the window in shared memory, NT threads per CTA.
template <typename T, int WMAX, int NT>
static cudaError_t run_sym_pass_smem(T* band, const PassArgs& P, int num_sms, int max_ctas, int* progress,
                                     int* status, cudaStream_t s) {
    auto kern = sym_pass_smem_kernel<T, WMAX, NT>;
    const size_t smem = sym_tile_bytes<T, WMAX>(P.b, P.t);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = std::min<long long>((long long)per_sm * num_sms, P.nsweeps);
    if (max_ctas > 0) grid = std::min<long long>(grid, max_ctas);
    err = cudaMemsetAsync(progress, 0, sizeof(int) * (size_t)P.nsweeps, s);
    if (err != cudaSuccess) return err;
    T* band_arg = band;
    PassArgs p_arg = P;
    int* prog_arg = progress;
    int* stat_arg = status;
    void* args[] = {&band_arg, &p_arg, &prog_arg, &stat_arg};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(NT), args, smem, s);
}

template <typename T, int WMAX>
static cudaError_t run_sym_pass(T* band, const PassArgs& P, int num_sms, int max_ctas, int* progress, int* status,
                                cudaStream_t s) {
    if (P.nsweeps <= 0) return cudaSuccess;
    // 512 threads for the 32-wide kernel on wide passes; the wider kernels
    // keep 256 (their registers would spill at 512)
    if (sym_tile_bytes<T, WMAX>(P.b, P.t) <= kSymTileMax) {
        if constexpr (WMAX == 32) {
            if (P.b >= 96) return run_sym_pass_smem<T, WMAX, 512>(band, P, num_sms, max_ctas, progress, status, s);
        }
        return run_sym_pass_smem<T, WMAX, 256>(band, P, num_sms, max_ctas, progress, status, s);
    }
    auto kern = sym_pass_kernel<T, WMAX>;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSymThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = std::min<long long>((long long)per_sm * num_sms, P.nsweeps);
    if (max_ctas > 0) grid = std::min<long long>(grid, max_ctas);
    err = cudaMemsetAsync(progress, 0, sizeof(int) * (size_t)P.nsweeps, s);
    if (err != cudaSuccess) return err;
    T* band_arg = band;
    PassArgs p_arg = P;
    int* prog_arg = progress;
    int* stat_arg = status;
    void* args[] = {&band_arg, &p_arg, &prog_arg, &stat_arg};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(kSymThreads), args, 0, s);
}

// The pass arguments of pass (b, t) of the symmetric chase.
static PassArgs sym_pass_args(long long n, long long ldab, int b, int t, const SymLaunch& L) {
    PassArgs P{};
    P.n = n;
    P.ldab = ldab;
    P.b = b;
    P.t = t;
    P.bp = b - t;
    P.ku = 0;
    P.nsweeps = (int)std::max<long long>(0, n - (b - t) - 1);
    P.lag = sym_pass_lag(b, t);
    P.lagh = P.lag;
    P.stall_sweep = L.stall_sweep;
    P.wait_budget = L.wait_budget;
    return P;
}

bool sym_any_group(long long n, int bw, int tw, const SymLaunch& L, size_t elem) {
    for (int b = bw; b > 1;) {
        const int t = std::min(tw, b - 1);
        if (sym_choose_group(sym_pass_args(n, 0, b, t, L), L.scheduler, L.group_size, elem, nullptr)) return true;
        b -= t;
    }
    return false;
}

template <typename T>
cudaError_t run_sym(T* band, long long n, long long ldab, int bw, int tw, T* d, T* e, const SymLaunch& L,
                    cudaStream_t s, long long* launches, SymPassStats* stats) {
    cudaError_t err = cudaSuccess;
    long long nl = 0;
    if (stats) {
        stats->kernel.clear();
        stats->group.clear();
    }
    const bool layout_ok = group_layout_ok(band, ldab, sizeof(T));
    if (n * (long long)tw > 0) {
        const long long total = n * (long long)tw;
        const unsigned grid = (unsigned)std::min<long long>((total + 255) / 256, 4LL * L.num_sms);
        sym_zero_fill_kernel<T><<<grid, 256, 0, s>>>(band, n, ldab, bw, tw);
        err = cudaGetLastError();
        ++nl;
    }
    int b = bw;
    while (err == cudaSuccess && b > 1) {
        const int t = std::min(tw, b - 1);
        const PassArgs P = sym_pass_args(n, ldab, b, t, L);
        const int w = t + 1;
        GroupArgs ga{};
        const bool grp = layout_ok && sym_choose_group(P, L.scheduler, L.group_size, sizeof(T), &ga);
        if (grp) {
            const int wmax = sym_group_wmax(w);
            auto launch = (wmax == 9) ? run_sym_group_pass<T, 9>
                                      : (wmax == 17) ? run_sym_group_pass<T, 17> : run_sym_group_pass<T, 33>;
            err = launch(band, P, ga, L.num_sms, L.max_ctas, L.progress, L.status, s);
        } else if (w <= 32) {
            err = run_sym_pass<T, 32>(band, P, L.num_sms, L.max_ctas, L.progress, L.status, s);
        } else if (w <= 64) {
            err = run_sym_pass<T, 64>(band, P, L.num_sms, L.max_ctas, L.progress, L.status, s);
        } else {
            err = run_sym_pass<T, 96>(band, P, L.num_sms, L.max_ctas, L.progress, L.status, s);
        }
        if (P.nsweeps > 0) ++nl;
        if (stats) {
            stats->kernel.push_back(grp ? 3 : 2);
            stats->group.push_back(grp ? ga.g : 0);
        }
        b -= t;
    }
    if (err == cudaSuccess) {
        const unsigned grid = (unsigned)std::max<long long>(1, std::min<long long>((n + 255) / 256, 4LL * L.num_sms));
        sym_extract_kernel<T><<<grid, 256, 0, s>>>(band, n, ldab, d, e);
        err = cudaGetLastError();
        ++nl;
    }
    if (launches) *launches = nl;
    return err;
}

template cudaError_t run_sym<float>(float*, long long, long long, int, int, float*, float*, const SymLaunch&,
                                    cudaStream_t, long long*, SymPassStats*);
template cudaError_t run_sym<double>(double*, long long, long long, int, int, double*, double*,
                                     const SymLaunch&, cudaStream_t, long long*, SymPassStats*);

}  // namespace bb
