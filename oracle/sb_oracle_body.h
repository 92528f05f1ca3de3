/*
 * Symmetric variant of the serial CPU oracle: a symmetric band matrix reduced
 * to symmetric tridiagonal form by the same successive band reduction, written
 * once and instantiated for float and double by bb_oracle.c after
 * bb_oracle_body.h (whose reflector, oracle_larfg, it uses).
 *
 * TEST INFRASTRUCTURE ONLY: nothing on the product path may include, link or
 * call this file.
 *
 * The variant is named by both pages: "A two-stage reduction on an Apple M5
 * Pro", Section 6 (band to tridiagonal by bulge chasing with LAPACK's
 * symmetric kernels, timed against ssytrd_sb2st), and "Accelerating
 * Bidiagonalization of Banded Matrices through Memory-Aware Bulge-Chasing on
 * GPUs", Section III (bandwidth BW -> BW - TW per pass, TW entries cleared
 * by one reflector).  The reading taken: the sweep/step geometry of the
 * bidiagonal oracle, with one reflector per step applied from both sides.
 *
 * A is symmetric with A(i, j) = 0 for |i - j| > b; only i >= j is stored:
 * A(i, j) at band[(i - j) + j * ldab] (LAPACK's lower band layout, column j
 * contiguous), ldab >= bw + tw + 1 so that the bulge (up to b + t below the
 * diagonal) fits.  Pass (b, t), b' = b - t; sweep r; step k:
 *   c = r + b' + k b,  p = r (k = 0) or c - b (k > 0),
 *   ce = min(c + t, n - 1),  cend = min(ce + b, n - 1),  w = ce - c + 1.
 * Reflector H = I - tau v v^T (xLARFG convention) from column p, rows c..ce:
 *   A(c, p) = beta, A(c+1..ce, p) = 0;
 *   left part   cols j in (p, c):    A(c..ce, j) <- H A(c..ce, j)
 *   block       rows/cols c..ce:     S <- H S H, as the symmetric rank-2
 *               update x = tau S v, x += -(tau/2)(x . v) v,
 *               S <- S - v x^T - x v^T (which equals H S H)
 *   below part  rows i in (ce, cend]: A(i, c..ce) <- A(i, c..ce) H
 * The three parts touch disjoint entries.  The dense mode applies H to every
 * column outside c..ce instead of the two windows and keeps both triangles;
 * the arithmetic on each entry is the same, so the two agree bitwise.
 */

#define CAT2(a, b) a##b
#define CAT(a, b) CAT2(a, b)
#define FN(name) CAT(name, SFX)

/* Symmetric band -> tridiagonal step.  LEFT_LO..LEFT_HI: the columns j < c
 * updated from the left; BELOW_LO..BELOW_HI: the rows i > ce updated from the
 * right.  GET(i, j) reads A(i, j) for i >= j; PUT(i, j, x) stores it (and its
 * mirror in the dense mode). */
#define SYM_STEP_BODY(LEFT_LO, LEFT_HI, BELOW_LO, BELOW_HI)                                 \
    do {                                                                                \
        int64_t c = r + (b - t) + k * b;                                                \
        int64_t p = (k == 0) ? r : c - b;                                               \
        int64_t ce = (c + t < n - 1) ? c + t : n - 1;                                   \
        int64_t cend = (ce + b < n - 1) ? ce + b : n - 1;                               \
        int64_t w = ce - c + 1;                                                         \
        REAL v[ORACLE_WMAX] = {0};                                                      \
        REAL x[ORACLE_WMAX] = {0};                                                      \
        REAL tau, beta;                                                                 \
        (void)cend;                                                                     \
        for (int64_t q = 0; q < w; ++q) v[q] = GET(c + q, p);                           \
        beta = v[0];                                                                    \
        FN(oracle_larfg)(w - 1, &beta, v + 1, 1, &tau);                                 \
        v[0] = 1;                                                                       \
        PUT(c, p, beta);                                                                \
        for (int64_t q = 1; q < w; ++q) PUT(c + q, p, (REAL)0);                         \
        if (tau != 0) {                                                                 \
            for (int64_t j = (LEFT_LO); j <= (LEFT_HI); ++j) {                          \
                if (j == p) continue;                                                   \
                REAL y = 0;                                                             \
                for (int64_t q = 0; q < w; ++q) y = y + v[q] * GET(c + q, j);           \
                REAL s = tau * y;                                                       \
                for (int64_t q = 0; q < w; ++q) PUT(c + q, j, GET(c + q, j) - s * v[q]); \
            }                                                                           \
            for (int64_t i = (BELOW_LO); i <= (BELOW_HI); ++i) {                        \
                REAL y = 0;                                                             \
                for (int64_t q = 0; q < w; ++q) y = y + v[q] * GET(i, c + q);           \
                REAL s = tau * y;                                                       \
                for (int64_t q = 0; q < w; ++q) PUT(i, c + q, GET(i, c + q) - s * v[q]); \
            }                                                                           \
            for (int64_t u = 0; u < w; ++u) {                                           \
                REAL y = 0;                                                             \
                for (int64_t q = 0; q < w; ++q)                                         \
                    y = y + ((u >= q) ? GET(c + u, c + q) : GET(c + q, c + u)) * v[q];  \
                x[u] = tau * y;                                                         \
            }                                                                           \
            REAL dot = 0;                                                               \
            for (int64_t u = 0; u < w; ++u) dot = dot + x[u] * v[u];                    \
            REAL alpha = -((REAL)0.5 * tau) * dot;                                      \
            for (int64_t u = 0; u < w; ++u) x[u] = x[u] + alpha * v[u];                 \
            for (int64_t u = 0; u < w; ++u)                                             \
                for (int64_t q = 0; q <= u; ++q)                                        \
                    PUT(c + u, c + q, GET(c + u, c + q) - v[u] * x[q] - x[u] * v[q]);   \
        }                                                                               \
    } while (0)

/* Band mode: A(i, j), i >= j, lives at band[(i - j) + j * ldab]. */
#define GET(i, j) band[((i) - (j)) + (j) * ldab]
#define PUT(i, j, val) (band[((i) - (j)) + (j) * ldab] = (val))

/* Whole reduction of the lower band storage to tridiagonal form, serial
 * order (pass plan and sweep/step order as oracle_reduce_band).  The fill
 * rows bw+1 .. bw+tw of every column are zeroed first.  Returns 0, or -1 on
 * invalid arguments. */
int FN(oracle_sym_reduce_band)(int64_t n, int64_t bw, int64_t tw, REAL* band, int64_t ldab) {
    if (n < 1 || bw < 0 || bw >= n || tw < 1 || ldab < bw + tw + 1) return -1;
    if (tw > (bw > 2 ? bw - 1 : 1)) return -1;
    if (tw + 1 > ORACLE_WMAX) return -1;
    for (int64_t j = 0; j < n; ++j)
        for (int64_t q = bw + 1; q <= bw + tw; ++q) band[q + j * ldab] = 0;
    int64_t b = bw;
    while (b > 1) {
        int64_t t = (tw < b - 1) ? tw : b - 1;
        for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r) {
            int64_t K = FN(oracle_sweep_steps)(n, b, t, r);
            for (int64_t k = 0; k < K; ++k) SYM_STEP_BODY(p + 1, c - 1, ce + 1, cend);
        }
        b -= t;
    }
    return 0;
}

/* One step (sweep r, step k) of pass (b, t) in lower band storage, the
 * windows as in the whole reduction; for schedule tests. */
void FN(oracle_sym_step_band)(int64_t n, int64_t b, int64_t t, REAL* band, int64_t ldab, int64_t r,
                              int64_t k) {
    SYM_STEP_BODY(p + 1, c - 1, ce + 1, cend);
}

/* Pipelined sweeps on host threads, as oracle_reduce_band_pipelined, one
 * step per unit: step k of sweep r starts once sweep r-1 has finished
 * min(k + L, K_{r-1}) steps, L = 2 when b - t >= 2 and 3 when b - t == 1 (the
 * least lockstep lag of this variant); the last step of a sweep waits for all
 * of sweep r-1. */
static void* FN(sym_pipe_worker_)(void* arg) {
    const FN(pipe_arg_)* a = (const FN(pipe_arg_)*)arg;
    const int64_t n = a->n, b = a->b, t = a->t;
    const int64_t L = (b - t >= 2) ? 2 : 3;
    const int64_t nsweeps = n - (b - t) - 1;
    for (int64_t r = a->thread; r < nsweeps; r += a->nthreads) {
        const int64_t K = FN(oracle_sweep_steps)(n, b, t, r);
        const int64_t Kp = (r > 0) ? FN(oracle_sweep_steps)(n, b, t, r - 1) : 0;
        for (int64_t k = 0; k < K; ++k) {
            if (r > 0) {
                int64_t need = (k + L < Kp) ? k + L : Kp;
                if (k == K - 1) need = Kp;
                if (!FN(pipe_wait_)(&a->done[r - 1], need, a)) return NULL;
            }
            FN(oracle_sym_step_band)(n, b, t, a->band, a->ldab, r, k);
            atomic_store_explicit(&a->done[r], k + 1, memory_order_release);
        }
    }
    return NULL;
}

/* Same arguments and result as oracle_sym_reduce_band, on nthreads (1 ..
 * 1024) threads; return codes as oracle_reduce_band_pipelined. */
int FN(oracle_sym_reduce_band_pipelined)(int64_t n, int64_t bw, int64_t tw, REAL* band, int64_t ldab,
                                         int64_t nthreads, double time_limit_s) {
    if (n < 1 || bw < 0 || bw >= n || tw < 1 || ldab < bw + tw + 1) return -1;
    if (tw > (bw > 2 ? bw - 1 : 1)) return -1;
    if (tw + 1 > ORACLE_WMAX) return -1;
    if (nthreads < 1 || nthreads > 1024 || !(time_limit_s > 0)) return -1;
    for (int64_t j = 0; j < n; ++j)
        for (int64_t q = bw + 1; q <= bw + tw; ++q) band[q + j * ldab] = 0;
    return FN(pipe_run_)(n, bw, tw, band, ldab, nthreads, time_limit_s, FN(sym_pipe_worker_), 0, INT64_MAX);
}

/* d_i = A(i, i), e_i = A(i+1, i) from the lower band storage. */
void FN(oracle_sym_extract_band)(int64_t n, const REAL* band, int64_t ldab, REAL* d, REAL* e) {
    for (int64_t i = 0; i < n; ++i) d[i] = GET(i, i);
    for (int64_t i = 0; i + 1 < n; ++i) e[i] = GET(i + 1, i);
}
#undef GET
#undef PUT

/* Dense mode: A is n x n, row-major, both triangles kept equal.  H is
 * applied to every column outside c..ce (the left part and, mirrored, the
 * below part of the band mode) and to the block; the band windows play no
 * part. */
#define GET(i, j) a[(i) * n + (j)]
#define PUT(i, j, val) (a[(i) * n + (j)] = a[(j) * n + (i)] = (val))
int FN(oracle_sym_reduce_dense)(int64_t n, int64_t bw, int64_t tw, REAL* a) {
    if (n < 1 || bw < 0 || bw >= n || tw < 1) return -1;
    if (tw > (bw > 2 ? bw - 1 : 1)) return -1;
    if (tw + 1 > ORACLE_WMAX) return -1;
    int64_t b = bw;
    while (b > 1) {
        int64_t t = (tw < b - 1) ? tw : b - 1;
        for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r) {
            int64_t K = FN(oracle_sweep_steps)(n, b, t, r);
            for (int64_t k = 0; k < K; ++k) SYM_STEP_BODY(0, c - 1, ce + 1, n - 1);
        }
        b -= t;
    }
    return 0;
}
#undef GET
#undef PUT
#undef SYM_STEP_BODY
#undef FN
#undef CAT
#undef CAT2
