/*
 * Body of the serial CPU oracle, written once and instantiated for float and
 * double by bb_oracle.c (which defines REAL, SFX and the precision constants).
 *
 * TEST INFRASTRUCTURE ONLY: nothing on the product path may include, link or
 * call this file.  See bb_oracle.c for the citations and the readings taken.
 */

#define CAT2(a, b) a##b
#define CAT(a, b) CAT2(a, b)
#define FN(name) CAT(name, SFX)

/* Element type of the band storage; the arithmetic type is REAL.  They are
 * the same except in the half-precision storage instantiation, where every
 * read widens to REAL and every write rounds to the storage type. */
#ifndef BAND_T
#define BAND_T REAL
#define BAND_T_DEFAULTED_
#endif

/* Euclidean norm of x[0], x[inc], ..., x[(m-1)*inc]: plain sum of squares in
 * index order.  When that sum under- or overflows while the entries are
 * finite and not all zero, the same sum is taken on entries divided by the
 * largest magnitude, so that a norm of zero means every entry is zero. */
static REAL FN(norm2_)(int64_t m, const REAL* x, int64_t inc) {
    REAL ssq = 0;
    for (int64_t q = 0; q < m; ++q) {
        REAL v = x[q * inc];
        ssq = ssq + v * v;
    }
    if (isfinite(ssq) && ssq >= REAL_MIN_NORMAL) return SQRT(ssq);
    REAL scale = 0;
    for (int64_t q = 0; q < m; ++q) {
        REAL a = FABS(x[q * inc]);
        if (a > scale) scale = a;
    }
    if (scale == 0) return 0;
    REAL s2 = 0;
    for (int64_t q = 0; q < m; ++q) {
        REAL v = x[q * inc] / scale;
        s2 = s2 + v * v;
    }
    return scale * SQRT(s2);
}

/* Householder reflector in the LAPACK xLARFG convention.
 *   input : alpha = x_1, x = (x_2 .. x_w) (m = w-1 entries, stride inc)
 *   output: *alpha = beta, x overwritten by (v_2 .. v_w) (v_1 = 1), *tau
 * so that (I - tau v v^T) (alpha, x)^T = (beta, 0, ..., 0)^T.
 *   xi = ||x||;  xi == 0  ->  tau = 0, beta = alpha (identity, no sign flip)
 *   else beta = -sign(alpha) * hypot(alpha, xi) with sign(+-0) = +,
 *        tau = (beta - alpha) / beta,  v = x * (1 / (alpha - beta)).
 * A beta below safmin = tiny/eps is handled as LAPACK does: x and alpha are
 * scaled by 1/safmin (at most 20 times), beta recomputed, and scaled back. */
void FN(oracle_larfg)(int64_t m, REAL* alpha, REAL* x, int64_t inc, REAL* tau) {
    if (m <= 0) { *tau = 0; return; }
    REAL xnorm = FN(norm2_)(m, x, inc);
    if (xnorm == 0) { *tau = 0; return; }
    REAL a = *alpha;
    REAL beta = (a >= 0) ? -HYPOT(a, xnorm) : HYPOT(a, xnorm);
    const REAL safmin = REAL_SAFMIN;
    const REAL rsafmn = 1 / safmin;
    int knt = 0;
    if (FABS(beta) < safmin) {
        do {
            ++knt;
            for (int64_t q = 0; q < m; ++q) x[q * inc] = x[q * inc] * rsafmn;
            beta = beta * rsafmn;
            a = a * rsafmn;
        } while (FABS(beta) < safmin && knt < 20);
        xnorm = FN(norm2_)(m, x, inc);
        beta = (a >= 0) ? -HYPOT(a, xnorm) : HYPOT(a, xnorm);
    }
    *tau = (beta - a) / beta;
    REAL scal = 1 / (a - beta);
    for (int64_t q = 0; q < m; ++q) x[q * inc] = x[q * inc] * scal;
    for (int j = 0; j < knt; ++j) beta = beta * safmin;
    *alpha = beta;
}

/* ---------------------------------------------------------------------------
 * One bulge-chasing step on an abstract matrix accessor.  ELEM(i, j) is an
 * lvalue for A(i, j); the band and dense modes below instantiate it.
 *
 * Pass (b, t), b' = b - t; sweep r; step k:
 *   c  = r + b' + k b,  p = r (k = 0) or c - b (k > 0),  ce = min(c + t, n-1)
 *   right: reflector from A(p, c..ce); A(p, c) = beta, A(p, c+1..ce) = 0;
 *          rows i in (p, ce]:  y = sum_m A(i, c+m) v_m,  A(i, c+m) -= (tau y) v_m
 *   left : reflector from A(c..ce, c); A(c, c) = beta, A(c+1..ce, c) = 0;
 *          cols j in (c, min(ce + b, n-1)]:
 *                y = sum_m v_m A(c+m, j),  A(c+m, j) -= (tau y) v_m
 * In the dense mode the row / column ranges of the two applications are the
 * whole matrix instead of the windows above (entries outside the windows are
 * exactly zero, so the arithmetic inside the windows is the same).
 * ------------------------------------------------------------------------- */
/* RECORD(side, c, w, v, tau) is a no-op except in the recording driver below,
 * which keeps every reflector for the back-transformation. */
#define RECORD(side, c, w, v, tau) ((void)0)

#define STEP_BODY(ROW_LO, ROW_HI, COL_LO, COL_HI, DO_RIGHT, DO_LEFT)                    \
    do {                                                                                \
        int64_t c = r + (b - t) + k * b;                                                \
        int64_t p = (k == 0) ? r : c - b;                                               \
        int64_t ce = (c + t < n - 1) ? c + t : n - 1;                                   \
        int64_t cend = (ce + b < n - 1) ? ce + b : n - 1;                               \
        int64_t w = ce - c + 1;                                                         \
        REAL v[ORACLE_WMAX] = {0};                                                      \
        (void)cend;                                                            \
        REAL tau, beta;                                                                 \
        if (DO_RIGHT) {                                                                 \
            for (int64_t q = 0; q < w; ++q) v[q] = ELEM(p, c + q);                      \
            beta = v[0];                                                                \
            FN(oracle_larfg)(w - 1, &beta, v + 1, 1, &tau);                             \
            v[0] = 1;                                                                   \
            RECORD(0, c, w, v, tau);                                                    \
            ELEM(p, c) = beta;                                                          \
            for (int64_t q = 1; q < w; ++q) ELEM(p, c + q) = 0;                         \
            if (tau != 0) {                                                             \
                for (int64_t i = (ROW_LO); i <= (ROW_HI); ++i) {                        \
                    if (i == p) continue;                                               \
                    REAL y = 0;                                                         \
                    for (int64_t q = 0; q < w; ++q) y = y + ELEM(i, c + q) * v[q];      \
                    REAL s = tau * y;                                                   \
                    for (int64_t q = 0; q < w; ++q) ELEM(i, c + q) = ELEM(i, c + q) - s * v[q]; \
                }                                                                       \
            }                                                                           \
        }                                                                               \
        if (DO_LEFT) {                                                                  \
            for (int64_t q = 0; q < w; ++q) v[q] = ELEM(c + q, c);                      \
            beta = v[0];                                                                \
            FN(oracle_larfg)(w - 1, &beta, v + 1, 1, &tau);                             \
            v[0] = 1;                                                                   \
            RECORD(1, c, w, v, tau);                                                    \
            ELEM(c, c) = beta;                                                          \
            for (int64_t q = 1; q < w; ++q) ELEM(c + q, c) = 0;                         \
            if (tau != 0) {                                                             \
                for (int64_t j = (COL_LO); j <= (COL_HI); ++j) {                        \
                    if (j == c) continue;                                               \
                    REAL y = 0;                                                         \
                    for (int64_t q = 0; q < w; ++q) y = y + v[q] * ELEM(c + q, j);      \
                    REAL s = tau * y;                                                   \
                    for (int64_t q = 0; q < w; ++q) ELEM(c + q, j) = ELEM(c + q, j) - s * v[q]; \
                }                                                                       \
            }                                                                           \
        }                                                                               \
    } while (0)

/* Band mode: A(i, j) lives at band[(ku + i - j) + j * ldab]. */
#define ELEM(i, j) band[(ku + (i) - (j)) + (j) * ldab]

/* One half-step (side 0 = right/horizontal, 1 = left/vertical) of sweep r,
 * step k of the pass (b, t), windows exactly as in STEP_BODY. */
void FN(oracle_halfstep_band)(int64_t n, int64_t b, int64_t t, int64_t ku, BAND_T* band, int64_t ldab,
                              int64_t r, int64_t k, int side) {
    if (side == 0) STEP_BODY(p, ce, c, cend, 1, 0);
    else           STEP_BODY(p, ce, c, cend, 0, 1);
}

/* Number of steps of sweep r in pass (b, t): k runs while c_k + 1 <= n - 1. */
int64_t FN(oracle_sweep_steps)(int64_t n, int64_t b, int64_t t, int64_t r) {
    int64_t last = n - 2 - r - (b - t);
    return last < 0 ? 0 : last / b + 1;
}

/* Whole reduction in band storage, serial order: for each pass of the plan
 * (b = bw; while b > 1: t = min(tw, b - 1); pass (b, t); b -= t), for each
 * sweep r ascending, for each step k ascending: right, then left.
 * Passes with index outside [pass_lo, pass_hi) are skipped (bandwidth still
 * advances), so that a run can be split at pass boundaries.
 * The fill rows 0..tw-1 and ku+1..ku+tw of every column are zeroed first when
 * pass_lo == 0.  Returns 0, or -1 on invalid arguments. */
int FN(oracle_reduce_band)(int64_t n, int64_t bw, int64_t tw, BAND_T* band, int64_t ldab,
                           int64_t pass_lo, int64_t pass_hi) {
    if (n < 1 || bw < 0 || bw >= n || tw < 1 || ldab < bw + 2 * tw + 1) return -1;
    if (tw > (bw > 2 ? bw - 1 : 1)) return -1;
    if (tw + 1 > ORACLE_WMAX) return -1;
    int64_t ku = bw + tw;
    if (pass_lo == 0) {
        for (int64_t j = 0; j < n; ++j) {
            for (int64_t q = 0; q < tw; ++q) band[q + j * ldab] = 0;
            for (int64_t q = ku + 1; q <= ku + tw; ++q) band[q + j * ldab] = 0;
        }
    }
    int64_t b = bw, pass = 0;
    while (b > 1) {
        int64_t t = (tw < b - 1) ? tw : b - 1;
        if (pass >= pass_lo && pass < pass_hi) {
            for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r) {
                int64_t K = FN(oracle_sweep_steps)(n, b, t, r);
                for (int64_t k = 0; k < K; ++k) STEP_BODY(p, ce, c, cend, 1, 1);
            }
        }
        b -= t;
        ++pass;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Pipelined sweeps on P host threads ("A two-stage reduction on an Apple M5
 * Pro", Section 6, the multi-threaded band chase): sweep r runs on thread
 * r mod P, every sweep publishes how many of its half-steps are finished, and
 * the next sweep spins on that count.  All P threads run at once (a sweep
 * waits only on its predecessor, which belongs to another running thread, or
 * to its own thread and is then finished), so nothing deadlocks.
 *
 * Dependency rule, the half-step form of the sweep separation: half-step h
 * (right of step k = 2k, left = 2k+1) of sweep r starts once sweep r-1 has
 * finished min(h + L, H_{r-1}) half-steps, with L = 2 when b - t >= 3, 3 when
 * b - t == 2 and 4 when b - t == 1 (H_r = 2 x steps of sweep r); the last
 * half-step of a sweep waits for all of sweep r-1.  Each half-step is
 * oracle_halfstep_band, so the result is the serial one bitwise as long as
 * the rule keeps every pair of overlapping half-steps in sweep order.  The
 * passes are separated by joining the threads.
 *
 * Counters are C11 atomics, stored with release and loaded with acquire, so
 * a sweep sees every write of the half-steps it waited for.  Every wait gives
 * up after time_limit_s seconds of wall clock for the whole call (then all
 * threads stop and -2 is returned).
 * ------------------------------------------------------------------------- */
typedef struct {
    int64_t n, b, t, ku, ldab, nthreads, thread;
    BAND_T* band;
    _Atomic int64_t* done;
    _Atomic int* stop;
    double deadline;
} FN(pipe_arg_);

static int FN(pipe_wait_)(_Atomic int64_t* count, int64_t need, const FN(pipe_arg_)* a) {
    uint64_t spins = 0;
    while (atomic_load_explicit(count, memory_order_acquire) < need) {
        if (atomic_load_explicit(a->stop, memory_order_relaxed)) return 0;
        if ((++spins & 0x3FF) == 0) {
            if (oracle_now_() > a->deadline) {
                atomic_store_explicit(a->stop, 1, memory_order_relaxed);
                return 0;
            }
            sched_yield();
        }
    }
    return 1;
}

static void* FN(pipe_worker_)(void* arg) {
    const FN(pipe_arg_)* a = (const FN(pipe_arg_)*)arg;
    const int64_t n = a->n, b = a->b, t = a->t;
    const int64_t L = (b - t >= 3) ? 2 : ((b - t == 2) ? 3 : 4);
    const int64_t nsweeps = n - (b - t) - 1;
    for (int64_t r = a->thread; r < nsweeps; r += a->nthreads) {
        const int64_t H = 2 * FN(oracle_sweep_steps)(n, b, t, r);
        const int64_t Hp = (r > 0) ? 2 * FN(oracle_sweep_steps)(n, b, t, r - 1) : 0;
        for (int64_t h = 0; h < H; ++h) {
            if (r > 0) {
                int64_t need = (h + L < Hp) ? h + L : Hp;
                if (h == H - 1) need = Hp;
                if (!FN(pipe_wait_)(&a->done[r - 1], need, a)) return NULL;
            }
            FN(oracle_halfstep_band)(n, b, t, a->ku, a->band, a->ldab, r, h >> 1, (int)(h & 1));
            atomic_store_explicit(&a->done[r], h + 1, memory_order_release);
        }
    }
    return NULL;
}

/* The reduction as oracle_reduce_band (all passes, same arithmetic and
 * order), also keeping every reflector H = I - tau v v^T in the order applied:
 * for reflector q, side[q] = 0 for a right one (A <- A H on columns
 * start[q] .. start[q] + width[q] - 1) or 1 for a left one (A <- H A on those
 * rows), tau[q], and v at vs[q * (tw + 1) + 0 .. width[q] - 1] (v_0 = 1).
 * With B the result, A = U B V^T where U = L_1 L_2 ... (the left reflectors
 * in order) and V = R_1 R_2 ... (the right ones): the back-transformation
 * that gives the singular vectors ("Accelerating Bidiagonalization of Banded
 * Matrices through Memory-Aware Bulge-Chasing on GPUs", Section III: the
 * reflector vectors are written back for it).  cap is the room for
 * reflectors.  Returns the number recorded, -1 on invalid arguments, -2 when
 * cap is too small. */
int64_t FN(oracle_reduce_band_record)(int64_t n, int64_t bw, int64_t tw, BAND_T* band, int64_t ldab, int64_t cap,
                                      int8_t* side, int64_t* start, int32_t* width, REAL* taus, REAL* vs) {
    if (n < 1 || bw < 0 || bw >= n || tw < 1 || ldab < bw + 2 * tw + 1) return -1;
    if (tw > (bw > 2 ? bw - 1 : 1)) return -1;
    if (tw + 1 > ORACLE_WMAX || cap < 0) return -1;
    const int64_t ku = bw + tw;
    for (int64_t j = 0; j < n; ++j) {
        for (int64_t q = 0; q < tw; ++q) band[q + j * ldab] = 0;
        for (int64_t q = ku + 1; q <= ku + tw; ++q) band[q + j * ldab] = 0;
    }
    int64_t nrec = 0;
#undef RECORD
#define RECORD(SIDE, C, W, V, TAU)                                                     \
    do {                                                                               \
        if (nrec < cap) {                                                              \
            side[nrec] = (int8_t)(SIDE);                                               \
            start[nrec] = (C);                                                         \
            width[nrec] = (int32_t)(W);                                                \
            taus[nrec] = (TAU);                                                        \
            for (int64_t u_ = 0; u_ < (W); ++u_) vs[nrec * (tw + 1) + u_] = (V)[u_];    \
        }                                                                              \
        ++nrec;                                                                        \
    } while (0)
    int64_t b = bw;
    while (b > 1) {
        int64_t t = (tw < b - 1) ? tw : b - 1;
        for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r) {
            int64_t K = FN(oracle_sweep_steps)(n, b, t, r);
            for (int64_t k = 0; k < K; ++k) STEP_BODY(p, ce, c, cend, 1, 1);
        }
        b -= t;
    }
#undef RECORD
#define RECORD(side, c, w, v, tau) ((void)0)
    return nrec <= cap ? nrec : -2;
}

/* Runs every pass of the plan on nthreads threads with `worker` (the
 * bidiagonal or the symmetric one), joining the threads between passes.
 * Returns 0, -2 when the time limit ran out, -3 when the threads or the
 * counters could not be created. */
static int FN(pipe_run_)(int64_t n, int64_t bw, int64_t tw, BAND_T* band, int64_t ldab, int64_t nthreads,
                         double time_limit_s, void* (*worker)(void*), int64_t pass_lo, int64_t pass_hi) {
    const int64_t ku = bw + tw;
    _Atomic int64_t* done = (_Atomic int64_t*)malloc((size_t)n * sizeof(_Atomic int64_t));
    pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
    FN(pipe_arg_)* args = (FN(pipe_arg_)*)malloc((size_t)nthreads * sizeof(FN(pipe_arg_)));
    _Atomic int stop;
    atomic_init(&stop, 0);
    int rc = 0;
    if (!done || !th || !args) rc = -3;
    const double deadline = oracle_now_() + time_limit_s;
    int64_t b = bw;
    for (int64_t pass = 0; rc == 0 && b > 1; ++pass) {
        const int64_t t = (tw < b - 1) ? tw : b - 1;
        if (pass < pass_lo || pass >= pass_hi) {  /* skipped: the bandwidth still follows the plan */
            b -= t;
            continue;
        }
        const int64_t nsweeps = n - (b - t) - 1;
        for (int64_t r = 0; r < n; ++r) atomic_init(&done[r], 0);
        int64_t P = nthreads < nsweeps ? nthreads : nsweeps, started = 0;
        for (int64_t q = 0; q < P; ++q) {
            args[q] = (FN(pipe_arg_)){n, b, t, ku, ldab, P, q, band, done, &stop, deadline};
            if (pthread_create(&th[q], NULL, worker, &args[q]) != 0) {
                atomic_store_explicit(&stop, 1, memory_order_relaxed);
                rc = -3;
                break;
            }
            ++started;
        }
        for (int64_t q = 0; q < started; ++q) pthread_join(th[q], NULL);
        if (rc == 0 && atomic_load_explicit(&stop, memory_order_relaxed)) rc = -2;
        b -= t;
    }
    free(done);
    free(th);
    free(args);
    return rc;
}

/* Same arguments and result as oracle_reduce_band over passes [pass_lo,
 * pass_hi) of the plan (the fill rows are zeroed only when pass_lo == 0), on
 * nthreads (1 .. 1024) threads.  Returns 0; -1 on invalid arguments; -2 when
 * time_limit_s ran out (the band is then partly reduced); -3 when the
 * threads or the counters could not be created. */
int FN(oracle_reduce_band_pipelined_range)(int64_t n, int64_t bw, int64_t tw, BAND_T* band, int64_t ldab,
                                           int64_t nthreads, double time_limit_s, int64_t pass_lo,
                                           int64_t pass_hi) {
    if (n < 1 || bw < 0 || bw >= n || tw < 1 || ldab < bw + 2 * tw + 1) return -1;
    if (tw > (bw > 2 ? bw - 1 : 1)) return -1;
    if (tw + 1 > ORACLE_WMAX) return -1;
    if (nthreads < 1 || nthreads > 1024 || !(time_limit_s > 0)) return -1;
    const int64_t ku = bw + tw;
    if (pass_lo == 0) {
        for (int64_t j = 0; j < n; ++j) {
            for (int64_t q = 0; q < tw; ++q) band[q + j * ldab] = 0;
            for (int64_t q = ku + 1; q <= ku + tw; ++q) band[q + j * ldab] = 0;
        }
    }
    return FN(pipe_run_)(n, bw, tw, band, ldab, nthreads, time_limit_s, FN(pipe_worker_), pass_lo, pass_hi);
}

/* All passes (oracle_reduce_band_pipelined_range over the whole plan). */
int FN(oracle_reduce_band_pipelined)(int64_t n, int64_t bw, int64_t tw, BAND_T* band, int64_t ldab,
                                     int64_t nthreads, double time_limit_s) {
    return FN(oracle_reduce_band_pipelined_range)(n, bw, tw, band, ldab, nthreads, time_limit_s, 0, INT64_MAX);
}

/* d_i = A(i, i), e_i = A(i, i+1) from band storage. */
void FN(oracle_extract_band)(int64_t n, int64_t ku, const BAND_T* band, int64_t ldab, REAL* d, REAL* e) {
    for (int64_t i = 0; i < n; ++i) d[i] = ELEM(i, i);
    for (int64_t i = 0; i + 1 < n; ++i) e[i] = ELEM(i, i + 1);
}
#undef ELEM

/* Dense mode: A is n x n, row-major, A(i, j) = a[i * n + j].  Each reflector
 * is applied to every row (right) or every column (left) of the matrix, which
 * is the definition of A <- A H and A <- H A; the band windows play no part.
 * Same pass plan and serial order as the band mode. */
#define ELEM(i, j) a[(i) * n + (j)]
int FN(oracle_reduce_dense)(int64_t n, int64_t bw, int64_t tw, REAL* a) {
    if (n < 1 || bw < 0 || bw >= n || tw < 1) return -1;
    if (tw > (bw > 2 ? bw - 1 : 1)) return -1;
    if (tw + 1 > ORACLE_WMAX) return -1;
    int64_t b = bw;
    while (b > 1) {
        int64_t t = (tw < b - 1) ? tw : b - 1;
        for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r) {
            int64_t K = FN(oracle_sweep_steps)(n, b, t, r);
            for (int64_t k = 0; k < K; ++k) STEP_BODY(0, n - 1, 0, n - 1, 1, 1);
        }
        b -= t;
    }
    return 0;
}
#undef ELEM

#undef RECORD
#undef FN
#undef CAT
#undef CAT2
#ifdef BAND_T_DEFAULTED_
#undef BAND_T
#undef BAND_T_DEFAULTED_
#endif
