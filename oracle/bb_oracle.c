/*
 * Serial CPU oracle for the reduction of an upper-banded matrix to upper
 * bidiagonal form by Householder bulge chasing.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow reference that the
 * GPU library is checked against.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may build, load or call it.  It shares no
 * code, header or table with the CUDA library, and the library never calls it.
 *
 * What it computes follows "Accelerating Bidiagonalization of Banded Matrices
 * through Memory-Aware Bulge-Chasing on GPUs" (arXiv 2510.12705):
 *   - Section III (bulge-chasing sweeps): a sweep for row R annihilates one
 *     horizontal group of TW entries of a row and then one vertical group in
 *     the leftmost column of the bulge that creates, and moves BW columns to
 *     the right per cycle; each pass lowers the bandwidth from BW to BW - TW
 *     ("successive band reduction"), repeated down to bidiagonal form.
 *   - Algorithm 2 text: the TW entries to annihilate plus the one to their
 *     left form the reflector input; the reflector is applied to the row
 *     block (rows of width TW+1) and then the same is done for the column.
 *   - The Householder construction follows tile-QR prior work; it is read
 *     here as LAPACK's xLARFG convention (beta = -sign(alpha) ||x||,
 *     tau = (beta - alpha) / beta, v_1 = 1, annihilated entries set to 0).
 * The listings themselves (Algorithms 1 and 2) are not available; the window
 * indices in bb_oracle_body.h are the plainest reading consistent with the
 * text: the data touched in one cycle spans rows R .. R+BW+TW and the same
 * number of columns, and the first cycle of a sweep touches fewer rows.
 *
 * Arithmetic is in the working precision of the instantiation (float or
 * double), in the index order written, compiled without contraction of
 * multiply-add pairs (-ffp-contract=off) so that runs are reproducible.
 *
 * Parity pins (in tests/): dense mode == band mode bitwise; the dense result
 * is exactly bidiagonal; Frobenius norm and singular values (against a
 * brute-force Jacobi SVD) are preserved; |d|, |e| agree with a textbook dense
 * Golub-Kahan bidiagonalisation; larfg agrees with LAPACK's slarfg/dlarfg;
 * any schedule that respects the sweep dependencies gives the serial result
 * bitwise (also when run on host threads by oracle_reduce_band_pipelined);
 * power-of-two scaling commutes bitwise; diagonal and zero inputs.
 *
 * sb_oracle_body.h adds the symmetric variant (symmetric band -> tridiagonal
 * by the same passes, one two-sided reflector per step), pinned the same way
 * against LAPACK's dsytrd and eigenvalues.
 */
#define _POSIX_C_SOURCE 200809L
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <time.h>

#define ORACLE_WMAX 129 /* tw <= 128 */

/* wall clock in seconds, for the pipelined driver's time limit */
static double oracle_now_(void) {
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec + 1e-9 * (double)ts.tv_nsec;
}

/* double instantiation */
#define REAL double
#define SFX _d
#define SQRT sqrt
#define FABS fabs
#define HYPOT hypot
#define REAL_MIN_NORMAL DBL_MIN
#define REAL_SAFMIN (DBL_MIN / (DBL_EPSILON * 0.5))
#include "bb_oracle_body.h"
#include "sb_oracle_body.h"
#undef REAL
#undef SFX
#undef SQRT
#undef FABS
#undef HYPOT
#undef REAL_MIN_NORMAL
#undef REAL_SAFMIN
#undef STEP_BODY

/* float instantiation */
#define REAL float
#define SFX _f
#define SQRT sqrtf
#define FABS fabsf
#define HYPOT hypotf
#define REAL_MIN_NORMAL FLT_MIN
#define REAL_SAFMIN (FLT_MIN / (FLT_EPSILON * 0.5f))
#include "bb_oracle_body.h"
#include "sb_oracle_body.h"
#undef STEP_BODY

/* half-precision storage, float arithmetic (suffix _h): the band is IEEE
 * binary16; every half-step reads its entries into float, forms and applies
 * the reflector in float, and rounds each entry it writes to binary16 (round
 * to nearest even).  Built where the compiler has _Float16. */
#ifdef __FLT16_MANT_DIG__
#undef SFX
#define SFX _h
#define BAND_T _Float16
#include "bb_oracle_body.h"
#undef STEP_BODY
#undef BAND_T
int oracle_has_half(void) { return 1; }
#else
int oracle_has_half(void) { return 0; }
#endif
