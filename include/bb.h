/*
 * bb.h -- C ABI of the GB300 band -> bidiagonal reduction library (libbb.so).
 *
 * The library performs the second stage of a two-stage SVD: it reduces an
 * upper-banded n x n matrix of bandwidth bw to upper bidiagonal form (main
 * diagonal d, superdiagonal e) by Householder bulge chasing, as described in
 * "Accelerating Bidiagonalization of Banded Matrices through Memory-Aware
 * Bulge-Chasing on GPUs" (arXiv 2510.12705), Section III:
 *   - successive band reduction: each pass lowers the bandwidth from b to
 *     b - t by annihilating t entries per reflector; passes repeat until the
 *     bandwidth is 1 (plan: b = bw; while b > 1 { t = min(tw, b - 1); b -= t });
 *   - within a pass, sweep r annihilates t entries of row r, then chases the
 *     bulge down the band, one horizontal and one vertical reflector per
 *     cycle, moving b columns per cycle;
 *   - consecutive sweeps run concurrently, separated by the cycle lag that
 *     keeps their data windows disjoint (the paper's three-cycle rule).
 * Reflectors follow the LAPACK xLARFG convention (beta = -sign(alpha)||x||,
 * tau = (beta - alpha)/beta, v_1 = 1; annihilated entries become exactly 0),
 * the reading taken of the paper's tile-QR reference.  Results are therefore
 * defined up to the signs of d and e; |d| and |e| are unique.
 *
 * Storage (all pointers below are device pointers unless stated otherwise):
 *   compact column-major band storage with fill rows, LAPACK "gb" style with
 *   ku = bw + tw upper and kl = tw lower diagonals:
 *       A(i, j) = band[(ku + i - j) + j * ldab],   0 <= i, j < n
 *   The input band occupies band rows tw .. tw + bw (0 <= j - i <= bw); band
 *   rows 0 .. tw-1 and ku+1 .. ku+tw hold the bulge fill and are zeroed by
 *   bb_reduce.  ldab >= bw + 2*tw + 1.  Rows beyond ku + tw are not touched.
 *
 * Threading: a handle may be used by one host thread at a time, with at most
 * one reduction in flight (bb_reduce, bb_reduce_host, bb_sym_reduce or
 * bb_back_transform: they share the handle's progress counters, status
 * word and working band).  All calls are asynchronous on the given stream
 * unless stated otherwise.
 */
#ifndef BB_H_
#define BB_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the band, d and e.  BB_F16: IEEE binary16 storage with
 * float arithmetic -- every step reads its entries into float, builds and
 * applies its reflectors in float, and writes every entry it changes back
 * rounded to binary16 (round to nearest even); d and e are binary16 too.
 * The paper runs the method in FP16 as well (Section V).  BB_F16 handles
 * run each pass on the group kernel with binary16 columns in shared memory
 * (where BB_PARAM_SCHEDULER 0 or 3 picks it, by the rule of bb_reduce, for
 * reflectors of up to 33 elements; on a band whose column stride is not a
 * multiple of 16 bytes through an aligned working copy) or on the binary16
 * flag kernel (every other pass, and every pass under schedulers 1, 2 and
 * 4); both give bitwise equal results.  They are accepted by bb_create,
 * bb_reduce, bb_reduce_host and bb_status_sync only. */
typedef enum { BB_F32 = 0, BB_F64 = 1, BB_F16 = 2 } bb_dtype;

/* Return codes. */
typedef enum {
    BB_OK = 0,
    BB_ERR_INVALID_ARG = 1, /* a size, pointer or parameter is out of range     */
    BB_ERR_LDAB = 2,        /* ldab < bw + 2*tw + 1                              */
    BB_ERR_DTYPE = 3,       /* dtype unknown                                     */
    BB_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed       */
    BB_ERR_TIMEOUT = 5,     /* a device-side wait gave up (latched on the device) */
    BB_ERR_NOMEM = 6,       /* a device or host allocation failed                */
    BB_ERR_INTERNAL = 7     /* a device-side consistency check failed (a bug)    */
} bb_status;

/* A cudaStream_t, passed as a plain pointer (NULL = the legacy default stream). */
typedef void* bb_stream_t;

/* Opaque handle: owns the per-sweep progress counters (n int32; the group
 * kernel keeps one watermark per group there), a device status word, and,
 * once needed, staging buffers (bb_reduce_host) and a working copy of the
 * band (see BB_PARAM_SCHEDULER). */
typedef struct bb_handle bb_handle;

/* Create a handle for n x n matrices of upper bandwidth bw (0 <= bw < n) and
 * element type dtype, on the current CUDA device.  Allocates device memory.
 * Returns NULL on error; bb_last_error() says why. */
bb_handle* bb_create(int64_t n, int64_t bw, bb_dtype dtype);

/* Reduce the band in place to bidiagonal form and write d (n entries) and e
 * (n-1 entries).  band_ptr, d_out and e_out are device pointers owned by the
 * caller; band_ptr holds ldab * n elements and is overwritten (destroyed).
 * tw: entries annihilated per reflector, 1 <= tw <= max(1, bw - 1), tw <= 64.
 * Stream-ordered and asynchronous: the return code covers argument checks and
 * launch errors only.  A device-side failure (a progress wait that ran out of
 * its budget, or BB_ERR_INTERNAL from a consistency check) is latched in the
 * handle's status word and reported by bb_status_sync.  When a pass runs on
 * the group kernel and the band's base or column stride is not a multiple of
 * 16 bytes, the first such call allocates the handle's working copy (n x ldab
 * rounded up to 16 bytes; BB_ERR_NOMEM if that fails).  No C++ exception
 * leaves the library: a failed host allocation is BB_ERR_NOMEM.  Covers the
 * paper's Algorithms 1 and 2 (Section III). */
bb_status bb_reduce(bb_handle* h, void* band_ptr, int64_t ldab, int64_t tw, void* d_out,
                    void* e_out, bb_stream_t stream);

/* Same as bb_reduce with HOST buffers: copies band_host (ldab * n elements,
 * not modified) to a device staging buffer owned by the handle, reduces it,
 * copies d and e back to d_host / e_host, and synchronizes the stream before
 * returning (so device-side failures are reported here too).  Pinned host
 * memory gives the fastest copies.  The first call allocates the staging
 * buffers (kept until bb_destroy). */
bb_status bb_reduce_host(bb_handle* h, const void* band_host, int64_t ldab, int64_t tw,
                         void* d_host, void* e_host, bb_stream_t stream);

/* Free the handle and everything it owns.  NULL is ignored. */
void bb_destroy(bb_handle* h);

/* Smallest valid ldab: bw + 2*tw + 1. */
int64_t bb_required_ldab(int64_t bw, int64_t tw);

/* Synchronize the stream, then return and clear the handle's device status
 * word: BB_OK, or BB_ERR_TIMEOUT if a wait in an earlier bb_reduce gave up
 * (its results are then invalid). */
bb_status bb_status_sync(bb_handle* h, bb_stream_t stream);

/* Tuning and test parameters (bb_set_param / bb_get_param). */
enum {
    BB_PARAM_SCHEDULER = 0,     /* 0: automatic (default): per pass, the group kernel
                                      where at least 5 sweeps' columns fit shared
                                      memory, else the flag kernel;
                                   1: one kernel launch per cycle;
                                   2: persistent flag kernel (one CTA per sweep, per-
                                      sweep progress counters) for every pass;
                                   3: group kernel (CTA per group of sweeps, columns in
                                      shared memory) wherever one sweep fits, else 2;
                                   4: as 1, with each pass's launches captured once in
                                      a CUDA graph (on a stream of the handle) and
                                      replayed on the caller's stream; the graph is
                                      kept by the handle and captured again when the
                                      band pointer, ldab or the pass changes.
                                   The group kernel moves columns with 16-byte bulk
                                   copies: on a band whose base or column stride
                                   (ldab * element size) is not a multiple of 16
                                   bytes, bb_reduce runs it on a working copy
                                   (allocated by the handle on first use, n x ldab
                                   rounded up; copied in and back on the stream)   */
    BB_PARAM_TPB = 1,           /* threads per block, multiple of 32 in [32, 1024];
                                   0 = automatic (default).  With MAX_CTAS, the
                                   "Threads per block" and "Max blocks" of the
                                   hyperparameter study of "Accelerating
                                   Bidiagonalization of Banded Matrices through
                                   Memory-Aware Bulge-Chasing on GPUs", Section V-B
                                   (its third, the inner tile width, is tw)        */
    BB_PARAM_MAX_CTAS = 2,      /* cap on the persistent grid; 0 = co-resident maximum  */
    BB_PARAM_WAIT_BUDGET_MS = 3,/* bound of one device-side wait, in ms (default 4000)  */
    BB_PARAM_PASS_LO = 4,       /* run only passes [PASS_LO, PASS_HI) (default 0 .. all); */
    BB_PARAM_PASS_HI = 5,       /*   the fill rows are zeroed only when PASS_LO == 0    */
    BB_PARAM_STALL_SWEEP = 6,   /* fault injection: the CTA running this sweep of every
                                   pass never reports progress (-1 = off, default)      */
    BB_PARAM_TIMING = 7,        /* 1: record CUDA events around every pass launch, read
                                   back with bb_last_pass_ms (default 0)                */
    BB_PARAM_GROUP_SIZE = 8,    /* sweeps per group of the group kernel: 0 = largest
                                   that fits shared memory, at most 13, or 5 when a
                                   reflector of tw + 1 elements takes more than 68
                                   bytes (default)                                      */
    BB_PARAM_RECORD = 9         /* 1: keep every reflector of the next whole reductions
                                   (all passes) for bb_back_transform; the passes then
                                   run on the flag kernel (scheduler 2) and the handle
                                   holds 2 x steps x (tw + 1) + 2 x steps elements of
                                   device memory (default 0)                            */
};
bb_status bb_set_param(bb_handle* h, int param, int64_t value);
int64_t bb_get_param(const bb_handle* h, int param);

/* Symmetric variant: reduce a symmetric band matrix to symmetric tridiagonal
 * form with the same passes BW -> BW - TW, one two-sided Householder
 * reflector per step (the band to tridiagonal chase of "A two-stage
 * reduction on an Apple M5 Pro", Section 6, with the passes of
 * "Accelerating Bidiagonalization of Banded Matrices through Memory-Aware
 * Bulge-Chasing on GPUs", Section III).
 *   h        handle from bb_create(n, bw, dtype) (n, bw, dtype as there)
 *   band_ptr device, LAPACK lower band storage, column-major: A(i, j) for
 *            0 <= i - j <= bw at band[(i - j) + j * ldab]; rows bw+1 ..
 *            bw+tw of each column are fill space (zeroed here).  Reduced in
 *            place; on return the rows below the subdiagonal are zero.
 *   ldab     >= bb_sym_required_ldab(bw, tw) = bw + tw + 1 (else BB_ERR_LDAB)
 *   tw       1 <= tw <= max(1, bw - 1), tw <= 64
 *   d_out    device, n entries: the diagonal; e_out device, n - 1 entries:
 *            the subdiagonal (may be null when n == 1)
 * Stream-ordered and asynchronous like bb_reduce.  Schedulers, per pass
 * (BB_PARAM_SCHEDULER; BB_PARAM_GROUP_SIZE, BB_PARAM_MAX_CTAS,
 * BB_PARAM_WAIT_BUDGET_MS and BB_PARAM_STALL_SWEEP apply as for bb_reduce):
 *   flag kernel: one CTA per sweep with the handle's progress counters (step
 *     k of sweep r after sweep r-1 finished min(k + L, its steps), L = 2, or
 *     3 when b - t = 1);
 *   group kernel: g sweeps per CTA in lockstep with the same lag, their
 *     columns in shared memory (bb_sym_group_plan); it takes a pass with a
 *     reflector of at most 33 elements on a band whose base and ldab *
 *     element size are multiples of 16 bytes: under scheduler 0 (default)
 *     where at least 3 sweeps fit (float) or 5 (double), under 3 wherever
 *     one fits; every other
 *     pass, and every pass under schedulers 1, 2 and 4, runs on the flag
 *     kernel.
 * Both give bitwise equal results; bb_last_pass_kernel / bb_last_pass_group
 * report the choice (2 or 3) per pass.  Device-side failures are reported
 * by bb_status_sync. */
bb_status bb_sym_reduce(bb_handle* h, void* band_ptr, int64_t ldab, int64_t tw, void* d_out, void* e_out,
                        bb_stream_t stream);
int64_t bb_sym_required_ldab(int64_t bw, int64_t tw);
/* Back-transformation of the last whole reduction run with BB_PARAM_RECORD:
 * U = L_1 L_2 ... and V = R_1 R_2 ..., the products of the left and right
 * reflectors in the order applied, so that A = U B V^T with B the bidiagonal
 * (d, e).  U and V are device, column-major n x n (leading dimensions ldu,
 * ldv >= n), the handle's element type; either may be null to skip it.  The
 * singular vectors of A are then U U_b and V V_b for B = U_b S V_b^T.  Both
 * are formed from the identity, one launch per sweep and matrix (the
 * reflectors of a sweep act on disjoint columns and run at once).
 * Asynchronous on `stream`.  BB_ERR_INVALID_ARG without such a reduction on
 * this handle, or for bad arguments. */
bb_status bb_back_transform(bb_handle* h, void* U, int64_t ldu, void* V, int64_t ldv, bb_stream_t stream);

/* Pass plan of (bw, tw) (b = bw; while b > 1: t = min(tw, b - 1); b -= t):
 * the number of passes, ceil((bw - 1) / tw), and the (b, t) of pass i,
 * b = bw - i tw, t = min(tw, b - 1).  Host-only and computed in closed form;
 * bb_num_passes returns 0 when bw <= 1, tw < 1 or bw > 2^30, and
 * bb_pass_info BB_ERR_INVALID_ARG for an index outside the plan. */
int64_t bb_num_passes(int64_t bw, int64_t tw);
bb_status bb_pass_info(int64_t bw, int64_t tw, int64_t i, int64_t* b, int64_t* t);

/* Group-kernel plan of pass `pass` of an n x n reduction (element size
 * elem_bytes: 4 or 8, or 2 for binary16 storage, whose group kernel takes
 * reflectors of up to 33 elements): the sweeps per group g (0 when the group
 * kernel cannot take the pass), the columns of its shared-memory buffer (nslot),
 * the loader's run-ahead in ticks, and the rows a buffered column holds
 * (lds).  group_size as BB_PARAM_GROUP_SIZE (0 = the largest that fits).
 * Host-only, for inspection and tests.  BB_ERR_INVALID_ARG unless
 * 1 <= n < 2^30, 0 <= bw < n, 1 <= tw <= max(1, bw - 1), the pass is in the
 * plan, elem_bytes is 2, 4 or 8 and group_size >= 0. */
bb_status bb_group_plan(int64_t n, int64_t bw, int64_t tw, int64_t elem_bytes, int64_t pass, int64_t group_size,
                        int64_t* g, int64_t* nslot, int64_t* ahead, int64_t* lds);

/* As bb_group_plan, for the symmetric chase of bb_sym_reduce (lower band
 * storage, one two-sided step per tick): g = 0 when its group kernel cannot
 * take the pass (no group fits shared memory, or a reflector of more than 33
 * elements).  Same arguments and errors. */
bb_status bb_sym_group_plan(int64_t n, int64_t bw, int64_t tw, int64_t elem_bytes, int64_t pass,
                            int64_t group_size, int64_t* g, int64_t* nslot, int64_t* ahead, int64_t* lds);

/* Algorithmic bytes of pass i (or of all passes when i < 0) of an n x n
 * reduction with element size elem_bytes: every element of each step's right
 * block (rows p..ce x cols c..ce) and left block (rows c..ce x cols c..cend)
 * counted once read and once written.  This is the traffic model behind the
 * effective GB/s figure. */
double bb_model_bytes(int64_t n, int64_t bw, int64_t tw, int64_t elem_bytes, int64_t pass);

/* Number of steps (one horizontal plus one vertical reflector each) of pass
 * i (all passes when i < 0). */
int64_t bb_model_steps(int64_t n, int64_t bw, int64_t tw, int64_t pass);

/* Kernel launches made by the last bb_reduce / bb_reduce_host on this handle
 * (fill-row zeroing, the passes, and the d/e extraction). */
int64_t bb_last_launches(const bb_handle* h);

/* Kernel that ran pass i of the last reduction: 1 per-cycle, 2 flag kernel,
 * 3 group kernel (for BB_F16 handles: with binary16 columns), 4 per-cycle
 * launches replayed from a CUDA graph, 5 the binary16 flag kernel (-1 if out
 * of range), and, for the group kernel,
 * its group size (sweeps per CTA; 0 otherwise).  With scheduler 4, bb_last_launches counts the kernels the
 * graphs ran. */
int64_t bb_last_pass_kernel(const bb_handle* h, int64_t i);
int64_t bb_last_pass_group(const bb_handle* h, int64_t i);

/* With BB_PARAM_TIMING on: after the stream of the last bb_reduce has been
 * synchronized, the number of passes it ran and the device time of pass i in
 * milliseconds (CUDA events recorded on the launching stream around the
 * pass's kernel launches).  Returns BB_ERR_INVALID_ARG if i is out of range
 * or timing was off. */
int64_t bb_last_num_passes(const bb_handle* h);
bb_status bb_last_pass_ms(bb_handle* h, int64_t i, double* ms);

/* Message of the last error on the calling thread ("" if none). */
const char* bb_last_error(void);

/* The whole reduction without allocating device memory (the paper has no
 * counterpart; this is a library convenience).  For callers that cannot
 * allocate when they need the reduction: their device memory belongs to
 * another allocator or a fixed pool, or they cannot afford cudaMalloc /
 * cudaFree there (cudaFree synchronizes the device; both can stall or fail
 * under a memory budget).  bb_create allocates, so those callers use this
 * instead.  The caller passes the band (ldab * n elements, overwritten) and
 * d_out (n) / e_out (n-1), all device pointers, with the same meaning and
 * limits as bb_reduce, plus n <= 65536.  Larger n is rejected with
 * BB_ERR_INVALID_ARG and nothing is launched.
 * Scratch: the persistent scheduler's progress counters and status word live
 * in a fixed array of the library's device image (65536 + 64 int32, held by
 * every device that loads the library until the process exits).  The first
 * call on a device looks up that array's device address (cudaGetSymbolAddress)
 * with the device current; make that first call before any stream capture.
 * Every call uses the same array: calls that overlapped on the GPU would race,
 * so the function serializes its callers, clears the status word each call,
 * and returns only after the work on `stream` has finished (it synchronizes
 * the stream) -- which also lets it report a device-side timeout
 * (BB_ERR_TIMEOUT) directly.  Calls no allocating CUDA or library routine. */
bb_status bb_reduce_noalloc(void* band_ptr, int64_t n, int64_t bw, int64_t ldab, int64_t tw,
                            bb_dtype dtype, void* d_out, void* e_out, bb_stream_t stream);

/* Singular values of the upper bidiagonal matrix with diagonal d (n
 * entries) and superdiagonal e (n - 1 entries; may be NULL when n == 1), in
 * descending order, into sigma_out (n entries).  All three are device
 * pointers owned by the caller, of element type dtype; n >= 1.  Computed by
 * multisection on Sturm counts of the 2n x 2n Golub-Kahan tridiagonal (zero
 * diagonal, off-diagonal d_0, e_0, d_1, ..., d_{n-1}) with LAPACK xSTEBZ's
 * pivmin guard: a group of P lanes per value (P a power of two, the most that
 * fill the GPU, at most 32 in float and 8 in double) splits the interval
 * into P + 1 parts per step, down to about one ulp of the Gershgorin bound
 * max_i(|a_{i-1}| + |a_i|), the absolute accuracy.  This is the step
 * after the reduction in "A two-stage reduction on an Apple M5 Pro"
 * (Section 7).  Asynchronous on `stream`; allocates nothing; the return code
 * covers arguments and the launch. */
bb_status bb_singular_values(bb_dtype dtype, int64_t n, const void* d, const void* e, void* sigma_out,
                             bb_stream_t stream);
/* As bb_singular_values with the lanes per value fixed: 0 for the default
 * rule (the most that fill the GPU, at most 32 in float and 8 in double),
 * else a power of two in [1, 32] (BB_ERR_INVALID_ARG otherwise).  For
 * measurement and tests. */
bb_status bb_singular_values_lanes(bb_dtype dtype, int64_t n, const void* d, const void* e, void* sigma_out,
                                   int64_t lanes, bb_stream_t stream);

/* Stage 1 of the two-stage SVD, the step before this library's reduction:
 * the dense n x n matrix a (device, column-major, leading dimension
 * lda >= n, element type dtype: BB_F32 or BB_F64) is reduced in place to
 * upper band form of bandwidth bw >= 1 by orthogonal transformations, the
 * block Householder reduction that the accuracy protocol of "Accelerating
 * Bidiagonalization of Banded Matrices through Memory-Aware Bulge-Chasing
 * on GPUs" (Section V) runs before the band stage.  For each panel of bw
 * columns k .. k+bw-1: QR of the panel column by column (the reflector of
 * A(j.., j), LAPACK xLARFG convention, applied from the left to every later
 * column), then LQ of the panel's rows right of the band (the reflector of
 * A(i, i+bw ..), applied from the right to every later row).  Entries outside
 * the band (0 <= j - i <= bw) become exactly zero.  Blocked, 16 reflectors
 * at a time (a panel's QR reflectors in order, then its LQ reflectors): one
 * kernel factorizes the block (reflectors, and the T of their compact WY
 * form, LAPACK xLARFT), and the rest of the matrix is updated by matrix
 * products, A -= V T^T (V^T A) for QR blocks and A -= (A U) T U^T for LQ
 * blocks; the result equals the reflector-by-reflector sequence up to
 * rounding.  workspace: device memory of at least
 * bb_dense_to_band_workspace(n, bw, dtype) bytes (18 n b + b^2 + 2 b + 64
 * elements, b = min(bw, n, 16)), owned by the caller and not read
 * afterwards.  Asynchronous on `stream` (per block of reflectors: one panel
 * kernel, two matrix products, one reduction); the return code covers
 * arguments and launches.  bb_dense_to_band_workspace returns -1 for
 * invalid arguments (n < 1, n >= 2^30, bw < 1, dtype). */
int64_t bb_dense_to_band_workspace(int64_t n, int64_t bw, bb_dtype dtype);
bb_status bb_dense_to_band(bb_dtype dtype, int64_t n, int64_t bw, void* a, int64_t lda, void* workspace,
                           int64_t workspace_bytes, bb_stream_t stream);

/* Copy the upper band (0 <= j - i <= bw) of the dense column-major matrix a
 * (device, lda >= n) into the band storage of bb_reduce (device, ldab >=
 * bw + 2*tw + 1, A(i, j) at band[(bw + tw + i - j) + j * ldab]), every other
 * stored entry zero, so that stage 1's result feeds bb_reduce directly.
 * dtype BB_F32 or BB_F64; 0 <= bw < n, tw >= 0.  Asynchronous on `stream`. */
bb_status bb_pack_band(bb_dtype dtype, int64_t n, int64_t bw, int64_t tw, const void* a, int64_t lda, void* band,
                       int64_t ldab, bb_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BB_H_ */
