"""Serial CPU oracle (TEST INFRASTRUCTURE ONLY).

Python face of bb_oracle.c, the plain serial C implementation of the band ->
bidiagonal bulge-chasing reduction (arXiv 2510.12705, Section III and the text
of Algorithms 1-2; Householder convention of LAPACK xLARFG).  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library never calls it and shares no code with
it.

Functions take numpy arrays in the layout of ``band_inputs``: band storage of
shape (n, ldab), A(i, j) = band[j, ku + i - j], ku = bw + tw.

Also here:
  * ``reduce_band_pipelined``: the same reduction on host threads (sweep r on
    thread r mod P, "A two-stage reduction on an Apple M5 Pro", Section 6),
    bitwise equal to the serial order;
  * the symmetric variant (``sym_*``, ``tridiagonal``): symmetric band ->
    tridiagonal by the same passes, lower band storage
    A(i, j) = band[j, i - j];
  * ``bidiagonal_singular_values``: singular values of a bidiagonal by the
    Golub-Kahan tridiagonal's eigenvalues;
  * ``bidiagonal_with_vectors``: the reduction with its reflectors kept and
    applied to the identity, A = U B V^T (the back-transformation);
  * ``dense_to_band``: stage 1, a dense matrix to upper band form by block
    Householder (numpy, with this oracle's larfg);
  * half-precision storage: a float16 band is reduced with float arithmetic,
    every entry written back rounded to binary16 (``has_half``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bb_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_bb_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile bb_oracle.c with gcc (no contraction of multiply-adds)."""
    srcs = [_SRC, os.path.join(_HERE, "bb_oracle_body.h"), os.path.join(_HERE, "sb_oracle_body.h")]
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(s) for s in srcs)):
        return _LIB_PATH
    return compile_library(_SRC, _LIB_PATH)


def compile_library(src: str, out: str) -> str:
    """gcc the oracle source src (bb_oracle.c, which includes its body from
    the same folder) into the shared library out, atomically."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
                           "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the argument and result types of the oracle's C functions."""
    i64, p, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.oracle_has_half.argtypes = []
    lib.oracle_has_half.restype = ci
    for sfx in ("_d", "_f", "_h"):
        if sfx == "_h" and not lib.oracle_has_half():
            continue
        getattr(lib, "oracle_larfg" + sfx).argtypes = [i64, p, p, i64, p]
        getattr(lib, "oracle_larfg" + sfx).restype = None
        getattr(lib, "oracle_reduce_band" + sfx).argtypes = [i64, i64, i64, p, i64, i64, i64]
        getattr(lib, "oracle_reduce_band" + sfx).restype = ci
        getattr(lib, "oracle_reduce_dense" + sfx).argtypes = [i64, i64, i64, p]
        getattr(lib, "oracle_reduce_dense" + sfx).restype = ci
        getattr(lib, "oracle_halfstep_band" + sfx).argtypes = [i64, i64, i64, i64, p, i64, i64, i64, ci]
        getattr(lib, "oracle_halfstep_band" + sfx).restype = None
        getattr(lib, "oracle_sweep_steps" + sfx).argtypes = [i64, i64, i64, i64]
        getattr(lib, "oracle_sweep_steps" + sfx).restype = i64
        getattr(lib, "oracle_extract_band" + sfx).argtypes = [i64, i64, p, i64, p, p]
        getattr(lib, "oracle_extract_band" + sfx).restype = None
        getattr(lib, "oracle_reduce_band_pipelined" + sfx).argtypes = [i64, i64, i64, p, i64, i64,
                                                                       ctypes.c_double]
        getattr(lib, "oracle_reduce_band_pipelined" + sfx).restype = ci
        getattr(lib, "oracle_reduce_band_pipelined_range" + sfx).argtypes = [i64, i64, i64, p, i64, i64,
                                                                             ctypes.c_double, i64, i64]
        getattr(lib, "oracle_reduce_band_pipelined_range" + sfx).restype = ci
        getattr(lib, "oracle_reduce_band_record" + sfx).argtypes = [i64, i64, i64, p, i64, i64, p, p, p, p, p]
        getattr(lib, "oracle_reduce_band_record" + sfx).restype = i64
        if sfx == "_h":
            continue  # the symmetric variant has no half-precision storage instantiation
        getattr(lib, "oracle_sym_reduce_band" + sfx).argtypes = [i64, i64, i64, p, i64]
        getattr(lib, "oracle_sym_reduce_band" + sfx).restype = ci
        getattr(lib, "oracle_sym_reduce_dense" + sfx).argtypes = [i64, i64, i64, p]
        getattr(lib, "oracle_sym_reduce_dense" + sfx).restype = ci
        getattr(lib, "oracle_sym_extract_band" + sfx).argtypes = [i64, p, i64, p, p]
        getattr(lib, "oracle_sym_extract_band" + sfx).restype = None
        getattr(lib, "oracle_sym_step_band" + sfx).argtypes = [i64, i64, i64, p, i64, i64, i64]
        getattr(lib, "oracle_sym_step_band" + sfx).restype = None
        getattr(lib, "oracle_sym_reduce_band_pipelined" + sfx).argtypes = [i64, i64, i64, p, i64, i64,
                                                                           ctypes.c_double]
        getattr(lib, "oracle_sym_reduce_band_pipelined" + sfx).restype = ci
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build()))
    return _lib


def _sfx(arr: np.ndarray) -> str:
    if arr.dtype == np.float64:
        return "_d"
    if arr.dtype == np.float32:
        return "_f"
    if arr.dtype == np.float16:
        if not has_half():
            raise TypeError("this build of the oracle has no half-precision storage (no _Float16)")
        return "_h"
    raise TypeError(f"unsupported dtype {arr.dtype}")


def has_half() -> bool:
    """Whether the oracle was built with the half-precision storage variant."""
    return bool(_load().oracle_has_half())


def _arith(dt) -> np.dtype:
    """Arithmetic type of a band of dtype dt (float for half storage)."""
    return np.dtype(np.float32) if np.dtype(dt) == np.float16 else np.dtype(dt)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def larfg(alpha: float, x: np.ndarray):
    """LAPACK-convention reflector of (alpha, x): returns (beta, v_tail, tau)."""
    x = np.array(x, copy=True)
    lib = _load()
    a = np.array([alpha], dtype=x.dtype)
    tau = np.zeros(1, dtype=x.dtype)
    getattr(lib, "oracle_larfg" + _sfx(x))(x.size, _ptr(a), _ptr(x), 1, _ptr(tau))
    return a[0], x, tau[0]


def pass_plan(bw: int, tw: int):
    """[(b, t), ...]: b = bw; while b > 1: t = min(tw, b - 1); b -= t."""
    plan, b = [], bw
    while b > 1:
        t = min(tw, b - 1)
        plan.append((b, t))
        b -= t
    return plan


def reduce_band(band: np.ndarray, n: int, bw: int, tw: int, pass_lo: int = 0,
                pass_hi: int = 1 << 30) -> np.ndarray:
    """Reduce band storage in place (serial order); returns the same array."""
    assert band.flags.c_contiguous and band.shape[0] == n
    ldab = band.shape[1]
    rc = getattr(_load(), "oracle_reduce_band" + _sfx(band))(n, bw, tw, _ptr(band), ldab,
                                                              pass_lo, pass_hi)
    if rc != 0:
        raise ValueError("oracle_reduce_band: invalid arguments")
    return band


def reduce_band_pipelined(band: np.ndarray, n: int, bw: int, tw: int, threads: int,
                          time_limit: float = 600.0, pass_lo: int = 0, pass_hi: int = 1 << 62) -> np.ndarray:
    """reduce_band on host threads: sweep r on thread r mod threads, each sweep
    spinning on its predecessor's count of finished half-steps (the pipelined
    chase of "A two-stage reduction on an Apple M5 Pro", Section 6, with the
    half-step separation rule).  Bitwise equal to reduce_band (also over a
    pass range [pass_lo, pass_hi)).  Raises TimeoutError after time_limit
    seconds of waiting."""
    assert band.flags.c_contiguous and band.shape[0] == n
    rc = getattr(_load(), "oracle_reduce_band_pipelined_range" + _sfx(band))(
        n, bw, tw, _ptr(band), band.shape[1], threads, float(time_limit), pass_lo, pass_hi)
    if rc == -1:
        raise ValueError("oracle_reduce_band_pipelined: invalid arguments")
    if rc == -2:
        raise TimeoutError("oracle_reduce_band_pipelined: time limit reached")
    if rc != 0:
        raise RuntimeError("oracle_reduce_band_pipelined: could not start the threads")
    return band


def reflector_count(n: int, bw: int, tw: int) -> int:
    """Reflectors of a whole reduction: two per step (right, then left)."""
    return 2 * sum(sweep_steps(n, b, t, r) for (b, t) in pass_plan(bw, tw) for r in range(n))


def reduce_band_record(band: np.ndarray, n: int, bw: int, tw: int):
    """reduce_band in place, also returning every reflector in the order
    applied: (side, start, width, tau, v) with side 0 = right (columns
    start .. start+width-1), 1 = left (those rows), v of shape (count, tw+1)."""
    assert band.flags.c_contiguous and band.shape[0] == n
    cap = reflector_count(n, bw, tw)
    side = np.zeros(cap, dtype=np.int8)
    start = np.zeros(cap, dtype=np.int64)
    width = np.zeros(cap, dtype=np.int32)
    taus = np.zeros(cap, dtype=_arith(band.dtype))
    vs = np.zeros((cap, tw + 1), dtype=_arith(band.dtype))
    got = getattr(_load(), "oracle_reduce_band_record" + _sfx(band))(
        n, bw, tw, _ptr(band), band.shape[1], cap, _ptr(side), _ptr(start), _ptr(width), _ptr(taus), _ptr(vs))
    if got == -1:
        raise ValueError("oracle_reduce_band_record: invalid arguments")
    if got != cap:
        raise RuntimeError(f"oracle_reduce_band_record: {got} reflectors, expected {cap}")
    return side, start, width, taus, vs


def bidiagonal_with_vectors(band: np.ndarray, n: int, bw: int, tw: int):
    """(d, e, U, V) with A = U B V^T, B the upper bidiagonal (d, e), U, V
    orthogonal (float64).  U = L_1 L_2 ... and V = R_1 R_2 ... in the order the
    reduction applied the left and right reflectors, formed by applying each
    reflector to the identity with numpy (the back-transformation)."""
    work = np.ascontiguousarray(band.copy())
    side, start, width, taus, vs = reduce_band_record(work, n, bw, tw)
    d, e = extract(work, n, bw + tw)
    U = np.eye(n)
    V = np.eye(n)
    for q in range(side.size):
        tau = float(taus[q])
        if tau == 0.0:
            continue
        c, w = int(start[q]), int(width[q])
        v = vs[q, :w].astype(np.float64)
        M = U if side[q] == 1 else V
        # M <- M H on columns c .. c+w-1
        y = M[:, c:c + w] @ v
        M[:, c:c + w] -= tau * np.outer(y, v)
    return d, e, U, V


def reduce_dense(a: np.ndarray, bw: int, tw: int) -> np.ndarray:
    """Reduce a dense row-major n x n array in place (reflectors on whole rows/cols)."""
    assert a.flags.c_contiguous and a.shape[0] == a.shape[1]
    rc = getattr(_load(), "oracle_reduce_dense" + _sfx(a))(a.shape[0], bw, tw, _ptr(a))
    if rc != 0:
        raise ValueError("oracle_reduce_dense: invalid arguments")
    return a


def halfstep_band(band: np.ndarray, n: int, b: int, t: int, ku: int, r: int, k: int,
                  side: int) -> None:
    """One half-step (side 0: right/row reflector, 1: left/column) in place."""
    getattr(_load(), "oracle_halfstep_band" + _sfx(band))(n, b, t, ku, _ptr(band),
                                                          band.shape[1], r, k, side)


def sweep_steps(n: int, b: int, t: int, r: int) -> int:
    return int(_load().oracle_sweep_steps_d(n, b, t, r))


def extract(band: np.ndarray, n: int, ku: int):
    """(d, e) of band storage, in the arithmetic type (float for half storage)."""
    d = np.zeros(n, dtype=_arith(band.dtype))
    e = np.zeros(max(n - 1, 0), dtype=_arith(band.dtype))
    getattr(_load(), "oracle_extract_band" + _sfx(band))(n, ku, _ptr(band), band.shape[1],
                                                         _ptr(d), _ptr(e))
    return d, e


def bidiagonal(band: np.ndarray, n: int, bw: int, tw: int):
    """(d, e) of the reduction of a copy of band (serial oracle)."""
    work = np.ascontiguousarray(band.copy())
    reduce_band(work, n, bw, tw)
    return extract(work, n, bw + tw)


def bidiagonal_pipelined(band: np.ndarray, n: int, bw: int, tw: int, threads: int,
                         time_limit: float = 600.0):
    """(d, e) of the pipelined reduction of a copy of band."""
    work = np.ascontiguousarray(band.copy())
    reduce_band_pipelined(work, n, bw, tw, threads, time_limit)
    return extract(work, n, bw + tw)


# ------------------------------------------------ stage 1: dense -> band ---

def dense_to_band(a: np.ndarray, bw: int) -> np.ndarray:
    """Stage 1 of the two-stage SVD: an n x n matrix reduced to upper band
    form of bandwidth bw by orthogonal transformations, the "classical block
    Householder reduction" of the accuracy protocol ("Accelerating
    Bidiagonalization of Banded Matrices through Memory-Aware Bulge-Chasing on
    GPUs", Section V; the GPU stage of "A two-stage reduction on an Apple M5
    Pro" uses the same panels).  For each panel of bw columns k .. k+bw-1:
    QR of the panel column by column (reflector of A(j.., j), applied from the
    left to every later column), then LQ of the panel's rows to the right of
    the band, row by row (reflector of A(i, i+bw ..), applied from the right
    to every later row).  Reflectors are this oracle's larfg; annihilated
    entries are set to exactly zero.  Returns a new array (same dtype)."""
    a = np.array(a, copy=True)
    n = a.shape[0]
    if bw < 1:
        raise ValueError("bw must be at least 1")
    for k in range(0, n, bw):
        kb = min(k + bw, n)
        for j in range(k, kb):
            if j + 1 >= n:
                break
            beta, v, tau = larfg(a[j, j], a[j + 1:, j].copy())
            a[j, j] = beta
            a[j + 1:, j] = 0
            if tau != 0:
                u = np.concatenate([[1.0], v]).astype(a.dtype)
                y = u @ a[j:, j + 1:]
                a[j:, j + 1:] -= tau * np.outer(u, y)
        for i in range(k, kb):
            c0 = i + bw
            if c0 + 1 >= n:
                break
            beta, v, tau = larfg(a[i, c0], a[i, c0 + 1:].copy())
            a[i, c0] = beta
            a[i, c0 + 1:] = 0
            if tau != 0:
                u = np.concatenate([[1.0], v]).astype(a.dtype)
                y = a[i + 1:, c0:] @ u
                a[i + 1:, c0:] -= tau * np.outer(y, u)
    return a


# ------------------------------------------------ symmetric variant -------
# Symmetric band -> tridiagonal (sb_oracle_body.h): lower band storage of shape
# (n, ldab), A(i, j) = band[j, i - j] for 0 <= i - j < ldab, ldab >= bw + tw + 1.

def sym_reduce_band(band: np.ndarray, n: int, bw: int, tw: int) -> np.ndarray:
    """Reduce symmetric lower band storage to tridiagonal form in place."""
    assert band.flags.c_contiguous and band.shape[0] == n
    rc = getattr(_load(), "oracle_sym_reduce_band" + _sfx(band))(n, bw, tw, _ptr(band), band.shape[1])
    if rc != 0:
        raise ValueError("oracle_sym_reduce_band: invalid arguments")
    return band


def sym_reduce_dense(a: np.ndarray, bw: int, tw: int) -> np.ndarray:
    """Reduce a dense symmetric row-major n x n array in place (both triangles)."""
    assert a.flags.c_contiguous and a.shape[0] == a.shape[1]
    rc = getattr(_load(), "oracle_sym_reduce_dense" + _sfx(a))(a.shape[0], bw, tw, _ptr(a))
    if rc != 0:
        raise ValueError("oracle_sym_reduce_dense: invalid arguments")
    return a


def sym_extract(band: np.ndarray, n: int):
    """(d, e): diagonal and subdiagonal of the lower band storage."""
    d = np.zeros(n, dtype=band.dtype)
    e = np.zeros(max(n - 1, 0), dtype=band.dtype)
    getattr(_load(), "oracle_sym_extract_band" + _sfx(band))(n, _ptr(band), band.shape[1], _ptr(d), _ptr(e))
    return d, e


def sym_reduce_band_pipelined(band: np.ndarray, n: int, bw: int, tw: int, threads: int,
                              time_limit: float = 600.0) -> np.ndarray:
    """sym_reduce_band on host threads (sweep r on thread r mod threads, step k
    of sweep r after sweep r-1 finished min(k + L, its steps), L = 2, or 3
    when b - t = 1).  Bitwise equal to sym_reduce_band."""
    assert band.flags.c_contiguous and band.shape[0] == n
    rc = getattr(_load(), "oracle_sym_reduce_band_pipelined" + _sfx(band))(
        n, bw, tw, _ptr(band), band.shape[1], threads, float(time_limit))
    if rc == -1:
        raise ValueError("oracle_sym_reduce_band_pipelined: invalid arguments")
    if rc == -2:
        raise TimeoutError("oracle_sym_reduce_band_pipelined: time limit reached")
    if rc != 0:
        raise RuntimeError("oracle_sym_reduce_band_pipelined: could not start the threads")
    return band


def sym_step_band(band: np.ndarray, n: int, b: int, t: int, r: int, k: int) -> None:
    """One step (sweep r, step k) of pass (b, t) in place (lower band storage)."""
    getattr(_load(), "oracle_sym_step_band" + _sfx(band))(n, b, t, _ptr(band), band.shape[1], r, k)


def tridiagonal(band: np.ndarray, n: int, bw: int, tw: int):
    """(d, e) of the symmetric reduction of a copy of band (serial oracle)."""
    work = np.ascontiguousarray(band.copy())
    sym_reduce_band(work, n, bw, tw)
    return sym_extract(work, n)


def bidiagonal_singular_values(d: np.ndarray, e: np.ndarray) -> np.ndarray:
    """Singular values of the upper bidiagonal matrix (d, e), descending, in
    float64: by definition the non-negative eigenvalues of the 2n x 2n
    Golub-Kahan tridiagonal with zero diagonal and off-diagonal
    (d_0, e_0, d_1, ..., d_{n-1}), taken with LAPACK's symmetric tridiagonal
    eigensolver (scipy.linalg.eigvalsh_tridiagonal).  The oracle of
    bb_singular_values ("A two-stage reduction on an Apple M5 Pro",
    Section 7: bidiagonal singular values by bisection on this matrix)."""
    import scipy.linalg as sla
    d = np.asarray(d, dtype=np.float64)
    e = np.asarray(e, dtype=np.float64)
    n = d.size
    if n == 0:
        return np.zeros(0)
    if n == 1:
        return np.abs(d)
    off = np.empty(2 * n - 1)
    off[0::2] = d
    off[1::2] = e[: n - 1]
    # sigma(s B) = |s| sigma(B): scale by the power of two that brings the
    # largest entry near 1 (exact), so that the eigensolver's internal
    # squares neither under- nor overflow, and scale the result back
    amax = float(np.abs(off).max())
    k = int(np.floor(np.log2(amax))) if amax > 0 and np.isfinite(amax) else 0
    ev = sla.eigvalsh_tridiagonal(np.zeros(2 * n), np.ldexp(off, -k))
    return np.ldexp(np.sort(ev)[::-1][:n].clip(min=0.0), k)

