"""Seeded synthetic inputs for the band -> bidiagonal reduction.

This module only draws random numbers and lays them out; it holds none of the
reduction's arithmetic.  Both the CUDA library's tests/benchmark and the CPU
oracle's tests take their inputs from here, so the two sides see the same
arrays.  The one construction beyond that, the band with prescribed singular
values, runs the *first* stage of the two-stage SVD (dense -> band) with
numpy's QR; the band -> bidiagonal reduction itself appears nowhere here.

Storage is compact column-major band storage with fill rows (LAPACK "gb"
layout with ku = bw + tw upper and kl = tw lower diagonals):

    A(i, j)  <->  band[j, ku + i - j]          (numpy array of shape (n, ldab))

so column j of the matrix occupies the contiguous row band[j, :].  An upper
band of bandwidth bw occupies band rows tw .. tw + bw; the fill rows
0 .. tw-1 and ku+1 .. ku+tw start at zero, and ldab >= bw + 2 tw + 1.

Draw order (identical for every workload): Z = rng.<dist>(size=(n, bw+1)) in
float64 with rng = numpy.random.default_rng(seed); entry A(i, j), 0 <= j-i <=
bw, i >= 0, is Z[j, bw - (j - i)], i.e. band[j, tw + q] = Z[j, q]; draws that
would fall above row 0 are discarded.  A graded workload multiplies column j by
10 ** (-8 j / n) (correctly rounded).  float32 workloads round the float64
draws.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n: int
    bw: int
    tw: int
    dtype: str          # "f32" or "f64"
    dist: str           # "normal" or "uniform"
    graded: bool
    seed: int

    @property
    def np_dtype(self):
        return np.float32 if self.dtype == "f32" else np.float64

    @property
    def ldab(self) -> int:
        return self.bw + 2 * self.tw + 1

    def describe(self) -> str:
        g = ", column j scaled by 10^(-8j/N)" if self.graded else ""
        d = "N(0,1)" if self.dist == "normal" else "U[-1,1]"
        return (f"N={self.n} upper band BW={self.bw} TW={self.tw} {self.dtype}, "
                f"in-band entries iid {d}{g}, seed {self.seed}")


# The five workloads the benchmark and the full-size tests use.  Seeds are the
# workload's index.
WORKLOADS = [
    Workload("n256_bw8_tw7_f64", 256, 8, 7, "f64", "normal", False, 0),
    Workload("n4096_bw16_tw8_f32", 4096, 16, 8, "f32", "uniform", False, 1),
    Workload("n8192_bw64_tw16_f32", 8192, 64, 16, "f32", "normal", False, 2),
    Workload("n16384_bw128_tw32_f64_graded", 16384, 128, 32, "f64", "normal", True, 3),
    Workload("n32768_bw256_tw32_f32", 32768, 256, 32, "f32", "normal", False, 4),
]


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def make_band(n: int, bw: int, tw: int, dtype="f64", dist="normal", graded=False,
              seed=0, ldab: int | None = None) -> np.ndarray:
    """Band storage (shape (n, ldab), C-contiguous) of a random upper band."""
    if ldab is None:
        ldab = bw + 2 * tw + 1
    if ldab < bw + 2 * tw + 1:
        raise ValueError("ldab too small")
    rng = np.random.default_rng(seed)
    if dist == "normal":
        z = rng.standard_normal(size=(n, bw + 1))
    elif dist == "uniform":
        z = rng.uniform(-1.0, 1.0, size=(n, bw + 1))
    elif dist == "zeros":
        z = np.zeros((n, bw + 1))
    else:
        raise ValueError(dist)
    if graded:
        z = z * graded_scale(n)[:, None]
    npd = np.float32 if dtype == "f32" else np.float64
    band = np.zeros((n, ldab), dtype=npd)
    # column j holds rows i = j - bw + q, q = 0..bw; drop i < 0
    q = np.arange(bw + 1)
    j = np.arange(n)[:, None]
    keep = (j - bw + q[None, :]) >= 0
    band[:, tw:tw + bw + 1] = np.where(keep, z, 0.0).astype(npd)
    return band


def graded_scale(n: int) -> np.ndarray:
    """10 ** (-8 j / n), j = 0 .. n-1, each correctly rounded to float64
    (decimal arithmetic), so that the graded workload's input is the same on
    every machine (vectorised power routines differ in the last bit)."""
    import decimal
    ctx = decimal.Context(prec=40)
    ten, den = decimal.Decimal(10), decimal.Decimal(n)
    return np.array([float(ctx.power(ten, ctx.divide(decimal.Decimal(-8 * j), den))) for j in range(n)],
                    dtype=np.float64)


def make_workload(w: Workload, ldab: int | None = None, n: int | None = None) -> np.ndarray:
    """Band of workload w (optionally at another size n, same recipe)."""
    return make_band(n if n is not None else w.n, w.bw, w.tw, w.dtype, w.dist, w.graded,
                     w.seed, ldab)


def perturb_ulp(band: np.ndarray, seed: int) -> np.ndarray:
    """A copy of band with every entry multiplied by 1 + eps * N(0, 1) (eps of
    the band's dtype; rng = numpy.random.default_rng(seed), draws in band
    order), rounded back to that dtype: a relative perturbation of about one
    ulp, which the tests use to measure how much the reduction's output moves
    under rounding-sized changes of its input."""
    rng = np.random.default_rng(seed)
    eps = np.finfo(band.dtype).eps
    return (band * (1 + eps * rng.standard_normal(band.shape))).astype(band.dtype)


# Seeds of the one-ulp perturbations behind the measured sensitivity.
SENSITIVITY_SEEDS = (101, 202, 303)


def band_to_dense(band: np.ndarray, n: int, ku: int) -> np.ndarray:
    """Dense n x n matrix of every entry the band storage can hold."""
    ldab = band.shape[1]
    a = np.zeros((n, n), dtype=band.dtype)
    for j in range(n):
        for d in range(ldab):
            i = j + d - ku
            if 0 <= i < n:
                a[i, j] = band[j, d]
    return a


def dense_to_band(a: np.ndarray, ku: int, ldab: int) -> np.ndarray:
    """Band storage of the entries of a with -(ldab-1-ku) <= j-i <= ku."""
    n = a.shape[0]
    band = np.zeros((n, ldab), dtype=a.dtype)
    for j in range(n):
        for d in range(ldab):
            i = j + d - ku
            if 0 <= i < n:
                band[j, d] = a[i, j]
    return band


# ------------------------------------------------ prescribed singular values ---
#
# Accuracy protocol of "Accelerating Bidiagonalization of Banded Matrices
# through Memory-Aware Bulge-Chasing on GPUs" (Section V, accuracy study):
# A = U diag(sigma) V^T with random orthogonal U, V and sigma in [0, 1] from
# one of three profiles (uniform spacing, logarithmic decay, quarter-circle),
# reduced to band form in double precision by block Householder; the
# band -> bidiagonal reduction then runs in the precision under test and the
# singular values of its result are compared with sigma.

SPECTRA = ("arithmetic", "logarithmic", "quarter_circle")


def spectrum(kind: str, n: int, seed: int = 0, decades: float = 8.0) -> np.ndarray:
    """n singular values in [0, 1], descending, float64.

    arithmetic      k / n, k = n .. 1 (uniform spacing);
    logarithmic     10 ** (-decades * k / (n - 1)), k = 0 .. n-1;
    quarter_circle  n seeded draws from the density (4 / pi) sqrt(1 - x^2) on
                    [0, 1] (the limit law of the singular values of a scaled
                    square Gaussian matrix): |sqrt(u1) cos(2 pi u2)| is the
                    |abscissa| of a point uniform in the unit disc;
    rank_deficient  the arithmetic profile of n - n // 2 values, then n // 2
                    exact zeros.
    """
    if n == 0:
        return np.zeros(0)
    if kind == "arithmetic":
        s = np.arange(n, 0, -1, dtype=np.float64) / n
    elif kind == "logarithmic":
        s = 10.0 ** (-decades * np.arange(n, dtype=np.float64) / max(n - 1, 1))
    elif kind == "quarter_circle":
        rng = np.random.default_rng(seed)
        u1 = rng.random(n)
        u2 = rng.random(n)
        s = np.sort(np.abs(np.sqrt(u1) * np.cos(2.0 * np.pi * u2)))[::-1]
    elif kind == "rank_deficient":
        m = n - n // 2
        s = np.concatenate([np.arange(m, 0, -1, dtype=np.float64) / m, np.zeros(n // 2)])
    else:
        raise ValueError(kind)
    return np.ascontiguousarray(s)


def _haar_orthogonal(n: int, rng) -> np.ndarray:
    """Haar-distributed orthogonal matrix: QR of a Gaussian matrix with the
    signs of R's diagonal moved into Q."""
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    sg = np.sign(np.diag(r))
    sg[sg == 0] = 1.0
    return q * sg


def dense_to_upper_band(a: np.ndarray, bw: int) -> np.ndarray:
    """Orthogonally equivalent upper band of bandwidth bw (float64), by block
    Householder: for each panel of bw columns, the QR factorisation of the
    panel (rows below) zeroes it under the diagonal; the LQ factorisation of
    the bw rows to the right of the panel (as QR of their transpose) leaves
    them lower triangular, so row i ends at column i + bw.  LAPACK's compact
    reflectors (geqrf through scipy's raw QR) are applied with ormqr.  The
    rounding residue left outside the band (a few eps * ||a||) is set to
    zero."""
    import scipy.linalg as sla
    from scipy.linalg import lapack

    a = np.array(a, dtype=np.float64, copy=True, order="F")
    n = a.shape[0]
    if bw < 1:
        raise ValueError("bw must be at least 1")
    for k in range(0, n, bw):
        kb = min(k + bw, n)
        (qr, tau), _ = sla.qr(a[k:, k:kb], mode="raw")
        c = np.asfortranarray(a[k:, k:])
        c, _, info = lapack.dormqr("L", "T", qr[:, :tau.size], tau, c, max(1, c.shape[1] * 64))
        assert info == 0
        a[k:, k:] = c
        if kb < n:
            (qr, tau), _ = sla.qr(a[k:kb, kb:].T, mode="raw")
            # rows above k are already zero in columns kb..
            c = np.asfortranarray(a[k:, kb:])
            c, _, info = lapack.dormqr("R", "N", qr[:, :tau.size], tau, c, max(1, c.shape[0] * 64))
            assert info == 0
            a[k:, kb:] = c
    i, j = np.indices(a.shape)
    a[(j < i) | (j - i > bw)] = 0.0
    return np.ascontiguousarray(a)


def make_band_with_spectrum(n: int, bw: int, tw: int, sigma: np.ndarray, dtype="f64", seed=0,
                            ldab: int | None = None) -> np.ndarray:
    """Band storage (shape (n, ldab)) of an upper band of bandwidth bw whose
    singular values are sigma up to the float64 rounding of the construction:
    A = U diag(sigma) V^T with U, V Haar-random (seeded), reduced to band form
    by dense_to_upper_band.  float32 rounds the float64 band."""
    if ldab is None:
        ldab = bw + 2 * tw + 1
    if ldab < bw + 2 * tw + 1:
        raise ValueError("ldab too small")
    sigma = np.asarray(sigma, dtype=np.float64)
    if sigma.shape != (n,):
        raise ValueError("sigma must have n entries")
    rng = np.random.default_rng(seed)
    u = _haar_orthogonal(n, rng)
    v = _haar_orthogonal(n, rng)
    a = dense_to_upper_band((u * sigma) @ v.T, max(bw, 1))
    npd = np.float32 if dtype == "f32" else np.float64
    return dense_to_band(a, bw + tw, ldab).astype(npd)


# ------------------------------------------------------ symmetric variant ---
#
# Symmetric band matrices in LAPACK's lower band layout with fill rows:
# A(i, j), 0 <= i - j < ldab, at sband[j, i - j] (numpy array of shape
# (n, ldab)); an input of bandwidth bw occupies rows 0 .. bw, the fill rows
# bw+1 .. bw+tw start at zero, ldab >= bw + tw + 1.


def make_sym_band(n: int, bw: int, tw: int, dtype="f64", dist="normal", seed=0,
                  ldab: int | None = None) -> np.ndarray:
    """Lower band storage of a random symmetric band matrix: Z = rng.<dist>(
    size=(n, bw+1)) in float64, sband[j, q] = Z[j, q] (entry A(j+q, j)),
    draws that would fall below row n - 1 discarded."""
    if ldab is None:
        ldab = bw + tw + 1
    if ldab < bw + tw + 1:
        raise ValueError("ldab too small")
    rng = np.random.default_rng(seed)
    if dist == "normal":
        z = rng.standard_normal(size=(n, bw + 1))
    elif dist == "uniform":
        z = rng.uniform(-1.0, 1.0, size=(n, bw + 1))
    elif dist == "zeros":
        z = np.zeros((n, bw + 1))
    else:
        raise ValueError(dist)
    npd = np.float32 if dtype == "f32" else np.float64
    sband = np.zeros((n, ldab), dtype=npd)
    keep = (np.arange(n)[:, None] + np.arange(bw + 1)[None, :]) < n
    sband[:, :bw + 1] = np.where(keep, z, 0.0).astype(npd)
    return sband


def sym_band_to_dense(sband: np.ndarray, n: int) -> np.ndarray:
    """Dense symmetric n x n matrix of the lower band storage."""
    a = np.zeros((n, n), dtype=sband.dtype)
    for j in range(n):
        for q in range(sband.shape[1]):
            if j + q < n:
                a[j + q, j] = sband[j, q]
                a[j, j + q] = sband[j, q]
    return a


def dense_to_sym_band(a: np.ndarray, ldab: int) -> np.ndarray:
    """Lower band storage of the entries of a with 0 <= i - j < ldab."""
    n = a.shape[0]
    sband = np.zeros((n, ldab), dtype=a.dtype)
    for j in range(n):
        for q in range(ldab):
            if j + q < n:
                sband[j, q] = a[j + q, j]
    return sband


def dense_to_sym_band_form(a: np.ndarray, bw: int) -> np.ndarray:
    """Orthogonally similar symmetric band of bandwidth bw (float64), by block
    Householder: for each panel of bw columns, the QR factorisation of the
    panel's rows below the band, applied from both sides, leaves it upper
    triangular there.  The rounding residue outside the band is set to zero
    and the result symmetrised exactly from its lower triangle."""
    import scipy.linalg as sla
    from scipy.linalg import lapack

    a = np.array(a, dtype=np.float64, copy=True, order="F")
    n = a.shape[0]
    if bw < 1:
        raise ValueError("bw must be at least 1")
    for k in range(0, n, bw):
        r0 = k + bw
        if r0 >= n:
            break
        kb = min(k + bw, n)
        (qr, tau), _ = sla.qr(a[r0:, k:kb], mode="raw")
        c = np.asfortranarray(a[r0:, :])
        c, _, info = lapack.dormqr("L", "T", qr[:, :tau.size], tau, c, max(1, c.shape[1] * 64))
        assert info == 0
        a[r0:, :] = c
        c = np.asfortranarray(a[:, r0:])
        c, _, info = lapack.dormqr("R", "N", qr[:, :tau.size], tau, c, max(1, c.shape[0] * 64))
        assert info == 0
        a[:, r0:] = c
    i, j = np.indices(a.shape)
    a[np.abs(i - j) > bw] = 0.0
    low = np.tril(a)
    return np.ascontiguousarray(low + np.tril(low, -1).T)


def make_sym_band_with_spectrum(n: int, bw: int, tw: int, lam: np.ndarray, dtype="f64", seed=0,
                                ldab: int | None = None) -> np.ndarray:
    """Lower band storage of a symmetric band of bandwidth bw whose
    eigenvalues are lam up to the float64 rounding of the construction:
    A = Q diag(lam) Q^T with Q Haar-random (seeded), reduced to band form by
    dense_to_sym_band_form.  float32 rounds the float64 band."""
    if ldab is None:
        ldab = bw + tw + 1
    if ldab < bw + tw + 1:
        raise ValueError("ldab too small")
    lam = np.asarray(lam, dtype=np.float64)
    if lam.shape != (n,):
        raise ValueError("lam must have n entries")
    rng = np.random.default_rng(seed)
    q = _haar_orthogonal(n, rng)
    a = (q * lam) @ q.T
    a = dense_to_sym_band_form(0.5 * (a + a.T), max(bw, 1))
    npd = np.float32 if dtype == "f32" else np.float64
    return dense_to_sym_band(a, ldab).astype(npd)
