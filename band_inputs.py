"""Seeded synthetic inputs for the band -> bidiagonal reduction.

This module only draws random numbers and lays them out; it holds none of the
reduction's arithmetic.  Both the CUDA library's tests/benchmark and the CPU
oracle's tests take their inputs from here, so the two sides see the same
arrays.

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
10 ** (-8 j / n).  float32 workloads round the float64 draws.
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
        z = z * (10.0 ** (-8.0 * np.arange(n, dtype=np.float64) / n))[:, None]
    npd = np.float32 if dtype == "f32" else np.float64
    band = np.zeros((n, ldab), dtype=npd)
    # column j holds rows i = j - bw + q, q = 0..bw; drop i < 0
    q = np.arange(bw + 1)
    j = np.arange(n)[:, None]
    keep = (j - bw + q[None, :]) >= 0
    band[:, tw:tw + bw + 1] = np.where(keep, z, 0.0).astype(npd)
    return band


def make_workload(w: Workload, ldab: int | None = None, n: int | None = None) -> np.ndarray:
    """Band of workload w (optionally at another size n, same recipe)."""
    return make_band(n if n is not None else w.n, w.bw, w.tw, w.dtype, w.dist, w.graded,
                     w.seed, ldab)


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
