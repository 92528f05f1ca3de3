"""Shared helpers of the GPU tests: run the CUDA library through the C ABI and
compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import scipy.linalg as sla
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb

# Acceptance tolerances on max |sigma - sigma_ref| / ||A||_F (singular values
# of the GPU bidiagonal against those of the oracle's), and the floor of the
# tolerance on max(| |d|-|d_ref| |, | |e|-|e_ref| |) / ||A||_F.
TOL = {"f64": 1e-12, "f32": 2e-5}

# |d| and |e| are unique in exact arithmetic but, for these random upper-band
# inputs, ill-conditioned functions of A: the oracle's own output moves by
# more than TOL when its input is perturbed by one ulp (singular values move
# by ~eps).  The |d|,|e| tolerance is therefore max(TOL, DE_FACTOR * S) with S
# the oracle's measured sensitivity to a one-ulp relative perturbation of the
# input (largest of three random perturbations).  The GPU differs from the
# oracle by rounding only (fused multiply-adds, reduction order), i.e. by a
# backward perturbation of a few ulps per operation; the largest ratio of its
# |d|,|e| error to S measured on the parity cases is about 2.7.
DE_FACTOR = 4.0

# Float32 forward error: the GPU's |d|,|e| distance from the float64 oracle
# run on the same (float32) input may be at most FWD_FACTOR times the float32
# oracle's own distance from it (plus TOL): the GPU may not be less accurate
# than the float32 oracle by more than rounding noise.
FWD_FACTOR = 2.0


def torch_dtype(dt: str):
    return torch.float64 if dt == "f64" else torch.float32


def gpu_reduce(band: np.ndarray, n: int, bw: int, tw: int, dt: str, scheduler: int = 0,
               params: dict | None = None, return_band: bool = False):
    """Reduce a copy of band on cuda:0 via bb_reduce; returns numpy (d, e[, band])."""
    dev = torch.device("cuda:0")
    x = torch.from_numpy(np.ascontiguousarray(band)).to(dev)
    d = torch.empty(n, dtype=x.dtype, device=dev)
    e = torch.empty(max(n - 1, 1), dtype=x.dtype, device=dev)
    h = bb.bb_create(n, bw, bb.dtype_code(dt))
    try:
        bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, scheduler)
        for k, v in (params or {}).items():
            bb.bb_set_param(h, k, v)
        s = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        st = bb.bb_status_sync(h, s)
        assert st == bb.BB_OK, f"device status {st}: {bb.bb_last_error()}"
    finally:
        bb.bb_destroy(h)
    out = (d.cpu().numpy(), e[: max(n - 1, 0)].cpu().numpy())
    if return_band:
        out = out + (x.cpu().numpy(),)
    return out


def oracle_sensitivity(band: np.ndarray, n: int, bw: int, tw: int, seeds=bi.SENSITIVITY_SEEDS) -> float:
    """max over seeds of max | |d'|-|d| |, | |e'|-|e| | / ||A||_F where (d', e') is
    the oracle's result on band_inputs.perturb_ulp(band, seed) (same precision)."""
    import oracle
    d, e = oracle.bidiagonal(band, n, bw, tw)
    fro = fro_of_band(band)
    worst = 0.0
    for sd in seeds:
        d2, e2 = oracle.bidiagonal(bi.perturb_ulp(band, sd), n, bw, tw)
        worst = max(worst, de_error(d2, e2, d, e, fro))
    return worst


def record(kind: str, **kw) -> None:
    """Append a parity record (JSON line) to the file named by the environment
    variable BB_PARITY_RECORDS, when it is set."""
    import json
    import os
    path = os.environ.get("BB_PARITY_RECORDS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"kind": kind, **kw}) + "\n")


def sigma_bidiagonal(d, e):
    n = d.size
    if n == 1:
        return np.abs(d.astype(np.float64))
    off = np.empty(2 * n - 1)
    off[0::2] = d
    off[1::2] = e
    ev = sla.eigvalsh_tridiagonal(np.zeros(2 * n), off)
    return np.sort(ev)[::-1][:n]


def de_error(d, e, d_ref, e_ref, fro):
    err_d = np.abs(np.abs(d.astype(np.float64)) - np.abs(d_ref.astype(np.float64))).max() if d.size else 0.0
    err_e = np.abs(np.abs(e.astype(np.float64)) - np.abs(e_ref.astype(np.float64))).max() if e.size else 0.0
    return max(err_d, err_e) / max(fro, np.finfo(np.float64).tiny)


def fro_of_band(band: np.ndarray) -> float:
    return float(np.linalg.norm(band.astype(np.float64)))


def off_bidiagonal_nonzeros(band_after: np.ndarray, n: int, ku: int) -> int:
    """Stored entries of the valid matrix area other than d and e that are not 0."""
    ldab = band_after.shape[1]
    j = np.arange(n)[:, None]
    q = np.arange(ldab)[None, :]
    i = j + q - ku
    valid = (i >= 0) & (i < n)
    keep = (q == ku) | (q == ku - 1)  # d: i == j, e: i == j - 1
    mask = valid & ~keep
    return int(np.count_nonzero(band_after[mask]))


def fourth_moment_band(band: np.ndarray, n: int, bw: int, tw: int) -> float:
    """sum sigma_i^4 = ||A^T A||_F^2 of the input band (float64), from the
    column inner products a_j . a_{j+delta}, delta = 0..bw."""
    a = band.astype(np.float64)
    total = 0.0
    for delta in range(bw + 1):
        g = (a[: n - delta, tw + delta: tw + bw + 1] * a[delta:, tw: tw + bw + 1 - delta]).sum(axis=1)
        total += (1.0 if delta == 0 else 2.0) * float(g @ g)
    return total


def fourth_moment_bidiagonal(d, e) -> float:
    """||B^T B||_F^2 of the upper bidiagonal (d, e): B^T B is tridiagonal with
    diagonal d_i^2 + e_{i-1}^2 and off-diagonal d_i e_i."""
    d = d.astype(np.float64)
    e = e.astype(np.float64)
    diag = d * d
    diag[1:] += e * e
    off = d[:-1] * e
    return float(diag @ diag + 2.0 * (off @ off))
