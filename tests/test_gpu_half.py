"""Binary16 storage on the GPU (BB_F16): the band, d and e in IEEE binary16,
the arithmetic in float ("Accelerating Bidiagonalization of Banded Matrices
through Memory-Aware Bulge-Chasing on GPUs", Section V, runs the method in
FP16 too), against the oracle's binary16-storage variant (the same reading:
every write rounded to binary16).

Bars, with u = 2^-11 the unit roundoff of binary16 (those of the oracle's own
pins in tests/test_oracle_half.py):
  * singular values: max |sigma - sigma_ref| <= 4 u ||A||_F, against the
    binary16 oracle and against the float64 oracle on the same input;
  * |d|, |e| against the binary16 oracle: at most max(4 u, 4 x the binary16
    oracle's own change under a one-ulp input perturbation) ||A||_F;
  * prescribed spectra: ||sigma - sigma_exact|| <= 4 u ||sigma_exact||;
  * every stored entry off the bidiagonal is exactly zero afterwards.
"""
import numpy as np
import pytest
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb
import oracle
from gpu_helpers import DE_FACTOR, de_error, fro_of_band, gpu_reduce, off_bidiagonal_nonzeros, oracle_sensitivity, \
    record, sigma_bidiagonal

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not oracle.has_half(), reason="oracle built without _Float16")]

U16 = 2.0 ** -11
TOL16 = 4 * U16


def half_band(n, bw, tw, seed, dist="uniform", ldab=None):
    return bi.make_band(n, bw, tw, "f64", dist, seed=seed, ldab=ldab).astype(np.float16)


def check_half(band, n, bw, tw):
    d_ref, e_ref = oracle.bidiagonal(band, n, bw, tw)
    d, e, after = gpu_reduce(band, n, bw, tw, "f16", 0, return_band=True)
    assert d.dtype == np.float16
    fro = max(fro_of_band(band), 1e-300)
    serr = float(np.abs(sigma_bidiagonal(d, e) - sigma_bidiagonal(d_ref, e_ref)).max()) / fro if n else 0.0
    err = de_error(d, e, d_ref, e_ref, fro)
    tol = TOL16
    sens = None
    if err > tol:
        sens = oracle_sensitivity(band, n, bw, tw)
        tol = max(tol, DE_FACTOR * sens)
    record("half_parity", n=n, bw=bw, tw=tw, sigma_err=serr, de_err=err, de_sens=sens, de_tol=tol)
    assert serr <= TOL16, f"sigma error {serr:.3e} > {TOL16:.3e}"
    assert err <= tol, f"|d|,|e| error {err:.3e} > {tol:.3e}"
    assert off_bidiagonal_nonzeros(after, n, bw + tw) == 0
    return d, e


CASES = [(1, 0, 1), (2, 1, 1), (5, 3, 2), (16, 8, 7), (33, 10, 4), (64, 16, 8), (64, 16, 15), (70, 17, 16),
         (97, 33, 32), (300, 100, 33), (257, 128, 64), (600, 96, 32), (1000, 64, 16), (777, 256, 32)]


@pytest.mark.parametrize("n,bw,tw", CASES)
def test_half_edge_cases(n, bw, tw):
    check_half(half_band(n, bw, tw, seed=n + 17 * bw + tw), n, bw, tw)


def test_half_main_workload_recipe_full_size():
    """n = 4096, bw = 16, tw = 8 with U[-1, 1] entries (the main workload's
    recipe) in binary16 storage."""
    w = bi.WORKLOADS[1]
    check_half(bi.make_band(w.n, w.bw, w.tw, "f64", w.dist, seed=w.seed).astype(np.float16), w.n, w.bw, w.tw)


@pytest.mark.parametrize("n,bw,tw", [(512, 16, 8), (1500, 64, 16), (2111, 256, 32)])
def test_half_accuracy_against_float64(n, bw, tw):
    band = half_band(n, bw, tw, seed=n, dist="normal")
    d, e = gpu_reduce(band, n, bw, tw, "f16", 0)
    d64, e64 = oracle.bidiagonal(band.astype(np.float64), n, bw, tw)
    fro = fro_of_band(band)
    s = sigma_bidiagonal(d, e)
    s64 = oracle.bidiagonal_singular_values(d64, e64)
    record("half_vs_f64", n=n, bw=bw, tw=tw, sigma_err=float(np.abs(s - s64).max() / fro))
    assert np.abs(s - s64).max() <= TOL16 * fro
    assert np.linalg.norm(s - s64) <= TOL16 * np.linalg.norm(s64)


@pytest.mark.parametrize("kind", bi.SPECTRA)
def test_half_prescribed_spectrum(kind):
    n, bw, tw = 512, 32, 8
    sigma = bi.spectrum(kind, n, seed=n + bw)
    band = bi.make_band_with_spectrum(n, bw, tw, sigma, seed=5 * n).astype(np.float16)
    d, e = gpu_reduce(band, n, bw, tw, "f16", 0)
    got = sigma_bidiagonal(d, e)
    assert np.linalg.norm(got - sigma) <= TOL16 * np.linalg.norm(sigma)


def test_half_host_entry_and_grid_independence():
    n, bw, tw = 900, 40, 12
    band = half_band(n, bw, tw, seed=4)
    d0, e0 = gpu_reduce(band, n, bw, tw, "f16", 0)
    d1, e1 = gpu_reduce(band, n, bw, tw, "f16", 0, {bb.BB_PARAM_MAX_CTAS: 5})
    assert np.array_equal(d0, d1) and np.array_equal(e0, e1)
    h = bb.bb_create(n, bw, bb.BB_F16)
    try:
        d = np.zeros(n, np.float16)
        e = np.zeros(n - 1, np.float16)
        src = band.copy()
        bb.bb_reduce_host(h, src, band.shape[1], tw, d, e)
        assert [bb.bb_last_pass_kernel(h, i) for i in range(bb.bb_last_num_passes(h))] == \
            [5] * bb.bb_num_passes(bw, tw)
    finally:
        bb.bb_destroy(h)
    assert np.array_equal(src, band)
    assert np.array_equal(d, d0) and np.array_equal(e, e0)


def test_half_stalled_sweep_times_out_and_context_survives():
    n, bw, tw = 800, 16, 8
    band = half_band(n, bw, tw, seed=2)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(band).to(dev)
    d = torch.empty(n, dtype=torch.float16, device=dev)
    e = torch.empty(n - 1, dtype=torch.float16, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F16)
    try:
        bb.bb_set_param(h, bb.BB_PARAM_WAIT_BUDGET_MS, 50)
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, 5)
        s = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_ERR_TIMEOUT
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, -1)
        x.copy_(torch.from_numpy(band).to(dev))
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK
    finally:
        bb.bb_destroy(h)


def test_half_entry_points_that_do_not_take_it():
    n, bw, tw = 100, 10, 3
    dev = torch.device("cuda:0")
    h = bb.bb_create(n, bw, bb.BB_F16)
    x = torch.zeros((n, bw + tw + 1), dtype=torch.float16, device=dev)
    d = torch.empty(n, dtype=torch.float16, device=dev)
    e = torch.empty(n - 1, dtype=torch.float16, device=dev)
    try:
        with pytest.raises(bb.BBError) as ex:
            bb.bb_sym_reduce(h, x, bw + tw + 1, tw, d, e)
        assert ex.value.status == bb.BB_ERR_DTYPE
    finally:
        bb.bb_destroy(h)
    sig = torch.empty(n, dtype=torch.float16, device=dev)
    with pytest.raises(bb.BBError):
        bb.bb_singular_values(bb.BB_F16, n, d, e, sig)
    xb = torch.zeros((n, bw + 2 * tw + 1), dtype=torch.float16, device=dev)
    with pytest.raises(bb.BBError):
        bb.bb_reduce_noalloc(xb, n, bw, bw + 2 * tw + 1, tw, bb.BB_F16, d, e)
