"""Parity of bb_sym_reduce (symmetric band -> tridiagonal, through the C ABI)
with the CPU oracle's symmetric variant.

Acceptance, as for the bidiagonal path (the oracle runs in the same
precision as the GPU):
  * eigenvalues of the tridiagonal: max |lambda - lambda_ref| / ||A||_F at
    most 1e-12 (float64) or 2e-5 (float32);
  * |d| and |e|: at most max(that tolerance, 4 x the oracle's own change
    under a one-ulp input perturbation), since the entries, unlike the
    eigenvalues, can be ill-conditioned functions of A;
  * stored entries below the subdiagonal are exactly zero afterwards;
  * prescribed eigenvalues of A = Q diag(lam) Q^T are recovered.
"""
import numpy as np
import pytest
import scipy.linalg as sla
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb
import oracle
from gpu_helpers import DE_FACTOR, TOL, de_error, record

pytestmark = pytest.mark.gpu


def tri_eigs(d, e):
    d = np.asarray(d, np.float64)
    return d.copy() if d.size == 1 else sla.eigvalsh_tridiagonal(d, np.asarray(e, np.float64))


def sym_fro(sb, n):
    a = sb.astype(np.float64)
    return float(np.sqrt((a[:, 0] ** 2).sum() + 2 * (a[:, 1:] ** 2).sum()))


def gpu_sym(sb, n, bw, tw, dt, params=None, return_band=False):
    dev = torch.device("cuda:0")
    x = torch.from_numpy(np.ascontiguousarray(sb)).to(dev)
    d = torch.empty(n, dtype=x.dtype, device=dev)
    e = torch.empty(max(n - 1, 1), dtype=x.dtype, device=dev)
    h = bb.bb_create(n, bw, bb.dtype_code(dt))
    try:
        for k, v in (params or {}).items():
            bb.bb_set_param(h, k, v)
        s = torch.cuda.current_stream(dev)
        bb.bb_sym_reduce(h, x, sb.shape[1], tw, d, e, s)
        st = bb.bb_status_sync(h, s)
        assert st == bb.BB_OK, f"device status {st}: {bb.bb_last_error()}"
    finally:
        bb.bb_destroy(h)
    out = (d.cpu().numpy(), e[: max(n - 1, 0)].cpu().numpy())
    return out + (x.cpu().numpy(),) if return_band else out


def sym_sensitivity(sb, n, bw, tw, seeds=bi.SENSITIVITY_SEEDS):
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    fro = sym_fro(sb, n)
    worst = 0.0
    for sd in seeds:
        d2, e2 = oracle.tridiagonal(bi.perturb_ulp(sb, sd), n, bw, tw)
        worst = max(worst, de_error(d2, e2, d, e, fro))
    return worst


def check(sb, n, bw, tw, dt, params=None):
    d_ref, e_ref = oracle.tridiagonal(sb, n, bw, tw)
    d, e, after = gpu_sym(sb, n, bw, tw, dt, params, return_band=True)
    fro = max(sym_fro(sb, n), 1e-300)
    lerr = float(np.abs(np.sort(tri_eigs(d, e)) - np.sort(tri_eigs(d_ref, e_ref))).max()) / fro
    err = de_error(d, e, d_ref, e_ref, fro)
    tol = TOL[dt]
    if err > tol:
        tol = max(tol, DE_FACTOR * sym_sensitivity(sb, n, bw, tw))
    record("sym_parity", n=n, bw=bw, tw=tw, dt=dt, eig_err=lerr, de_err=err, de_tol=tol)
    assert lerr <= TOL[dt], f"eigenvalue error {lerr:.3e}"
    assert err <= tol, f"|d|,|e| error {err:.3e} > {tol:.3e}"
    assert np.count_nonzero(after[:, 2:]) == 0


CASES = [(1, 0, 1), (2, 1, 1), (3, 2, 1), (5, 3, 2), (8, 4, 3), (16, 8, 7), (24, 6, 2), (33, 10, 4),
         (40, 8, 7), (48, 12, 5), (64, 16, 8), (64, 16, 15), (70, 17, 16), (97, 33, 32), (130, 64, 32),
         (300, 100, 33), (257, 128, 64), (600, 96, 32), (1000, 64, 16)]


@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("n,bw,tw", CASES)
def test_edge_cases(n, bw, tw, dt):
    check(bi.make_sym_band(n, bw, tw, dt, seed=n + 17 * bw + tw), n, bw, tw, dt)


@pytest.mark.parametrize("n,bw,tw,dt", [(4096, 16, 8, "f32"), (4096, 64, 16, "f32"), (2048, 128, 32, "f64")])
def test_larger_bands(n, bw, tw, dt):
    check(bi.make_sym_band(n, bw, tw, dt, "uniform", seed=n + bw), n, bw, tw, dt)


@pytest.mark.parametrize("max_ctas", [1, 3, 17])
def test_fewer_ctas_than_sweeps(max_ctas):
    # CTAs take several sweeps each and wait on sweeps of other CTAs
    n, bw, tw = 500, 24, 7
    check(bi.make_sym_band(n, bw, tw, "f64", seed=3), n, bw, tw, "f64", {bb.BB_PARAM_MAX_CTAS: max_ctas})


def test_larger_ldab():
    n, bw, tw = 300, 20, 6
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=4, ldab=bw + tw + 9)
    check(sb, n, bw, tw, "f64")


@pytest.mark.parametrize("kind", bi.SPECTRA + ("rank_deficient",))
@pytest.mark.parametrize("dt", ["f64", "f32"])
def test_prescribed_eigenvalues(kind, dt):
    n, bw, tw = 512, 32, 8
    lam = bi.spectrum(kind, n, seed=n + bw) * np.where(np.arange(n) % 2, -1.0, 1.0)
    sb = bi.make_sym_band_with_spectrum(n, bw, tw, lam, dt, seed=5 * n + tw)
    d, e = gpu_sym(sb, n, bw, tw, dt)
    got = np.sort(tri_eigs(d, e))
    assert np.abs(got - np.sort(lam)).max() <= TOL[dt] * np.abs(lam).max()


def test_stalled_sweep_times_out_and_context_survives():
    n, bw, tw = 800, 16, 8
    sb = bi.make_sym_band(n, bw, tw, "f32", seed=2)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(sb).to(dev)
    d = torch.empty(n, dtype=torch.float32, device=dev)
    e = torch.empty(n - 1, dtype=torch.float32, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F32)
    try:
        bb.bb_set_param(h, bb.BB_PARAM_WAIT_BUDGET_MS, 50)
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, 5)
        s = torch.cuda.current_stream(dev)
        bb.bb_sym_reduce(h, x, sb.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_ERR_TIMEOUT
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, -1)
        x.copy_(torch.from_numpy(sb).to(dev))
        bb.bb_sym_reduce(h, x, sb.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK
    finally:
        bb.bb_destroy(h)


def test_argument_errors():
    n, bw, tw = 100, 10, 3
    dev = torch.device("cuda:0")
    x = torch.zeros((n, bw + tw + 1), dtype=torch.float64, device=dev)
    d = torch.empty(n, dtype=torch.float64, device=dev)
    e = torch.empty(n - 1, dtype=torch.float64, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F64)
    try:
        with pytest.raises(bb.BBError) as ex:
            bb.bb_sym_reduce(h, x, bw + tw, tw, d, e)            # ldab too small
        assert ex.value.status == bb.BB_ERR_LDAB
        with pytest.raises(bb.BBError):
            bb.bb_sym_reduce(h, x, bw + tw + 1, bw, d, e)        # tw > bw - 1
        with pytest.raises(bb.BBError):
            bb.bb_sym_reduce(h, x.cpu(), bw + tw + 1, tw, d, e)  # host band
    finally:
        bb.bb_destroy(h)
    assert bb.bb_sym_required_ldab(bw, tw) == bw + tw + 1
