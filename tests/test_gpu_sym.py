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


def gpu_sym(sb, n, bw, tw, dt, params=None, return_band=False, kernels=None):
    """bb_sym_reduce of the lower band sb on cuda:0: (d, e[, band after]).
    kernels: a list that receives (kernel, group size) of every pass."""
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
        if kernels is not None:
            kernels.extend((bb.bb_last_pass_kernel(h, i), bb.bb_last_pass_group(h, i))
                           for i in range(bb.bb_last_num_passes(h)))
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


# Shapes for the group kernel: one and several groups, ragged last groups,
# reflectors of 8, 9, 17 and 33 elements (the compiled widths and a
# predicated one), passes with b - t = 1 (lag 3), float and double.
GROUP_CASES = [(40, 8, 7, "f64"), (64, 16, 8, "f32"), (129, 9, 8, "f64"), (257, 8, 7, "f32"),
               (300, 40, 12, "f64"), (500, 24, 7, "f32"), (1000, 64, 16, "f32"), (700, 48, 16, "f64"),
               (600, 96, 32, "f32"), (400, 66, 32, "f64"), (2000, 16, 8, "f32"), (1500, 32, 8, "f64")]


@pytest.mark.parametrize("n,bw,tw,dt", GROUP_CASES)
def test_group_kernel_bitwise_equals_flag_kernel(n, bw, tw, dt):
    """The two schedulers run the same arithmetic in the same order per
    entry: any difference is a race or a lost update."""
    sb = bi.make_sym_band(n, bw, tw, dt, seed=7 * n + bw)
    kf, kg = [], []
    d2, e2, b2 = gpu_sym(sb, n, bw, tw, dt, {bb.BB_PARAM_SCHEDULER: 2}, return_band=True, kernels=kf)
    d3, e3, b3 = gpu_sym(sb, n, bw, tw, dt, {bb.BB_PARAM_SCHEDULER: 3}, return_band=True, kernels=kg)
    assert all(k == 2 for k, _ in kf)
    planned = [bb.bb_sym_group_plan(n, bw, tw, 4 if dt == "f32" else 8, p)[0] for p in range(len(kg))]
    assert [k for k, _ in kg] == [3 if g > 0 else 2 for g in planned]
    assert any(k == 3 for k, _ in kg)
    record("sym_group_vs_flag", n=n, bw=bw, tw=tw, dt=dt, kernels=kg)
    assert np.array_equal(d2, d3) and np.array_equal(e2, e3)
    assert np.array_equal(b2, b3)


@pytest.mark.parametrize("group_size,max_ctas", [(1, 0), (2, 3), (5, 1), (13, 2), (7, 0)])
def test_group_kernel_group_sizes_and_grid_caps(group_size, max_ctas):
    """Groups of any size, and fewer CTAs than groups (each CTA then runs
    several groups in turn and waits on other CTAs' watermarks)."""
    n, bw, tw, dt = 700, 16, 8, "f32"
    sb = bi.make_sym_band(n, bw, tw, dt, seed=11)
    ref = gpu_sym(sb, n, bw, tw, dt, {bb.BB_PARAM_SCHEDULER: 2}, return_band=True)
    ks = []
    got = gpu_sym(sb, n, bw, tw, dt, {bb.BB_PARAM_SCHEDULER: 3, bb.BB_PARAM_GROUP_SIZE: group_size,
                                      bb.BB_PARAM_MAX_CTAS: max_ctas}, return_band=True, kernels=ks)
    assert ks == [(3, group_size)] * len(ks)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("n,bw,tw,dt", [(1000, 64, 16, "f32"), (700, 48, 16, "f64"), (2000, 16, 8, "f32")])
def test_group_kernel_parity(n, bw, tw, dt):
    check(bi.make_sym_band(n, bw, tw, dt, seed=n + 3 * bw), n, bw, tw, dt, {bb.BB_PARAM_SCHEDULER: 3})


def test_automatic_scheduler_takes_the_group_kernel():
    # the main workload's shape: both passes on the group kernel, 13 sweeps
    # per group; ldab = bw + tw + 1 is not a multiple of 16 bytes, so the
    # handle's aligned working copy is used (and the band is copied back)
    n, bw, tw, dt = 4096, 16, 8, "f32"
    sb = bi.make_sym_band(n, bw, tw, dt, seed=5)
    ks = []
    d, e, after = gpu_sym(sb, n, bw, tw, dt, return_band=True, kernels=ks)
    assert ks == [(3, 13), (3, 13)]
    d2, e2, after2 = gpu_sym(sb, n, bw, tw, dt, {bb.BB_PARAM_SCHEDULER: 2}, return_band=True)
    assert np.array_equal(d, d2) and np.array_equal(e, e2) and np.array_equal(after, after2)


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


@pytest.mark.parametrize("scheduler", [2, 3])
def test_stalled_sweep_times_out_and_context_survives(scheduler):
    """A sweep (flag kernel) or the group holding it (group kernel) that
    never reports progress: the waits give up, the status says so, and the
    context runs the next reduction."""
    n, bw, tw = 800, 16, 8
    sb = bi.make_sym_band(n, bw, tw, "f32", seed=2)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(sb).to(dev)
    d = torch.empty(n, dtype=torch.float32, device=dev)
    e = torch.empty(n - 1, dtype=torch.float32, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F32)
    try:
        bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, scheduler)
        bb.bb_set_param(h, bb.BB_PARAM_WAIT_BUDGET_MS, 50)
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, 5)
        s = torch.cuda.current_stream(dev)
        bb.bb_sym_reduce(h, x, sb.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_ERR_TIMEOUT
        assert bb.bb_last_pass_kernel(h, 0) == scheduler
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


@pytest.mark.parametrize("dt", ["f32", "f64"])
def test_group_kernel_on_unaligned_band_pointer(dt):
    """A band that starts one element past a 16-byte boundary, with a
    16-byte aligned column stride: the group kernel runs on the handle's
    aligned working copy, and the result (band included) equals the flag
    kernel's on the same storage; nothing outside the band is written."""
    n, bw, tw = 600, 24, 8
    q = 4 if dt == "f32" else 2
    ld = (bw + tw + 1 + q - 1) // q * q
    sb = bi.make_sym_band(n, bw, tw, dt, seed=21, ldab=ld)
    dev = torch.device("cuda:0")
    tdt = torch.float32 if dt == "f32" else torch.float64

    def run(sched):
        flat = torch.zeros(n * ld + 2, dtype=tdt, device=dev)
        x = flat[1:-1].view(n, ld)
        x.copy_(torch.from_numpy(sb))
        assert x.data_ptr() % 16 != 0
        d = torch.empty(n, dtype=tdt, device=dev)
        e = torch.empty(n - 1, dtype=tdt, device=dev)
        h = bb.bb_create(n, bw, bb.dtype_code(dt))
        try:
            bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, sched)
            s = torch.cuda.current_stream(dev)
            bb.bb_sym_reduce(h, x, ld, tw, d, e, s)
            assert bb.bb_status_sync(h, s) == bb.BB_OK
            ks = [bb.bb_last_pass_kernel(h, i) for i in range(bb.bb_last_num_passes(h))]
        finally:
            bb.bb_destroy(h)
        assert flat[0].item() == 0.0 and flat[-1].item() == 0.0
        return d.cpu().numpy(), e.cpu().numpy(), x.cpu().numpy(), ks

    d3, e3, b3, k3 = run(3)
    d2, e2, b2, k2 = run(2)
    assert 3 in k3 and all(k == 2 for k in k2)
    assert np.array_equal(d2, d3) and np.array_equal(e2, e3) and np.array_equal(b2, b3)
