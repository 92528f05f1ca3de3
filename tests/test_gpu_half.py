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
        # the group kernel (3) where at least 5 sweeps' binary16 columns fit,
        # else the binary16 flag kernel (5)
        want = [3 if bb.bb_group_plan(n, bw, tw, 2, p)[0] >= 5 else 5 for p in range(bb.bb_num_passes(bw, tw))]
        assert [bb.bb_last_pass_kernel(h, i) for i in range(bb.bb_last_num_passes(h))] == want
        assert 3 in want
    finally:
        bb.bb_destroy(h)
    assert np.array_equal(src, band)
    assert np.array_equal(d, d0) and np.array_equal(e, e0)


def half_kernels(band, n, bw, tw, params):
    """(d, e, band after, [(kernel, group) per pass]) of bb_reduce on cuda:0."""
    dev = torch.device("cuda:0")
    x = torch.from_numpy(np.ascontiguousarray(band)).to(dev)
    d = torch.empty(n, dtype=x.dtype, device=dev)
    e = torch.empty(max(n - 1, 1), dtype=x.dtype, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F16)
    try:
        for k, v in params.items():
            bb.bb_set_param(h, k, v)
        s = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK, bb.bb_last_error()
        ks = [(bb.bb_last_pass_kernel(h, i), bb.bb_last_pass_group(h, i)) for i in range(bb.bb_last_num_passes(h))]
    finally:
        bb.bb_destroy(h)
    return d.cpu().numpy(), e[: max(n - 1, 0)].cpu().numpy(), x.cpu().numpy(), ks


# one and several groups, ragged tails, reflectors of 8, 9, 13, 17 and 33
# elements, b - t = 1 passes; ldab of the storage layout (unaligned: through
# the working copy) and padded to a multiple of 8 (aligned: in place)
HALF_GROUP_CASES = [(64, 16, 8, None), (257, 8, 7, None), (300, 40, 12, None), (1000, 64, 16, None),
                    (600, 96, 32, None), (2000, 16, 8, None), (700, 24, 8, 48), (513, 33, 16, 72)]


@pytest.mark.parametrize("n,bw,tw,ldab", HALF_GROUP_CASES)
def test_half_group_kernel_bitwise_equals_flag_kernel(n, bw, tw, ldab):
    band = half_band(n, bw, tw, seed=n + bw, ldab=ldab)
    d2, e2, b2, k2 = half_kernels(band, n, bw, tw, {bb.BB_PARAM_SCHEDULER: 2})
    d3, e3, b3, k3 = half_kernels(band, n, bw, tw, {bb.BB_PARAM_SCHEDULER: 3})
    assert all(k == 5 for k, _ in k2)
    planned = [bb.bb_group_plan(n, bw, tw, 2, p)[0] for p in range(len(k3))]
    assert [k for k, _ in k3] == [3 if g > 0 else 5 for g in planned] and 3 in [k for k, _ in k3]
    record("half_group_vs_flag", n=n, bw=bw, tw=tw, kernels=k3)
    assert np.array_equal(d2, d3) and np.array_equal(e2, e3)
    assert np.array_equal(b2.view(np.uint16), b3.view(np.uint16))


@pytest.mark.parametrize("group_size,max_ctas", [(1, 0), (3, 2), (13, 1), (6, 0)])
def test_half_group_sizes_and_grid_caps(group_size, max_ctas):
    n, bw, tw = 700, 16, 8
    band = half_band(n, bw, tw, seed=9)
    ref = half_kernels(band, n, bw, tw, {bb.BB_PARAM_SCHEDULER: 2})
    got = half_kernels(band, n, bw, tw, {bb.BB_PARAM_SCHEDULER: 3, bb.BB_PARAM_GROUP_SIZE: group_size,
                                         bb.BB_PARAM_MAX_CTAS: max_ctas})
    assert got[3] == [(3, group_size)] * len(got[3])
    for a, b in zip(ref[:3], got[:3]):
        assert np.array_equal(np.asarray(a).view(np.uint16), np.asarray(b).view(np.uint16))


@pytest.mark.parametrize("scheduler", [2, 3])
def test_half_stalled_sweep_times_out_and_context_survives(scheduler):
    n, bw, tw = 800, 16, 8
    band = half_band(n, bw, tw, seed=2)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(band).to(dev)
    d = torch.empty(n, dtype=torch.float16, device=dev)
    e = torch.empty(n - 1, dtype=torch.float16, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F16)
    try:
        bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, scheduler)
        bb.bb_set_param(h, bb.BB_PARAM_WAIT_BUDGET_MS, 50)
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, 5)
        s = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_ERR_TIMEOUT
        assert bb.bb_last_pass_kernel(h, 0) == (3 if scheduler == 3 else 5)
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


def test_half_group_kernel_on_unaligned_band_pointer():
    """A binary16 band one element past a 16-byte boundary (column stride a
    multiple of 16 bytes): the group kernel runs on the aligned working
    copy, bitwise equal to the binary16 flag kernel; nothing outside the
    band is written."""
    n, bw, tw = 500, 24, 8
    ld = (bw + 2 * tw + 1 + 7) // 8 * 8
    band = half_band(n, bw, tw, seed=31, ldab=ld)
    dev = torch.device("cuda:0")

    def run(sched):
        flat = torch.zeros(n * ld + 2, dtype=torch.float16, device=dev)
        x = flat[1:-1].view(n, ld)
        x.copy_(torch.from_numpy(band))
        assert x.data_ptr() % 16 != 0
        d = torch.empty(n, dtype=torch.float16, device=dev)
        e = torch.empty(n - 1, dtype=torch.float16, device=dev)
        h = bb.bb_create(n, bw, bb.BB_F16)
        try:
            bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, sched)
            s = torch.cuda.current_stream(dev)
            bb.bb_reduce(h, x, ld, tw, d, e, s)
            assert bb.bb_status_sync(h, s) == bb.BB_OK
            ks = [bb.bb_last_pass_kernel(h, i) for i in range(bb.bb_last_num_passes(h))]
        finally:
            bb.bb_destroy(h)
        assert flat[0].item() == 0.0 and flat[-1].item() == 0.0
        return d.cpu().numpy(), e.cpu().numpy(), x.cpu().numpy(), ks

    d3, e3, b3, k3 = run(3)
    d2, e2, b2, k2 = run(2)
    assert 3 in k3 and all(k == 5 for k in k2)
    assert np.array_equal(d2.view(np.uint16), d3.view(np.uint16))
    assert np.array_equal(e2.view(np.uint16), e3.view(np.uint16))
    assert np.array_equal(b2.view(np.uint16), b3.view(np.uint16))
