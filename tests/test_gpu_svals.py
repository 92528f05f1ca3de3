"""bb_singular_values (bisection on the Golub-Kahan tridiagonal) against the
oracle's singular values of the same bidiagonal.

Acceptance: max |sigma - sigma_ref| / ||B||_F at most 1e-12 (float64) or
2e-5 (float32), the tolerances of the reduction's own singular values.  The
bisection stops at about one ulp of the Gershgorin bound, so it meets them
with room.
"""
import numpy as np
import pytest
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb
import oracle

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-5, "f64": 1e-12}


def gpu_svals(d: np.ndarray, e: np.ndarray, dt: str) -> np.ndarray:
    dev = torch.device("cuda:0")
    tdt = torch.float32 if dt == "f32" else torch.float64
    n = d.size
    dd = torch.from_numpy(np.ascontiguousarray(d)).to(dev, tdt)
    ee = torch.from_numpy(np.ascontiguousarray(e if n > 1 else np.zeros(1))).to(dev, tdt)
    s = torch.empty(n, dtype=tdt, device=dev)
    bb.bb_singular_values(bb.dtype_code(dt), n, dd, ee if n > 1 else None, s, torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    return s.cpu().numpy()


def check(d, e, dt):
    got = gpu_svals(d, e, dt).astype(np.float64)
    want = oracle.bidiagonal_singular_values(d.astype(np.float64), e.astype(np.float64))
    a = np.abs(np.r_[d.astype(np.float64), e.astype(np.float64)])
    amax = float(a.max()) if a.size else 0.0
    # ||B||_F, scaled so that the squares of tiny entries do not underflow
    fro = max(amax * float(np.sqrt(((a / amax) ** 2).sum())) if amax > 0 else 0.0, np.finfo(np.float64).tiny)
    err = float(np.abs(got - want).max()) / fro if d.size else 0.0
    assert err <= TOL[dt], (d.size, dt, err)
    assert np.all(np.diff(got) <= 0)  # descending
    return err


@pytest.mark.parametrize("dt", ["f32", "f64"])
@pytest.mark.parametrize("n", [1, 2, 3, 17, 127, 128, 129, 1000, 2049, 4097])
def test_random_bidiagonals(n, dt):
    rng = np.random.default_rng(n)
    npdt = np.float32 if dt == "f32" else np.float64
    d = rng.normal(size=n).astype(npdt)
    e = rng.normal(size=max(n - 1, 0)).astype(npdt)
    check(d, e, dt)


@pytest.mark.parametrize("dt", ["f32", "f64"])
def test_special_bidiagonals(dt):
    npdt = np.float32 if dt == "f32" else np.float64
    n = 300
    check(np.zeros(n, npdt), np.zeros(n - 1, npdt), dt)                      # all zero
    check(np.linspace(-3, 3, n).astype(npdt), np.zeros(n - 1, npdt), dt)     # diagonal
    check(np.ones(n, npdt), np.ones(n - 1, npdt), dt)                        # path graph
    g = (10.0 ** (-8.0 * np.arange(n) / n)).astype(npdt)                     # graded
    rng = np.random.default_rng(9)
    check((rng.normal(size=n) * g).astype(npdt), (rng.normal(size=n - 1) * g[1:]).astype(npdt), dt)
    tiny = np.float32(1e-30) if dt == "f32" else 1e-290                      # near underflow
    check((rng.normal(size=n) * tiny).astype(npdt), (rng.normal(size=n - 1) * tiny).astype(npdt), dt)


@pytest.mark.parametrize("idx", [0, 1])
def test_after_the_reduction(idx):
    """The two stages chained on the GPU: reduce a workload band, then take
    the singular values of its bidiagonal; against the oracle's reduction and
    its singular values."""
    w = bi.WORKLOADS[idx]
    band = bi.make_workload(w)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(band).to(dev)
    d = torch.empty(w.n, dtype=x.dtype, device=dev)
    e = torch.empty(max(w.n - 1, 1), dtype=x.dtype, device=dev)
    s = torch.empty(w.n, dtype=x.dtype, device=dev)
    h = bb.bb_create(w.n, w.bw, bb.dtype_code(w.dtype))
    try:
        st = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], w.tw, d, e, st)
        bb.bb_singular_values(bb.dtype_code(w.dtype), w.n, d, e, s, st)
        assert bb.bb_status_sync(h, st) == bb.BB_OK
    finally:
        bb.bb_destroy(h)
    d_ref, e_ref = oracle.bidiagonal(band, w.n, w.bw, w.tw)
    want = oracle.bidiagonal_singular_values(d_ref, e_ref)
    fro = float(np.linalg.norm(band.astype(np.float64)))
    err = float(np.abs(s.cpu().numpy().astype(np.float64) - want).max()) / fro
    assert err <= TOL[w.dtype], err


@pytest.mark.parametrize("n", [32768, 40000, 80000])
def test_full_size_properties(n):
    """n = 32768 (the largest workload's order) and beyond, float32 (the lane
    group per value shrinks with n: 4, 2 and 1 lanes here): descending,
    bounded by the Gershgorin bound, and sum sigma^2 = ||B||_F^2; against the
    oracle at n = 32768."""
    rng = np.random.default_rng(4)
    d = rng.normal(size=n).astype(np.float32)
    e = rng.normal(size=n - 1).astype(np.float32)
    got = gpu_svals(d, e, "f32").astype(np.float64)
    assert np.all(np.diff(got) <= 0) and got[-1] >= 0
    bound = max(np.abs(np.r_[0, e]) + np.abs(d)).max() + np.abs(d).max()
    assert got[0] <= bound
    fro2 = float((d.astype(np.float64) ** 2).sum() + (e.astype(np.float64) ** 2).sum())
    assert abs((got ** 2).sum() - fro2) / fro2 < 1e-5
    if n == 32768:
        want = oracle.bidiagonal_singular_values(d, e)
        assert float(np.abs(got - want).max()) / np.sqrt(fro2) <= TOL["f32"]


def test_argument_errors():
    with pytest.raises(bb.BBError):
        bb.bb_singular_values(bb.BB_F32, 0, 1, 1, 1)
    with pytest.raises(bb.BBError):
        bb.bb_singular_values(bb.BB_F32, 5, None, None, None)


@pytest.mark.parametrize("lanes", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("dt", ["f32", "f64"])
def test_every_lane_count(lanes, dt):
    # the step count follows the lanes (each step keeps one of lanes + 1 parts)
    rng = np.random.default_rng(lanes)
    n = 700
    d = rng.standard_normal(n).astype(np.float32 if dt == "f32" else np.float64)
    e = rng.standard_normal(n - 1).astype(d.dtype)
    dev = torch.device("cuda:0")
    tdt = torch.float32 if dt == "f32" else torch.float64
    dd = torch.from_numpy(d).to(dev)
    ee = torch.from_numpy(e).to(dev)
    s = torch.empty(n, dtype=tdt, device=dev)
    bb.bb_singular_values_lanes(bb.dtype_code(dt), n, dd, ee, s, lanes, torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    got = s.cpu().numpy().astype(np.float64)
    want = oracle.bidiagonal_singular_values(d.astype(np.float64), e.astype(np.float64))
    fro = float(np.sqrt((d.astype(np.float64) ** 2).sum() + (e.astype(np.float64) ** 2).sum()))
    assert np.abs(got - want).max() <= TOL[dt] * fro
