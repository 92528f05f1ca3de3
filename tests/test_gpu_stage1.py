"""Stage 1 on the GPU (bb_dense_to_band: dense -> upper band by block
Householder, panels plus matrix-product updates) against the oracle's stage 1 (oracle.dense_to_band), and the two
stages chained on the GPU (bb_dense_to_band, bb_pack_band, bb_reduce).

Bars:
  * the band entry by entry: max |G - O| <= 1e-12 ||A||_F (float64) or
    2e-5 ||A||_F (float32), G the GPU's result and O the oracle's (the same
    reflector sequence in the xLARFG convention; only rounding differs);
  * every entry outside the band is exactly zero;
  * the chain's singular values against LAPACK's SVD of the dense input:
    max |sigma - sigma_ref| <= 1e-12 sigma_1 (float64) or 2e-5 sigma_1
    (float32), and against a prescribed spectrum.
"""
import numpy as np
import pytest
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb
import oracle
from gpu_helpers import record, sigma_bidiagonal

pytestmark = pytest.mark.gpu

TOL = {"f64": 1e-12, "f32": 2e-5}


def gpu_stage1(a: np.ndarray, bw: int):
    """Stage 1 of the row-major numpy matrix a on cuda:0; returns the band
    as a row-major numpy array."""
    n = a.shape[0]
    dev = torch.device("cuda:0")
    dt = "f64" if a.dtype == np.float64 else "f32"
    code = bb.dtype_code(dt)
    x = torch.from_numpy(np.ascontiguousarray(a.T)).to(dev)  # column-major n x n
    nbytes = bb.bb_dense_to_band_workspace(n, bw, code)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev)
    bb.bb_dense_to_band(code, n, bw, x, n, ws, nbytes, s)
    torch.cuda.synchronize()
    return x.cpu().numpy().T.copy(), x


def outside_band_nonzeros(g: np.ndarray, bw: int) -> int:
    n = g.shape[0]
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return int(np.count_nonzero(g[(j - i < 0) | (j - i > bw)]))


@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("n,bw", [(1, 1), (2, 1), (5, 2), (9, 8), (40, 1), (64, 16), (100, 7), (200, 32),
                                  (257, 64), (513, 48), (300, 299)])
def test_stage1_matches_oracle(n, bw, dt):
    rng = np.random.default_rng(n + bw)
    a = rng.standard_normal((n, n)).astype(np.float32 if dt == "f32" else np.float64)
    ref = oracle.dense_to_band(a, bw)
    got, _ = gpu_stage1(a, bw)
    fro = max(float(np.linalg.norm(a.astype(np.float64))), 1e-300)
    err = float(np.abs(got.astype(np.float64) - ref.astype(np.float64)).max()) / fro
    record("stage1", n=n, bw=bw, dt=dt, err=err)
    assert err <= TOL[dt], f"band entries differ by {err:.3e} ||A||_F"
    assert outside_band_nonzeros(got, bw) == 0


@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("n,bw,tw", [(300, 16, 8), (512, 32, 16), (700, 64, 16)])
def test_two_stages_chained_on_the_gpu(n, bw, tw, dt):
    """dense -> band (stage 1) -> band storage -> bidiagonal (stage 2), all on
    the GPU; singular values against LAPACK's SVD of the dense input."""
    rng = np.random.default_rng(7 * n + bw)
    a = rng.standard_normal((n, n)).astype(np.float32 if dt == "f32" else np.float64)
    code = bb.dtype_code(dt)
    _, x = gpu_stage1(a, bw)
    dev = x.device
    ldab = bb.bb_required_ldab(bw, tw)
    band = torch.empty((n, ldab), dtype=x.dtype, device=dev)
    s = torch.cuda.current_stream(dev)
    bb.bb_pack_band(code, n, bw, tw, x, n, band, ldab, s)
    d = torch.empty(n, dtype=x.dtype, device=dev)
    e = torch.empty(n - 1, dtype=x.dtype, device=dev)
    h = bb.bb_create(n, bw, code)
    try:
        bb.bb_reduce(h, band, ldab, tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK
    finally:
        bb.bb_destroy(h)
    sigma = sigma_bidiagonal(d.cpu().numpy(), e.cpu().numpy())
    ref = np.linalg.svd(a.astype(np.float64), compute_uv=False)
    err = float(np.abs(sigma - ref).max()) / ref[0]
    record("two_stages", n=n, bw=bw, tw=tw, dt=dt, err=err)
    assert err <= TOL[dt], f"singular values differ by {err:.3e} sigma_1"


@pytest.mark.parametrize("n,bw,dt", [(1700, 16, "f64"), (3400, 16, "f32"), (3300, 16, "f64")])
def test_two_stages_chained_with_tall_panels(n, bw, dt):
    """Panels taller than 16 columns of shared memory hold (1600 doubles,
    3200 floats) run in narrower blocks (n = 1700 double, 3400 float); in
    double, blocks narrower than 8 are not used, so panels taller than 3200
    rows go to the global-memory panel kernel (n = 3300).  The chain's
    singular values against LAPACK's SVD of the input, and the exact band
    form."""
    rng = np.random.default_rng(n + bw)
    a = rng.standard_normal((n, n)).astype(np.float32 if dt == "f32" else np.float64)
    got, x = gpu_stage1(a, bw)
    assert outside_band_nonzeros(got, bw) == 0
    tw = 8
    code = bb.dtype_code(dt)
    ldab = bb.bb_required_ldab(bw, tw)
    band = torch.empty((n, ldab), dtype=x.dtype, device=x.device)
    s = torch.cuda.current_stream(x.device)
    bb.bb_pack_band(code, n, bw, tw, x, n, band, ldab, s)
    d = torch.empty(n, dtype=x.dtype, device=x.device)
    e = torch.empty(n - 1, dtype=x.dtype, device=x.device)
    h = bb.bb_create(n, bw, code)
    try:
        bb.bb_reduce(h, band, ldab, tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK
    finally:
        bb.bb_destroy(h)
    sigma = sigma_bidiagonal(d.cpu().numpy(), e.cpu().numpy())
    ref = np.linalg.svd(a.astype(np.float64), compute_uv=False)
    err = float(np.abs(sigma - ref).max()) / ref[0]
    record("two_stages_tall", n=n, bw=bw, dt=dt, err=err)
    assert err <= TOL[dt], f"singular values differ by {err:.3e} sigma_1"


@pytest.mark.parametrize("kind", bi.SPECTRA)
def test_two_stages_prescribed_spectrum(kind):
    n, bw, tw = 400, 32, 8
    sigma = bi.spectrum(kind, n, seed=n)
    rng = np.random.default_rng(11)
    u, _ = np.linalg.qr(rng.standard_normal((n, n)))
    v, _ = np.linalg.qr(rng.standard_normal((n, n)))
    a = (u * sigma) @ v.T
    _, x = gpu_stage1(a, bw)
    ldab = bb.bb_required_ldab(bw, tw)
    band = torch.empty((n, ldab), dtype=x.dtype, device=x.device)
    s = torch.cuda.current_stream(x.device)
    bb.bb_pack_band(bb.BB_F64, n, bw, tw, x, n, band, ldab, s)
    d = torch.empty(n, dtype=x.dtype, device=x.device)
    e = torch.empty(n - 1, dtype=x.dtype, device=x.device)
    h = bb.bb_create(n, bw, bb.BB_F64)
    try:
        bb.bb_reduce(h, band, ldab, tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK
    finally:
        bb.bb_destroy(h)
    got = sigma_bidiagonal(d.cpu().numpy(), e.cpu().numpy())
    assert np.abs(got - sigma).max() <= 1e-12 * sigma[0]


def test_pack_band_layout():
    """bb_pack_band writes A(i, j), 0 <= j - i <= bw, at band[(ku + i - j) +
    j ldab] and zero elsewhere (the layout of band_inputs)."""
    n, bw, tw = 50, 6, 3
    rng = np.random.default_rng(2)
    a = np.triu(rng.standard_normal((n, n)))
    a = np.triu(a) - np.triu(a, bw + 1)  # an upper band of bandwidth bw
    dev = torch.device("cuda:0")
    x = torch.from_numpy(np.ascontiguousarray(a.T)).to(dev)
    ldab = bw + 2 * tw + 1 + 2
    band = torch.full((n, ldab), 7.0, dtype=torch.float64, device=dev)
    bb.bb_pack_band(bb.BB_F64, n, bw, tw, x, n, band, ldab)
    torch.cuda.synchronize()
    want = bi.dense_to_band(a, bw + tw, ldab)
    assert np.array_equal(band.cpu().numpy(), want)


def test_stage1_argument_errors():
    dev = torch.device("cuda:0")
    n = 16
    x = torch.zeros((n, n), dtype=torch.float64, device=dev)
    nbytes = bb.bb_dense_to_band_workspace(n, 4, bb.BB_F64)
    assert nbytes == (18 * n * 4 + 16 + 8 + 64) * 8 and bb.bb_dense_to_band_workspace(0, 4, bb.BB_F64) == -1
    assert bb.bb_dense_to_band_workspace(n, 0, bb.BB_F64) == -1
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    with pytest.raises(bb.BBError):
        bb.bb_dense_to_band(bb.BB_F64, n, 4, x, n, ws, nbytes - 8)       # workspace too small
    with pytest.raises(bb.BBError):
        bb.bb_dense_to_band(bb.BB_F64, n, 0, x, n, ws, nbytes)           # bw < 1
    with pytest.raises(bb.BBError):
        bb.bb_dense_to_band(bb.BB_F64, n, 4, x.cpu(), n, ws, nbytes)     # host matrix
    with pytest.raises(bb.BBError) as ex:
        bb.bb_dense_to_band(bb.BB_F16, n, 4, x, n, ws, nbytes)
    assert ex.value.status == bb.BB_ERR_DTYPE
    band = torch.zeros((n, 5), dtype=torch.float64, device=dev)
    with pytest.raises(bb.BBError) as ex:
        bb.bb_pack_band(bb.BB_F64, n, 4, 1, x, n, band, 5)               # ldab < bw + 2 tw + 1
    assert ex.value.status == bb.BB_ERR_LDAB
