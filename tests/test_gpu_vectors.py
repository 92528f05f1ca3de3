"""Back-transformation on the GPU (BB_PARAM_RECORD + bb_back_transform),
checked by what fixes U and V whatever the rounding of the reflectors:
A = U B V^T with B the GPU's bidiagonal, U and V orthogonal, U e_1 = V e_1 =
e_1 exactly (no reflector touches column 0), and the singular vectors
A (V V_b) = (U U_b) S.  The oracle's own U, V (bidiagonal_with_vectors) give
the same reconstruction on the same input."""
import numpy as np
import pytest
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb
import oracle

pytestmark = pytest.mark.gpu

TOL = {"f64": 1e-12, "f32": 2e-5}


def gpu_vectors(band, n, bw, tw, dt):
    dev = torch.device("cuda:0")
    tdt = torch.float32 if dt == "f32" else torch.float64
    x = torch.from_numpy(np.ascontiguousarray(band)).to(dev)
    d = torch.empty(n, dtype=tdt, device=dev)
    e = torch.empty(max(n - 1, 1), dtype=tdt, device=dev)
    U = torch.empty((n, n), dtype=tdt, device=dev)   # column-major: U[j] is column j
    V = torch.empty((n, n), dtype=tdt, device=dev)
    h = bb.bb_create(n, bw, bb.dtype_code(dt))
    try:
        bb.bb_set_param(h, bb.BB_PARAM_RECORD, 1)
        s = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        bb.bb_back_transform(h, U, n, V, n, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK, bb.bb_last_error()
    finally:
        bb.bb_destroy(h)
    # stored column-major: transpose the row-major view
    return (d.cpu().numpy().astype(np.float64), e[: max(n - 1, 0)].cpu().numpy().astype(np.float64),
            U.cpu().numpy().T.astype(np.float64), V.cpu().numpy().T.astype(np.float64))


def dense_b(d, e):
    B = np.diag(d)
    if d.size > 1:
        B += np.diag(e, 1)
    return B


@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("n,bw,tw", [(2, 1, 1), (5, 3, 2), (40, 8, 3), (64, 16, 8), (130, 24, 7), (300, 40, 12),
                                     (257, 64, 32)])
def test_reconstruction_orthogonality_and_first_column(n, bw, tw, dt):
    band = bi.make_band(n, bw, tw, dt, seed=n + bw)
    a = bi.band_to_dense(band, n, bw + tw).astype(np.float64)
    d, e, U, V = gpu_vectors(band, n, bw, tw, dt)
    fro = np.linalg.norm(a)
    tol = TOL[dt]
    assert np.linalg.norm(a - U @ dense_b(d, e) @ V.T) <= tol * fro
    assert np.abs(U.T @ U - np.eye(n)).max() <= tol * 10
    assert np.abs(V.T @ V - np.eye(n)).max() <= tol * 10
    e1 = np.eye(n)[0]
    assert np.array_equal(U[:, 0], e1) and np.array_equal(V[:, 0], e1)


@pytest.mark.parametrize("n,bw,tw", [(64, 16, 8), (200, 32, 8)])
def test_singular_vectors(n, bw, tw):
    band = bi.make_band(n, bw, tw, "f64", seed=3 * n)
    a = bi.band_to_dense(band, n, bw + tw)
    d, e, U, V = gpu_vectors(band, n, bw, tw, "f64")
    ub, s, vbt = np.linalg.svd(dense_b(d, e))
    Us, Vs = U @ ub, V @ vbt.T
    fro = np.linalg.norm(a)
    assert np.abs(a @ Vs - Us * s).max() <= 1e-12 * fro
    # and the singular values are the oracle's
    d0, e0 = oracle.bidiagonal(band, n, bw, tw)
    s0 = oracle.bidiagonal_singular_values(d0, e0)
    assert np.abs(s - s0).max() <= 1e-12 * fro


def test_back_transform_needs_a_recorded_reduction():
    n, bw, tw = 30, 6, 2
    dev = torch.device("cuda:0")
    U = torch.empty((n, n), dtype=torch.float64, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F64)
    try:
        with pytest.raises(bb.BBError):
            bb.bb_back_transform(h, U, n, None, n)
        x = torch.from_numpy(bi.make_band(n, bw, tw, "f64", seed=1)).to(dev)
        d = torch.empty(n, dtype=torch.float64, device=dev)
        e = torch.empty(n - 1, dtype=torch.float64, device=dev)
        bb.bb_reduce(h, x, x.shape[1], tw, d, e)          # not recorded
        with pytest.raises(bb.BBError):
            bb.bb_back_transform(h, U, n, None, n)
        bb.bb_set_param(h, bb.BB_PARAM_RECORD, 1)
        x.copy_(torch.from_numpy(bi.make_band(n, bw, tw, "f64", seed=1)).to(dev))
        bb.bb_reduce(h, x, x.shape[1], tw, d, e)
        with pytest.raises(bb.BBError):
            bb.bb_back_transform(h, U, n - 1, None, n)    # ldu < n
        bb.bb_back_transform(h, U, n, None, n)
        assert bb.bb_status_sync(h, None) == bb.BB_OK
    finally:
        bb.bb_destroy(h)
