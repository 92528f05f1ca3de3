"""Pins of the oracle's stage 1 (dense -> upper band by block Householder;
no GPU).

What fixes the result, independently of the oracle:
  * the form: every entry outside the upper band is exactly zero;
  * LAPACK: the same panel QR / LQ sequence done with LAPACK's geqrf and
    ormqr (band_inputs.dense_to_upper_band, used to build the accuracy
    protocol's inputs) uses the same reflector convention, so the band agrees
    entry by entry, signs included, up to rounding;
  * bandwidth n - 1 is plain QR: the result is LAPACK's R;
  * orthogonal invariance: singular values and Frobenius norm are kept, and
    a matrix built with prescribed singular values keeps them;
  * the two-stage chain: stage 1 to bandwidth 1, or stage 1 to a wider band
    followed by the band -> bidiagonal oracle, leave column 0 alone on the
    right (V e_1 = e_1), so both give the same |d|, |e| (Golub-Kahan-Lanczos
    uniqueness), and the chain's singular values are those of A.
"""
import numpy as np
import pytest

import band_inputs as bi
import oracle

CASES = [(2, 1), (5, 2), (33, 1), (50, 8), (64, 63), (97, 16), (120, 12), (130, 40)]


def sigma_bidiagonal(d, e):
    return oracle.bidiagonal_singular_values(np.asarray(d, np.float64), np.asarray(e, np.float64))


@pytest.mark.parametrize("n,bw", CASES)
def test_band_form_and_lapack_agreement(n, bw):
    a = np.random.default_rng(n + bw).standard_normal((n, n))
    b = oracle.dense_to_band(a, bw)
    i, j = np.indices(a.shape)
    assert not b[(j < i) | (j - i > bw)].any()
    fro = np.linalg.norm(a)
    assert np.abs(b - bi.dense_to_upper_band(a, bw)).max() <= 1e-13 * fro
    assert abs(np.linalg.norm(b) - fro) <= 1e-13 * fro
    sa = np.linalg.svd(a, compute_uv=False)
    assert np.abs(np.linalg.svd(b, compute_uv=False) - sa).max() <= 1e-13 * sa[0]


def test_bandwidth_n_minus_1_is_lapack_qr():
    n = 40
    a = np.random.default_rng(4).standard_normal((n, n))
    r = np.linalg.qr(a, mode="r")
    assert np.abs(oracle.dense_to_band(a, n - 1) - r).max() <= 1e-13 * np.linalg.norm(a)


@pytest.mark.parametrize("kind", bi.SPECTRA)
def test_prescribed_singular_values_kept(kind):
    n, bw = 120, 10
    sigma = bi.spectrum(kind, n, seed=3)
    rng = np.random.default_rng(5)
    q1, _ = np.linalg.qr(rng.standard_normal((n, n)))
    q2, _ = np.linalg.qr(rng.standard_normal((n, n)))
    b = oracle.dense_to_band((q1 * sigma) @ q2.T, bw)
    assert np.abs(np.linalg.svd(b, compute_uv=False) - sigma).max() <= 1e-13


def test_float32_close_to_float64():
    n, bw = 80, 8
    a = np.random.default_rng(6).standard_normal((n, n))
    b64 = oracle.dense_to_band(a, bw)
    b32 = oracle.dense_to_band(a.astype(np.float32), bw)
    assert b32.dtype == np.float32
    assert np.abs(b32 - b64).max() <= 1e-5 * np.linalg.norm(a)


@pytest.mark.parametrize("n,bw,tw", [(40, 8, 3), (64, 16, 8), (90, 12, 5)])
def test_two_stage_chain(n, bw, tw):
    a = np.random.default_rng(7 * n).standard_normal((n, n))
    fro = np.linalg.norm(a)
    # stage 1 to bandwidth bw, then the band -> bidiagonal oracle
    b = oracle.dense_to_band(a, bw)
    band = bi.dense_to_band(b, bw + tw, bw + 2 * tw + 1)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    # stage 1 straight to bandwidth 1
    b1 = oracle.dense_to_band(a, 1)
    d1, e1 = np.diag(b1), np.diag(b1, 1)
    assert np.abs(np.abs(d) - np.abs(d1)).max() <= 1e-10 * fro
    assert np.abs(np.abs(e) - np.abs(e1)).max() <= 1e-10 * fro
    sa = np.linalg.svd(a, compute_uv=False)
    assert np.abs(sigma_bidiagonal(d, e) - sa).max() <= 1e-12 * sa[0]


def test_invalid_bandwidth():
    with pytest.raises(ValueError):
        oracle.dense_to_band(np.eye(4), 0)
