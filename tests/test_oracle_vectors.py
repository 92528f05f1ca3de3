"""Pins of the oracle's back-transformation (singular vectors, no GPU).

The reduction applies left reflectors L_i and right reflectors R_i, so the
input is A = U B V^T with U = L_1 L_2 ..., V = R_1 R_2 ... and B bidiagonal.
What fixes U and V, independently of the oracle:
  * B is the plain reduction's result, bitwise (same arithmetic);
  * A = U B V^T and U, V are orthogonal (definition of the transforms);
  * no reflector touches row or column 0, so U e_1 = V e_1 = e_1 exactly;
  * with B = U_b S V_b^T (LAPACK's SVD of the small bidiagonal), the columns
    of U U_b and V V_b are singular vectors of A: A (V V_b) = (U U_b) S;
  * special cases: a band that is already bidiagonal and a diagonal input
    give U = V = I;
  * planted mistakes in the recording (a side swapped, tau or a v entry
    lost) break these.
"""
import ctypes
import os
import shutil

import numpy as np
import pytest

import band_inputs as bi
import oracle

CASES = [(2, 1, 1), (5, 3, 2), (24, 6, 2), (40, 8, 7), (48, 12, 5), (64, 16, 8), (70, 24, 7), (200, 32, 8)]


def dense_b(d, e):
    B = np.diag(d.astype(np.float64))
    if d.size > 1:
        B += np.diag(e.astype(np.float64), 1)
    return B


@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("n,bw,tw", CASES)
def test_vectors_reconstruct_and_are_orthogonal(n, bw, tw, dt):
    band = bi.make_band(n, bw, tw, dt, seed=n + bw)
    a = bi.band_to_dense(band, n, bw + tw).astype(np.float64)
    d, e, U, V = oracle.bidiagonal_with_vectors(band, n, bw, tw)
    d0, e0 = oracle.bidiagonal(band, n, bw, tw)
    assert np.array_equal(d, d0) and np.array_equal(e, e0)
    bar = 1e-13 if dt == "f64" else 1e-5
    fro = np.linalg.norm(a)
    assert np.linalg.norm(a - U @ dense_b(d, e) @ V.T) <= bar * fro
    assert np.abs(U.T @ U - np.eye(n)).max() <= bar
    assert np.abs(V.T @ V - np.eye(n)).max() <= bar
    e1 = np.eye(n)[0]
    assert np.array_equal(U[:, 0], e1) and np.array_equal(U[0], e1)
    assert np.array_equal(V[:, 0], e1) and np.array_equal(V[0], e1)


@pytest.mark.parametrize("n,bw,tw", [(40, 8, 3), (64, 16, 8), (120, 12, 5)])
def test_singular_vectors_of_a(n, bw, tw):
    band = bi.make_band(n, bw, tw, "f64", seed=3 * n)
    a = bi.band_to_dense(band, n, bw + tw)
    d, e, U, V = oracle.bidiagonal_with_vectors(band, n, bw, tw)
    ub, s, vbt = np.linalg.svd(dense_b(d, e))
    Us, Vs = U @ ub, V @ vbt.T
    fro = np.linalg.norm(a)
    assert np.abs(a @ Vs - Us * s).max() <= 1e-12 * fro
    assert np.abs(a.T @ Us - Vs * s).max() <= 1e-12 * fro


def test_prescribed_spectrum_vectors():
    # A = U0 diag(sigma) V0^T reduced to band form: the back-transformed
    # singular vectors of the band carry the prescribed singular values
    n, bw, tw = 150, 12, 5
    sigma = bi.spectrum("arithmetic", n)
    band = bi.make_band_with_spectrum(n, bw, tw, sigma, seed=7)
    a = bi.band_to_dense(band, n, bw + tw)
    d, e, U, V = oracle.bidiagonal_with_vectors(band, n, bw, tw)
    ub, s, vbt = np.linalg.svd(dense_b(d, e))
    Us, Vs = U @ ub, V @ vbt.T
    assert np.abs(s - sigma).max() <= 1e-12
    assert np.abs(np.linalg.norm(a @ Vs, axis=0) - sigma).max() <= 1e-12


def test_identity_transforms_for_bidiagonal_and_diagonal_inputs():
    n = 30
    band = bi.make_band(n, 1, 1, "f64", seed=2)
    _, _, U, V = oracle.bidiagonal_with_vectors(band, n, 1, 1)
    assert np.array_equal(U, np.eye(n)) and np.array_equal(V, np.eye(n))
    bw, tw = 8, 3
    band = np.zeros((n, bw + 2 * tw + 1))
    band[:, bw + tw] = np.arange(1.0, n + 1)
    d, e, U, V = oracle.bidiagonal_with_vectors(band, n, bw, tw)
    assert np.array_equal(U, np.eye(n)) and np.array_equal(V, np.eye(n))
    assert np.array_equal(d, np.arange(1.0, n + 1)) and not e.any()


def test_reflector_count_and_widths():
    n, bw, tw = 64, 16, 8
    band = bi.make_band(n, bw, tw, "f64", seed=1)
    side, start, width, taus, vs = oracle.reduce_band_record(band.copy(), n, bw, tw)
    assert side.size == oracle.reflector_count(n, bw, tw)
    assert np.all(side[0::2] == 0) and np.all(side[1::2] == 1)      # right, then left, per step
    assert np.all((width >= 2) & (width <= tw + 1)) and np.all(start >= 1)
    assert np.all(vs[:, 0] == 1.0)


# ----------------------------------------------------------- planted mistakes

MUTANTS = {
    "right_recorded_as_left": [("RECORD(0, c, w, v, tau);", "RECORD(1, c, w, v, tau);")],
    "tau_not_recorded": [("taus[nrec] = (TAU);", "taus[nrec] = 0;")],
    "last_v_entry_lost": [("for (int64_t u_ = 0; u_ < (W); ++u_)", "for (int64_t u_ = 0; u_ < (W) - 1; ++u_)")],
}


@pytest.fixture
def bound_library(monkeypatch):
    def use(path):
        monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(path)))
    return use


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_recording_mutant_is_caught(name, tmp_path, bound_library):
    here = os.path.dirname(oracle.__file__)
    for f in os.listdir(here):
        if f.endswith((".c", ".h")) and f != "bb_oracle_body.h":
            shutil.copy(os.path.join(here, f), tmp_path / f)
    body = open(os.path.join(here, "bb_oracle_body.h")).read()
    for old, new in MUTANTS[name]:
        assert old in body, old
        body = body.replace(old, new)
    (tmp_path / "bb_oracle_body.h").write_text(body)
    bound_library(oracle.compile_library(str(tmp_path / "bb_oracle.c"), str(tmp_path / "mutant.so")))
    n, bw, tw = 40, 8, 3
    band = bi.make_band(n, bw, tw, "f64", seed=5)
    a = bi.band_to_dense(band, n, bw + tw)
    d, e, U, V = oracle.bidiagonal_with_vectors(band, n, bw, tw)
    ok = (np.linalg.norm(a - U @ dense_b(d, e) @ V.T) <= 1e-13 * np.linalg.norm(a)
          and np.abs(U.T @ U - np.eye(n)).max() <= 1e-13 and np.abs(V.T @ V - np.eye(n)).max() <= 1e-13)
    assert not ok, f"mutant {name} passes"


def test_reflectors_of_one_sweep_are_disjoint_and_commute():
    # what a blocked back-transformation relies on: within one sweep the right
    # (left) reflectors act on disjoint column (row) ranges, so any order of
    # applying them gives the same U, V bit for bit; consecutive sweeps
    # overlap, so the order of the sweeps does matter
    n, bw, tw = 60, 12, 5
    band = bi.make_band(n, bw, tw, "f64", seed=8)
    side, start, width, taus, vs = oracle.reduce_band_record(band.copy(), n, bw, tw)
    # reflectors in order: pass -> sweep -> step -> (right, left)
    groups = []
    q = 0
    for (b, t) in oracle.pass_plan(bw, tw):
        for r in range(n):
            K = oracle.sweep_steps(n, b, t, r)
            if K:
                groups.append(list(range(q, q + 2 * K)))
                q += 2 * K
    assert q == side.size

    def apply(order):
        U, V = np.eye(n), np.eye(n)
        for i in order:
            c, w, tau = int(start[i]), int(width[i]), float(taus[i])
            if tau == 0.0:
                continue
            v = vs[i, :w]
            M = U if side[i] == 1 else V
            y = M[:, c:c + w] @ v
            M[:, c:c + w] -= tau * np.outer(y, v)
        return U, V

    U0, V0 = apply(range(q))
    rng = np.random.default_rng(0)
    for g in groups:
        for s_ in (0, 1):
            idx = [i for i in g if side[i] == s_]
            spans = sorted((int(start[i]), int(start[i]) + int(width[i]) - 1) for i in idx)
            assert all(a[1] < b_[0] for a, b_ in zip(spans, spans[1:]))   # disjoint
    shuffled = []
    for g in groups:
        g = list(g)
        rng.shuffle(g)
        shuffled += g
    U1, V1 = apply(shuffled)
    assert np.array_equal(U0, U1) and np.array_equal(V0, V1)
    # consecutive sweeps overlap: reversing the sweep order changes the result
    U2, V2 = apply([i for g in reversed(groups) for i in g])
    assert not (np.array_equal(U0, U2) and np.array_equal(V0, V2))
