"""The oracle's pins catch plausible mistakes planted in the oracle.

Each mutant is a copy of the oracle's C source with one mistake of the kinds
a reimplementation of the method could make (a wrong sign, a dropped term, a
wrong index or window bound, a transposed operand, a wrong pass plan).  It is
compiled into a temporary folder with the oracle's own flags and bound in
place of the real library for the duration of one test.  A compact version of
the pins (LAPACK's dlarfg, exact bidiagonal form, band mode == dense mode,
Frobenius norm, singular values of the input, prescribed singular values)
must pass on the real oracle and fail on every mutant.  All mutations keep
every access inside the arrays the oracle is given, and none can loop
forever.
"""
import ctypes
import os
import shutil

import numpy as np
import pytest
from scipy.linalg import lapack

import band_inputs as bi
import oracle

ORACLE_DIR = os.path.dirname(oracle.__file__)

# name -> list of (text in bb_oracle_body.h, replacement); every occurrence of
# the text is replaced, and each text must occur
MUTANTS = {
    "beta_sign": [("(a >= 0) ? -HYPOT(a, xnorm) : HYPOT(a, xnorm)",
                   "(a >= 0) ? HYPOT(a, xnorm) : -HYPOT(a, xnorm)")],
    "sign_of_zero": [("(a >= 0) ?", "(a > 0) ?")],
    "tau_numerator": [("*tau = (beta - a) / beta;", "*tau = (a - beta) / beta;")],
    "v_scale_sign": [("REAL scal = 1 / (a - beta);", "REAL scal = 1 / (beta - a);")],
    "norm_not_squared": [("ssq = ssq + v * v;", "ssq = ssq + FABS(v);")],
    "right_apply_drops_first_term": [
        ("for (int64_t q = 0; q < w; ++q) y = y + ELEM(i, c + q) * v[q];",
         "for (int64_t q = 1; q < w; ++q) y = y + ELEM(i, c + q) * v[q];")],
    "left_apply_drops_tau": [
        ("ELEM(c + q, j) = ELEM(c + q, j) - s * v[q];", "ELEM(c + q, j) = ELEM(c + q, j) - y * v[q];")],
    "window_one_short": [("int64_t ce = (c + t < n - 1) ? c + t : n - 1;",
                          "int64_t ce = (c + t - 1 < n - 1) ? c + t - 1 : n - 1;")],
    "left_columns_one_short": [("int64_t cend = (ce + b < n - 1) ? ce + b : n - 1;",
                                "int64_t cend = (ce + b - 1 < n - 1) ? ce + b - 1 : n - 1;")],
    "bulge_row_off_by_one": [("int64_t p = (k == 0) ? r : c - b;", "int64_t p = (k == 0) ? r : c - b + 1;")],
    "right_apply_skips_last_row": [("for (int64_t i = (ROW_LO); i <= (ROW_HI); ++i)",
                                    "for (int64_t i = (ROW_LO); i < (ROW_HI); ++i)")],
    "left_reflector_from_row": [("for (int64_t q = 0; q < w; ++q) v[q] = ELEM(c + q, c);",
                                 "for (int64_t q = 0; q < w; ++q) v[q] = ELEM(c, c + q);")],
    "sweep_one_step_short": [("int64_t last = n - 2 - r - (b - t);", "int64_t last = n - 3 - r - (b - t);")],
    "last_sweep_skipped": [("for (int64_t r = 0; r + (b - t) + 1 <= n - 1; ++r)",
                            "for (int64_t r = 0; r + (b - t) + 1 <= n - 2; ++r)")],
    "plan_stops_at_two": [("while (b > 1) {", "while (b > 2) {")],
    "superdiagonal_from_subdiagonal": [("e[i] = ELEM(i, i + 1);", "e[i] = ELEM(i + 1, i);")],
}

DENSE_CASES = [(24, 6, 2), (33, 10, 4), (40, 8, 7), (17, 16, 15)]


def _rel(x, y):
    return float(np.abs(np.asarray(x, np.float64) - np.asarray(y, np.float64)).max())


@np.errstate(all="ignore")  # mutants overflow
def compact_pins():
    """Names of the compact pins that fail for the oracle library now bound."""
    failed = []
    # 1. LAPACK's dlarfg on random vectors and on alpha = +0, -0, < 0; for
    #    alpha = -0 the reading sign(-0) = + makes the expected result LAPACK's
    #    at alpha = +0
    rng = np.random.default_rng(3)
    cases = [(float(rng.normal()), rng.normal(size=m)) for m in (1, 3, 8)]
    cases += [(0.0, np.array([3.0, 4.0])), (-0.0, np.array([3.0, 4.0])), (-2.0, np.array([1.0, 2.0])),
              (1e6, np.array([1e-3]))]
    for alpha, x in cases:
        beta, v, tau = oracle.larfg(alpha, x.copy())
        b_ref, v_ref, t_ref = lapack.dlarfg(x.size + 1, abs(alpha) if alpha == 0 else alpha, x.copy())
        scale = max(abs(b_ref), 1e-300)
        if not (abs(beta - b_ref) <= 1e-14 * scale and abs(tau - t_ref) <= 1e-14
                and _rel(v, v_ref) <= 1e-13 * max(1.0, float(np.abs(v_ref).max()))):
            failed.append("larfg")
            break
    # 2-4. exact form, band == dense, orthogonal invariance
    for n, bw, tw in DENSE_CASES:
        band = bi.make_band(n, bw, tw, "f64", "normal", seed=n + bw)
        a = bi.band_to_dense(band, n, bw + tw)
        s_in = np.linalg.svd(a, compute_uv=False)
        dense = a.copy()
        oracle.reduce_dense(dense, bw, tw)
        off = dense.copy()
        i = np.arange(n)
        off[i, i] = 0
        off[i[:-1], i[:-1] + 1] = 0
        if np.count_nonzero(off) or not np.isfinite(dense).all():
            failed.append(f"dense bidiagonal {n, bw, tw}")
        d, e = oracle.bidiagonal(band, n, bw, tw)
        if not (np.array_equal(d, np.diag(dense)) and np.array_equal(e, np.diag(dense, 1))):
            failed.append(f"band == dense {n, bw, tw}")
        fro = np.linalg.norm(a)
        if not abs(np.sqrt(d @ d + e @ e) - fro) <= 1e-13 * fro:
            failed.append(f"frobenius {n, bw, tw}")
        s = oracle.bidiagonal_singular_values(d, e) if np.isfinite(d).all() and np.isfinite(e).all() else None
        if s is None or not _rel(s, s_in) <= 1e-12 * s_in[0]:
            failed.append(f"singular values {n, bw, tw}")
    # 5. prescribed singular values
    n, bw, tw = 120, 12, 5
    sigma = bi.spectrum("quarter_circle", n, seed=2)
    band = bi.make_band_with_spectrum(n, bw, tw, sigma, seed=8)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    ok = np.isfinite(d).all() and np.isfinite(e).all()
    if not ok or not _rel(oracle.bidiagonal_singular_values(d, e), sigma) <= 1e-12:
        failed.append("prescribed singular values")
    return failed


@pytest.fixture
def bound_library(monkeypatch):
    """Bind a given oracle library in place of the real one for one test."""
    def use(path):
        monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(path)))
    return use


def build_mutant(tmp_path, edits):
    for f in os.listdir(ORACLE_DIR):
        if f.endswith((".c", ".h")) and f != "bb_oracle_body.h":
            shutil.copy(os.path.join(ORACLE_DIR, f), tmp_path / f)
    with open(os.path.join(ORACLE_DIR, "bb_oracle_body.h")) as f:
        body = f.read()
    for old, new in edits:
        assert old in body, f"mutation site not found: {old}"
        body = body.replace(old, new)
    (tmp_path / "bb_oracle_body.h").write_text(body)
    return oracle.compile_library(str(tmp_path / "bb_oracle.c"), str(tmp_path / "mutant.so"))


def test_real_oracle_passes_compact_pins():
    assert compact_pins() == []


def test_unmodified_copy_passes_compact_pins(tmp_path, bound_library):
    # the build-and-bind route itself changes nothing
    bound_library(build_mutant(tmp_path, []))
    assert compact_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, bound_library):
    bound_library(build_mutant(tmp_path, MUTANTS[name]))
    assert compact_pins(), f"mutant {name} passes every pin"
