"""Pins of the oracle's symmetric variant (symmetric band -> tridiagonal by
the same passes, one two-sided reflector per step; no GPU).

What fixes the result, independently of the oracle:
  * the target form: after the last pass every entry off the three central
    diagonals is exactly zero (dense mode), and the band mode, which applies
    the reflectors only inside their windows, agrees with the dense mode
    bitwise;
  * orthogonal similarity: the Frobenius norm and the eigenvalues of the input
    (LAPACK's symmetric eigensolver) are preserved;
  * uniqueness: no reflector touches row or column 0, so the tridiagonal is
    fixed up to signs by the input (implicit-Q theorem), and |d|, |e| must
    agree with LAPACK's dense Householder tridiagonalisation dsytrd (lower),
    whose transform also leaves row and column 0 alone;
  * prescribed eigenvalues: A = Q diag(lam) Q^T reduced to band form in
    float64 must end with eigenvalues lam;
  * special cases: bandwidth <= 1, diagonal and zero inputs, power-of-two
    scaling, tiny orders, invalid arguments;
  * planted mistakes in copies of the symmetric body fail these pins.
"""
import ctypes
import os
import shutil

import numpy as np
import pytest
import scipy.linalg as sla
from scipy.linalg import lapack

import band_inputs as bi
import oracle

CASES = [(2, 1, 1), (3, 2, 1), (5, 3, 2), (17, 16, 15), (24, 6, 2), (33, 10, 4), (40, 8, 7), (48, 12, 5),
         (60, 9, 8), (64, 16, 8), (70, 24, 7)]


def tri_eigs(d, e):
    d = np.asarray(d, np.float64)
    return d.copy() if d.size == 1 else sla.eigvalsh_tridiagonal(d, np.asarray(e, np.float64))


@pytest.mark.parametrize("n,bw,tw", CASES)
@pytest.mark.parametrize("dt", ["f64", "f32"])
def test_dense_exactly_tridiagonal_and_band_equals_dense(n, bw, tw, dt):
    sb = bi.make_sym_band(n, bw, tw, dt, seed=n + 3 * bw)
    a = bi.sym_band_to_dense(sb, n)
    oracle.sym_reduce_dense(a, bw, tw)
    off = a.copy()
    i = np.arange(n)
    off[i, i] = 0
    off[i[1:], i[:-1]] = 0
    off[i[:-1], i[1:]] = 0
    assert np.count_nonzero(off) == 0
    assert np.array_equal(a, a.T)
    work = sb.copy()
    oracle.sym_reduce_band(work, n, bw, tw)
    d, e = oracle.sym_extract(work, n)
    assert np.array_equal(d, np.diag(a)) and np.array_equal(e, np.diag(a, -1))
    # every stored entry below the subdiagonal is exactly zero
    assert np.count_nonzero(work[:, 2:]) == 0


@pytest.mark.parametrize("n,bw,tw", CASES)
def test_norm_and_eigenvalues_preserved(n, bw, tw):
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=7 * n + tw)
    a = bi.sym_band_to_dense(sb, n)
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    fro = np.linalg.norm(a)
    assert abs(np.sqrt(d @ d + 2 * (e @ e)) - fro) <= 1e-13 * fro
    assert np.abs(np.sort(tri_eigs(d, e)) - np.linalg.eigvalsh(a)).max() <= 1e-12 * fro


@pytest.mark.parametrize("n,bw,tw", [c for c in CASES if c[0] >= 3])
def test_abs_de_match_lapack_dsytrd(n, bw, tw):
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=3 * n + bw)
    a = bi.sym_band_to_dense(sb, n)
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    _, d2, e2, _, info = lapack.dsytrd(a.copy(), lower=1)
    assert info == 0
    fro = np.linalg.norm(a)
    assert np.abs(np.abs(d) - np.abs(d2)).max() <= 1e-10 * fro
    assert np.abs(np.abs(e) - np.abs(e2)).max() <= 1e-10 * fro


def test_float32_close_to_float64():
    n, bw, tw = 64, 16, 8
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=11)
    d64, e64 = oracle.tridiagonal(sb, n, bw, tw)
    d32, e32 = oracle.tridiagonal(sb.astype(np.float32), n, bw, tw)
    fro = np.linalg.norm(bi.sym_band_to_dense(sb, n))
    assert np.abs(np.sort(tri_eigs(d32, e32)) - np.sort(tri_eigs(d64, e64))).max() <= 1e-5 * fro


@pytest.mark.parametrize("kind", bi.SPECTRA + ("rank_deficient",))
@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("n,bw,tw", [(200, 16, 8), (300, 40, 12)])
def test_prescribed_eigenvalues(n, bw, tw, kind, dt):
    # eigenvalues of both signs: the profile with alternate signs
    lam = bi.spectrum(kind, n, seed=n + bw) * np.where(np.arange(n) % 2, -1.0, 1.0)
    sb = bi.make_sym_band_with_spectrum(n, bw, tw, lam, dt, seed=5 * n + tw)
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    got = np.sort(tri_eigs(d, e))
    want = np.sort(lam)
    bar = 1e-12 if dt == "f64" else 2e-5
    assert np.abs(got - want).max() <= bar * np.abs(lam).max()


def test_known_spectrum_generator():
    n, bw, tw = 150, 12, 5
    lam = np.linspace(-1.0, 2.0, n)
    sb = bi.make_sym_band_with_spectrum(n, bw, tw, lam, seed=2)
    a = bi.sym_band_to_dense(sb, n)
    i, j = np.indices(a.shape)
    assert not a[np.abs(i - j) > bw].any()
    assert np.abs(np.linalg.eigvalsh(a) - lam).max() <= 100 * np.finfo(np.float64).eps * 2.0


@pytest.mark.parametrize("bw", [0, 1])
def test_bandwidth_at_most_one_is_unchanged(bw):
    n, tw = 20, 1
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=5)
    a = bi.sym_band_to_dense(sb, n)
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    assert np.array_equal(d, np.diag(a)) and np.array_equal(e, np.diag(a, -1))


def test_diagonal_and_zero_inputs():
    n, bw, tw = 30, 8, 3
    sb = np.zeros((n, bw + tw + 1))
    sb[:, 0] = np.arange(1, n + 1, dtype=np.float64)
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    assert np.array_equal(d, sb[:, 0]) and not e.any()
    d, e = oracle.tridiagonal(np.zeros_like(sb), n, bw, tw)
    assert not d.any() and not e.any()


@pytest.mark.parametrize("dt,k", [("f64", 40), ("f64", -40), ("f32", 20), ("f32", -20)])
def test_power_of_two_scaling_commutes_bitwise(dt, k):
    n, bw, tw = 48, 12, 5
    sb = bi.make_sym_band(n, bw, tw, dt, seed=9)
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    ds, es = oracle.tridiagonal(np.ldexp(sb, k).astype(sb.dtype), n, bw, tw)
    assert np.array_equal(ds, np.ldexp(d, k).astype(d.dtype)) and np.array_equal(es, np.ldexp(e, k).astype(e.dtype))


def test_tiny_orders_and_invalid_arguments():
    d, e = oracle.tridiagonal(np.array([[3.0, 0.0]]), 1, 0, 1)
    assert d[0] == 3.0 and e.size == 0
    sb = bi.make_sym_band(10, 4, 2, "f64", seed=1)
    with pytest.raises(ValueError):
        oracle.sym_reduce_band(sb[:, :6].copy(), 10, 4, 2)   # ldab < bw + tw + 1
    with pytest.raises(ValueError):
        oracle.sym_reduce_band(sb.copy(), 10, 4, 4)           # tw > bw - 1
    with pytest.raises(ValueError):
        oracle.sym_reduce_band(bi.make_sym_band(4, 3, 1, "f64"), 4, 4, 1)  # bw >= n


# ------------------------------------------------------------------ schedule
#
# Lockstep schedule of concurrent sweeps, one step per tick: sweep r runs step
# k at tick k + L r.  With L = 2 when b - t >= 2 and L = 3 when b - t == 1,
# the steps of one tick touch disjoint entries and every pair of overlapping
# steps runs in sweep order (the pages' rule for the one-entry chase: sweep s
# takes step k once sweep s - 1 has finished step k + 2); L - 1 does not
# suffice.  Shown two ways: by the windows, and by running the oracle's own
# steps in that order with each tick's steps in reverse sweep order.


def sym_lag(b, t):
    return 2 if b - t >= 2 else 3


def sym_cells(n, b, t, r, k):
    c = r + (b - t) + k * b
    p = r if k == 0 else c - b
    ce = min(c + t, n - 1)
    cend = min(ce + b, n - 1)
    cells = {(i, j) for i in range(c, ce + 1) for j in range(p, i + 1)}
    cells |= {(i, j) for i in range(ce + 1, cend + 1) for j in range(c, ce + 1)}
    return cells


def sym_lockstep_ok(n, b, t, L):
    K = {r: oracle.sweep_steps(n, b, t, r) for r in range(n)}
    C = {(r, k): sym_cells(n, b, t, r, k) for r in K for k in range(K[r])}
    for (r, k), x in C.items():
        for rp in range(r + 1, min(r + 3 * b + 3, n)):
            for kp in range(K[rp]):
                if x & C[(rp, kp)] and not (k + L * r < kp + L * rp):
                    return False
    return True


@pytest.mark.parametrize("b,t", [(b, t) for b in range(2, 10) for t in range(1, b)])
def test_symmetric_lockstep_lag_valid_and_least(b, t):
    n = 4 * b + 9
    L = sym_lag(b, t)
    assert sym_lockstep_ok(n, b, t, L)
    assert not sym_lockstep_ok(n, b, t, L - 1)


def run_lockstep(sb, n, bw, tw, lag_of):
    work = sb.copy()
    work[:, bw + 1:bw + tw + 1] = 0
    for (b, t) in oracle.pass_plan(bw, tw):
        L = lag_of(b, t)
        K = {r: oracle.sweep_steps(n, b, t, r) for r in range(n)}
        S = [r for r in K if K[r] > 0]
        tmax = max(L * r + K[r] - 1 for r in S) if S else -1
        for T in range(tmax + 1):
            for r in sorted(S, reverse=True):
                k = T - L * r
                if 0 <= k < K[r]:
                    oracle.sym_step_band(work, n, b, t, r, k)
    return work


@pytest.mark.parametrize("n,bw,tw", [(40, 8, 3), (40, 8, 7), (48, 6, 4), (48, 6, 5), (60, 16, 14), (33, 5, 2),
                                     (64, 16, 8), (50, 3, 2), (50, 3, 1), (70, 24, 7)])
def test_symmetric_lockstep_reproduces_serial_bitwise(n, bw, tw):
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=n + bw + tw)
    serial = sb.copy()
    oracle.sym_reduce_band(serial, n, bw, tw)
    assert np.array_equal(run_lockstep(sb, n, bw, tw, sym_lag), serial)


def test_symmetric_short_lag_is_detected():
    n, bw, tw = 40, 8, 3
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=1)
    serial = sb.copy()
    oracle.sym_reduce_band(serial, n, bw, tw)
    assert not np.array_equal(run_lockstep(sb, n, bw, tw, lambda b, t: sym_lag(b, t) - 1), serial)


def async_order_run(sb, n, bw, tw, seed, lag_of):
    """Random interleaving allowed by the progress-flag rule: step k of sweep
    r starts once sweep r-1 has finished min(k + L, K_{r-1}) steps, and the
    last step of a sweep once all of sweep r-1 is done."""
    import random
    work = sb.copy()
    work[:, bw + 1:bw + tw + 1] = 0
    rng = random.Random(seed)
    for (b, t) in oracle.pass_plan(bw, tw):
        L = lag_of(b, t)
        K = {r: oracle.sweep_steps(n, b, t, r) for r in range(n)}
        S = [r for r in K if K[r] > 0]
        done = {r: 0 for r in S}
        while True:
            ready = []
            for r in S:
                k = done[r]
                if k >= K[r]:
                    continue
                if r > 0:
                    need = K[r - 1] if k == K[r] - 1 else min(k + L, K[r - 1])
                    if done[r - 1] < need:
                        continue
                ready.append(r)
            if not ready:
                break
            # prefer later sweeps, the order most likely to expose a race
            r = max(ready) if rng.random() < 0.7 else rng.choice(ready)
            oracle.sym_step_band(work, n, b, t, r, done[r])
            done[r] += 1
        assert all(done[r] == K[r] for r in S)
    return work


ASYNC_CASES = [(40, 8, 3), (40, 8, 7), (48, 6, 4), (48, 6, 5), (60, 16, 14), (33, 5, 2), (64, 16, 8),
               (50, 3, 2), (50, 3, 1), (70, 24, 7), (30, 2, 1), (45, 12, 11)]


@pytest.mark.parametrize("n,bw,tw", ASYNC_CASES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_symmetric_progress_rule_reproduces_serial_bitwise(n, bw, tw, seed):
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=n + bw)
    serial = sb.copy()
    oracle.sym_reduce_band(serial, n, bw, tw)
    assert np.array_equal(async_order_run(sb, n, bw, tw, seed, sym_lag), serial)


def test_symmetric_progress_rule_with_short_lag_fails():
    n, bw, tw = 40, 8, 3
    sb = bi.make_sym_band(n, bw, tw, "f64", seed=n + bw)
    serial = sb.copy()
    oracle.sym_reduce_band(serial, n, bw, tw)
    assert not np.array_equal(async_order_run(sb, n, bw, tw, 0, lambda b, t: sym_lag(b, t) - 1), serial)


@pytest.mark.parametrize("n,bw,tw", ASYNC_CASES + [(2, 1, 1), (3, 2, 1), (700, 32, 8), (600, 9, 8)])
@pytest.mark.parametrize("dt", ["f64", "f32"])
def test_symmetric_pipelined_threads_reproduce_serial_bitwise(n, bw, tw, dt):
    sb = bi.make_sym_band(n, bw, tw, dt, seed=n + tw)
    serial = sb.copy()
    oracle.sym_reduce_band(serial, n, bw, tw)
    for threads in (1, 2, 3, 8):
        work = sb.copy()
        oracle.sym_reduce_band_pipelined(work, n, bw, tw, threads)
        assert np.array_equal(work, serial), threads


# ----------------------------------------------------------- planted mistakes

SYM_MUTANTS = {
    "rank2_without_correction": [("REAL alpha = -((REAL)0.5 * tau) * dot;", "REAL alpha = 0;")],
    "rank2_one_sided": [("GET(c + u, c + q) - v[u] * x[q] - x[u] * v[q]", "GET(c + u, c + q) - v[u] * x[q]")],
    "left_part_skips_first_column": [("SYM_STEP_BODY(p + 1, c - 1, ce + 1, cend)",
                                      "SYM_STEP_BODY(p + 2, c - 1, ce + 1, cend)")],
    "below_part_one_row_short": [("SYM_STEP_BODY(p + 1, c - 1, ce + 1, cend)",
                                  "SYM_STEP_BODY(p + 1, c - 1, ce + 1, cend - 1)")],
    "reflector_from_row": [("for (int64_t q = 0; q < w; ++q) v[q] = GET(c + q, p);",
                            "for (int64_t q = 0; q < w; ++q) v[q] = GET(c + q, p + 1);")],
    "subdiagonal_from_diagonal": [("e[i] = GET(i + 1, i);", "e[i] = GET(i, i);")],
}


def sym_compact_pins():
    failed = []
    with np.errstate(all="ignore"):
        for n, bw, tw in [(24, 6, 2), (40, 8, 7), (33, 10, 4)]:
            sb = bi.make_sym_band(n, bw, tw, "f64", seed=n + 3 * bw)
            a = bi.sym_band_to_dense(sb, n)
            dn = a.copy()
            oracle.sym_reduce_dense(dn, bw, tw)
            d, e = oracle.tridiagonal(sb, n, bw, tw)
            if not (np.array_equal(d, np.diag(dn)) and np.array_equal(e, np.diag(dn, -1))):
                failed.append("band == dense")
            fro = np.linalg.norm(a)
            if not abs(np.sqrt(d @ d + 2 * (e @ e)) - fro) <= 1e-13 * fro:
                failed.append("frobenius")
            ok = np.isfinite(d).all() and np.isfinite(e).all()
            if not ok or not np.abs(np.sort(tri_eigs(d, e)) - np.linalg.eigvalsh(a)).max() <= 1e-12 * fro:
                failed.append("eigenvalues")
    return failed


@pytest.fixture
def bound_library(monkeypatch):
    def use(path):
        monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(path)))
    return use


def build_sym_mutant(tmp_path, edits):
    here = os.path.dirname(oracle.__file__)
    for f in os.listdir(here):
        if f.endswith((".c", ".h")) and f != "sb_oracle_body.h":
            shutil.copy(os.path.join(here, f), tmp_path / f)
    with open(os.path.join(here, "sb_oracle_body.h")) as f:
        body = f.read()
    for old, new in edits:
        assert old in body, f"mutation site not found: {old}"
        body = body.replace(old, new)
    (tmp_path / "sb_oracle_body.h").write_text(body)
    return oracle.compile_library(str(tmp_path / "bb_oracle.c"), str(tmp_path / "mutant.so"))


def test_real_symmetric_oracle_passes_compact_pins():
    assert sym_compact_pins() == []


@pytest.mark.parametrize("name", sorted(SYM_MUTANTS))
def test_symmetric_mutant_is_caught(name, tmp_path, bound_library):
    bound_library(build_sym_mutant(tmp_path, SYM_MUTANTS[name]))
    assert sym_compact_pins(), f"mutant {name} passes every pin"
