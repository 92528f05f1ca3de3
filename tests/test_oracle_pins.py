"""Pins of the CPU oracle against what the mathematics fixes (no GPU).

The oracle (oracle/bb_oracle.c) is checked here against facts that do not
come from the oracle itself:
  * LAPACK's slarfg/dlarfg (the reflector convention read for the paper's
    tile-QR reference, Section III, Algorithm 2 text);
  * the definition of the transforms: the dense mode applies every reflector
    to whole rows/columns, and the band mode must agree with it bitwise;
  * the target form: every entry off the diagonal and superdiagonal is exactly
    zero after the last pass (successive band reduction down to bandwidth 1);
  * orthogonal invariance: Frobenius norm and singular values of the input
    (a brute-force one-sided Jacobi SVD written here) are preserved;
  * uniqueness of |d|, |e|: a textbook Golub-Kahan Householder
    bidiagonalisation of the dense matrix gives the same |d|, |e|;
  * special cases with known answers, power-of-two scaling, and the paper's
    claim that the concurrent schedule reproduces the serial one exactly.
"""
import itertools
import random

import numpy as np
import pytest
import scipy.linalg as sla
from scipy.linalg import lapack

import band_inputs as bi
import oracle

F64_EPS = np.finfo(np.float64).eps
F32_EPS = np.finfo(np.float32).eps


def dense_of(band, n, bw, tw):
    return bi.band_to_dense(band, n, bw + tw)


def sigma_bidiagonal(d, e):
    """Singular values of upper bidiagonal (d, e) via the Golub-Kahan tridiagonal."""
    n = d.size
    if n == 1:
        return np.abs(d.astype(np.float64))
    off = np.empty(2 * n - 1)
    off[0::2] = d
    off[1::2] = e
    ev = sla.eigvalsh_tridiagonal(np.zeros(2 * n), off)
    return np.sort(ev)[::-1][:n]


def jacobi_svd_values(a, tol=1e-15, max_sweeps=60):
    """One-sided (Hestenes) Jacobi: rotate column pairs until mutually orthogonal."""
    u = np.array(a, dtype=np.float64, copy=True)
    n = u.shape[1]
    for _ in range(max_sweeps):
        off = 0.0
        for i in range(n - 1):
            for j in range(i + 1, n):
                al = u[:, i] @ u[:, i]
                be = u[:, j] @ u[:, j]
                ga = u[:, i] @ u[:, j]
                if ga == 0.0 or abs(ga) <= tol * np.sqrt(al * be):
                    continue
                off = max(off, abs(ga) / np.sqrt(al * be))
                zeta = (be - al) / (2.0 * ga)
                t = np.sign(zeta) / (abs(zeta) + np.sqrt(1.0 + zeta * zeta)) if zeta != 0 else 1.0
                c = 1.0 / np.sqrt(1.0 + t * t)
                s = c * t
                ui = u[:, i].copy()
                u[:, i] = c * ui - s * u[:, j]
                u[:, j] = s * ui + c * u[:, j]
        if off <= tol:
            break
    return np.sort(np.linalg.norm(u, axis=0))[::-1]


def golub_kahan_dense(a):
    """Textbook Householder bidiagonalisation: left reflector on column i
    (rows i..), then right reflector on row i (columns i+1..).  Returns d, e."""
    a = np.array(a, dtype=np.float64, copy=True)
    n = a.shape[0]

    def house(x):
        v = x.copy()
        nx = np.linalg.norm(x)
        if nx == 0:
            return v, 0.0
        v[0] += np.copysign(nx, x[0]) if x[0] != 0 else nx
        return v, 2.0 / (v @ v)

    for i in range(n):
        v, beta = house(a[i:, i])
        a[i:, i:] -= beta * np.outer(v, v @ a[i:, i:])
        if i < n - 2:
            v, beta = house(a[i, i + 1:])
            a[i:, i + 1:] -= beta * np.outer(a[i:, i + 1:] @ v, v)
    return np.diag(a).copy(), np.diag(a, 1).copy()


SMALL_CASES = [
    # (n, bw, tw)
    (2, 1, 1), (3, 2, 1), (5, 3, 2), (8, 4, 3), (16, 8, 7), (24, 6, 2), (24, 6, 4),
    (32, 8, 3), (33, 10, 4), (40, 8, 7), (48, 12, 5), (64, 16, 8), (64, 16, 15), (50, 20, 9),
    (60, 9, 8), (70, 17, 16), (30, 29, 7), (45, 40, 13),
]


# ----------------------------------------------------------------- larfg ---

@pytest.mark.parametrize("dt,ref,eps", [(np.float64, lapack.dlarfg, F64_EPS),
                                        (np.float32, lapack.slarfg, F32_EPS)])
def test_larfg_matches_lapack(dt, ref, eps):
    rng = np.random.default_rng(7)
    cases = []
    for m in range(1, 40):
        for scale in (1.0, 1e-3, 1e3):
            cases.append((dt(rng.standard_normal() * scale), (rng.standard_normal(m) * scale).astype(dt)))
    cases += [
        (dt(0.0), rng.standard_normal(5).astype(dt)),          # alpha = +0: beta = -||x||
        (dt(-2.5), rng.standard_normal(7).astype(dt)),         # alpha < 0: beta > 0
        (dt(3.0), np.zeros(6, dt)),                            # x = 0: identity
        (dt(-3.0), np.zeros(6, dt)),
        (dt(1e-30 if dt == np.float64 else 1e-20), np.full(4, 1e-30 if dt == np.float64 else 1e-20, dt)),
    ]
    if dt == np.float64:
        cases.append((dt(1e-300), np.full(3, 2e-300)))  # beta < safmin: LAPACK's rescaling branch
        cases.append((dt(3e200), np.full(5, 1e200)))    # sum of squares overflows
        cases.append((dt(1e-170), np.full(5, 1e-170)))  # sum of squares underflows
    else:
        cases.append((dt(1e-36), np.full(3, 2e-36, dt)))
        cases.append((dt(3e25), np.full(5, 1e25, dt)))
        cases.append((dt(1e-24), np.full(5, 1e-24, dt)))
    for alpha, x in cases:
        beta, v, tau = oracle.larfg(alpha, x)
        rb, rv, rt = ref(x.size + 1, alpha, x.copy())
        assert beta.dtype == dt and tau.dtype == dt
        assert np.isfinite(beta) and np.isfinite(tau)
        if not np.any(x):
            assert tau == 0 and beta == alpha and np.all(v == 0)
            assert rt == 0
            continue
        assert np.sign(beta) == np.sign(rb) and np.sign(beta) == (-1.0 if alpha >= 0 else 1.0)
        assert abs(beta - rb) <= 6 * eps * abs(rb), (alpha, x, beta, rb)
        assert abs(tau - rt) <= 6 * eps * max(1.0, abs(rt)), (tau, rt)
        assert np.all(np.abs(v - rv) <= 8 * eps * np.maximum(1.0, np.abs(rv))), (v, rv)
        # and the reflector does what it says: H (alpha, x) = (beta, 0)
        u = np.concatenate([[1.0], v.astype(np.float64)])
        y = np.concatenate([[alpha], x]).astype(np.float64)
        hy = y - tau * u * (u @ y)
        scale = np.abs(y).max()
        assert np.all(np.abs(hy[1:]) <= 50 * eps * scale * np.sqrt(y.size))
        assert abs(hy[0] - beta) <= 50 * eps * scale * np.sqrt(y.size)


def test_larfg_single_entry_is_identity():
    beta, v, tau = oracle.larfg(-1.5, np.zeros(0))
    assert beta == -1.5 and tau == 0 and v.size == 0


def test_larfg_negative_zero_alpha_reads_as_positive():
    # sign(+-0) = + (the reading taken; LAPACK's SIGN would follow the sign bit)
    x = np.array([3.0, 4.0])
    beta, v, tau = oracle.larfg(-0.0, x)
    assert beta == -5.0 and tau == 1.0


# ------------------------------------------------------- form and identity ---

@pytest.mark.parametrize("n,bw,tw", SMALL_CASES)
@pytest.mark.parametrize("dt", ["f64", "f32"])
def test_dense_result_exactly_bidiagonal_and_band_equals_dense(n, bw, tw, dt):
    band = bi.make_band(n, bw, tw, dt, "normal", seed=n * 131 + bw)
    a = dense_of(band, n, bw, tw)
    oracle.reduce_dense(a, bw, tw)
    off = a.copy()
    idx = np.arange(n)
    off[idx, idx] = 0
    off[idx[:-1], idx[:-1] + 1] = 0
    assert np.count_nonzero(off) == 0
    work = band.copy()
    oracle.reduce_band(work, n, bw, tw)
    d, e = oracle.extract(work, n, bw + tw)
    assert np.array_equal(d, np.diag(a)) and np.array_equal(e, np.diag(a, 1))
    # every stored entry off the bidiagonal is exactly zero in band mode too
    back = dense_of(work, n, bw, tw)
    back[idx, idx] = 0
    back[idx[:-1], idx[:-1] + 1] = 0
    assert np.count_nonzero(back) == 0


@pytest.mark.parametrize("n,bw,tw", SMALL_CASES)
def test_frobenius_and_singular_values_preserved(n, bw, tw):
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=7 * n + tw)
    a = dense_of(band, n, bw, tw)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    fro = np.linalg.norm(a)
    assert abs(np.sqrt(d @ d + e @ e) - fro) <= 1e-13 * fro
    if n <= 48:
        s_ref = jacobi_svd_values(a)
        # the brute-force SVD is itself checked against LAPACK
        assert np.abs(s_ref - np.linalg.svd(a, compute_uv=False)).max() <= 1e-13 * s_ref[0]
        s = sigma_bidiagonal(d, e)
        assert np.abs(s - s_ref).max() <= 1e-12 * s_ref[0]
        assert np.linalg.norm(s - s_ref) <= 1e-12 * np.linalg.norm(s_ref)


@pytest.mark.parametrize("n,bw,tw", [(8, 4, 3), (16, 8, 3), (24, 6, 2), (32, 8, 7), (40, 10, 4),
                                     (48, 12, 11), (64, 16, 8)])
def test_abs_de_match_textbook_golub_kahan(n, bw, tw):
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=3 * n + bw)
    a = dense_of(band, n, bw, tw)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    d2, e2 = golub_kahan_dense(a)
    fro = np.linalg.norm(a)
    assert np.abs(np.abs(d) - np.abs(d2)).max() <= 1e-10 * fro
    assert np.abs(np.abs(e) - np.abs(e2)).max() <= 1e-10 * fro


def test_float32_oracle_close_to_float64():
    n, bw, tw = 64, 16, 8
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=11)
    d64, e64 = oracle.bidiagonal(band, n, bw, tw)
    d32, e32 = oracle.bidiagonal(band.astype(np.float32), n, bw, tw)
    fro = np.linalg.norm(band)
    assert np.abs(np.abs(d32) - np.abs(d64)).max() <= 1e-5 * fro
    assert np.abs(np.abs(e32) - np.abs(e64)).max() <= 1e-5 * fro


# ------------------------------------------------------------ special cases ---

@pytest.mark.parametrize("bw", [0, 1])
def test_bandwidth_at_most_one_is_unchanged(bw):
    n, tw = 20, 1
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=5)
    a = dense_of(band, n, bw, tw)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    assert np.array_equal(d, np.diag(a)) and np.array_equal(e, np.diag(a, 1))


def test_diagonal_input_takes_identity_reflectors():
    n, bw, tw = 30, 8, 3
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=9)
    diag = band[:, bw + tw].copy()
    band[:, :] = 0
    band[:, bw + tw] = diag
    d, e = oracle.bidiagonal(band, n, bw, tw)
    assert np.array_equal(d, diag) and np.count_nonzero(e) == 0


def test_zero_columns_and_zero_matrix():
    n, bw, tw = 32, 8, 3
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=4)
    ku = bw + tw
    for j in (0, 5, 6, 17, 31):  # zero whole columns of A
        band[j, :] = 0
    a = dense_of(band, n, bw, tw)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    s_ref = np.linalg.svd(a, compute_uv=False)
    assert np.abs(sigma_bidiagonal(d, e) - s_ref).max() <= 1e-12 * s_ref[0]
    z = np.zeros_like(band)
    d, e = oracle.bidiagonal(z, n, bw, tw)
    assert np.count_nonzero(d) == 0 and np.count_nonzero(e) == 0
    del ku


@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("k", [-7, 3, 20])
def test_power_of_two_scaling_commutes_bitwise(dt, k):
    n, bw, tw = 48, 12, 5
    band = bi.make_band(n, bw, tw, dt, "normal", seed=12)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    s = band.dtype.type(2.0 ** k)
    d2, e2 = oracle.bidiagonal(band * s, n, bw, tw)
    assert np.array_equal(d2, d * s) and np.array_equal(e2, e * s)


@pytest.mark.parametrize("n,bw,tw", [(1, 0, 1), (2, 1, 1), (3, 2, 1), (4, 3, 1), (3, 2, 2)])
def test_tiny_orders(n, bw, tw):
    if tw > max(1, bw - 1):
        with pytest.raises(ValueError):
            oracle.reduce_band(bi.make_band(n, bw, tw, "f64", seed=1), n, bw, tw)
        return
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=1)
    a = dense_of(band, n, bw, tw)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    s_ref = np.linalg.svd(a, compute_uv=False)
    assert np.abs(sigma_bidiagonal(d, e) - s_ref).max() <= 1e-14 * max(s_ref[0], 1)


def test_invalid_arguments_rejected():
    band = bi.make_band(10, 4, 2, "f64", seed=1)
    with pytest.raises(ValueError):
        oracle.reduce_band(band[:, :6].copy(), 10, 4, 2)   # ldab too small
    with pytest.raises(ValueError):
        oracle.reduce_band(band, 10, 4, 4)                   # tw > bw - 1
    with pytest.raises(ValueError):
        oracle.reduce_band(bi.make_band(4, 3, 1, "f64"), 4, 4, 1)  # bw >= n


# ---------------------------------------------- prescribed singular values ---
#
# The paper's accuracy protocol (Section V): a band built from A = U diag(sigma)
# V^T in float64 must reduce to a bidiagonal whose singular values are sigma.
# Unlike the Jacobi pin above, the expected values here are the prescribed
# ones, not computed from the input.  The pages report no numbers, only
# float64 errors "near machine epsilon"; the bars are the acceptance bars of
# the parity tests (max |dsigma| <= 1e-12 sigma_1 in float64, 2e-5 sigma_1 in
# float32), and the paper's measure ||dsigma||_2 / ||sigma||_2 is held to
# 1e-13 (float64) and 1e-5 (float32).

KNOWN_SIGMA_CASES = [(200, 16, 8), (384, 24, 7), (300, 40, 12), (512, 32, 8)]
KNOWN_SIGMA_BARS = {"f64": (1e-12, 1e-13), "f32": (2e-5, 1e-5)}


@pytest.mark.parametrize("kind", bi.SPECTRA + ("rank_deficient",))
def test_known_spectrum_generator(kind):
    # the generator itself, against LAPACK's SVD of the dense band it returns
    n, bw, tw = 160, 12, 5
    sigma = bi.spectrum(kind, n, seed=4)
    assert np.all(np.diff(sigma) <= 0) and sigma[0] <= 1.0 and sigma[-1] >= 0.0
    band = bi.make_band_with_spectrum(n, bw, tw, sigma, seed=9)
    a = dense_of(band, n, bw, tw)
    i, j = np.indices(a.shape)
    assert not a[(j < i) | (j - i > bw)].any()
    assert np.abs(np.linalg.svd(a, compute_uv=False) - sigma).max() <= 50 * F64_EPS


def test_spectrum_profiles():
    n = 11
    assert np.array_equal(bi.spectrum("arithmetic", n), np.arange(n, 0, -1) / n)
    lg = bi.spectrum("logarithmic", n)
    assert lg[0] == 1.0 and abs(lg[-1] - 1e-8) <= 1e-22
    assert np.allclose(lg[1:] / lg[:-1], 10 ** -0.8, rtol=1e-14)
    rd = bi.spectrum("rank_deficient", n)
    assert np.count_nonzero(rd) == n - n // 2
    # quarter-circle law: mean 4 / (3 pi), second moment 1 / 4
    qc = bi.spectrum("quarter_circle", 200000, seed=1)
    assert abs(qc.mean() - 4 / (3 * np.pi)) < 3e-3 and abs((qc * qc).mean() - 0.25) < 3e-3


@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("kind", bi.SPECTRA + ("rank_deficient",))
@pytest.mark.parametrize("n,bw,tw", KNOWN_SIGMA_CASES)
def test_oracle_recovers_prescribed_singular_values(n, bw, tw, kind, dt):
    sigma = bi.spectrum(kind, n, seed=n + bw)
    band = bi.make_band_with_spectrum(n, bw, tw, sigma, dt, seed=3 * n + tw)
    d, e = oracle.bidiagonal(band, n, bw, tw)
    got = oracle.bidiagonal_singular_values(d.astype(np.float64), e.astype(np.float64))
    max_bar, norm_bar = KNOWN_SIGMA_BARS[dt]
    assert np.abs(got - sigma).max() <= max_bar * sigma[0]
    assert np.linalg.norm(got - sigma) <= norm_bar * np.linalg.norm(sigma)


def test_pass_plan_of_the_workloads():
    assert oracle.pass_plan(8, 7) == [(8, 7)]
    assert oracle.pass_plan(16, 8) == [(16, 8), (8, 7)]
    assert oracle.pass_plan(64, 16) == [(64, 16), (48, 16), (32, 16), (16, 15)]
    assert oracle.pass_plan(128, 32) == [(128, 32), (96, 32), (64, 32), (32, 31)]
    assert oracle.pass_plan(256, 32) == [(b, 32) for b in range(256, 32, -32)] + [(32, 31)]


def test_pass_split_equals_whole():
    n, bw, tw = 64, 24, 5
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=2)
    whole = band.copy()
    oracle.reduce_band(whole, n, bw, tw)
    split = band.copy()
    oracle.reduce_band(split, n, bw, tw, 0, 2)
    oracle.reduce_band(split, n, bw, tw, 2, 100)
    assert np.array_equal(whole, split)


# --------------------------------------------------------------- schedules ---

def _lag_cycle(b, t):
    return 2 if b > t + 1 else 3


def _lag_half(b, t):
    return 2 if b - t >= 3 else (3 if b - t == 2 else 4)


def _run_order(band, n, bw, tw, order_fn):
    work = band.copy()
    ku = bw + tw
    for q in range(tw):
        work[:, q] = 0
    for q in range(ku + 1, ku + tw + 1):
        work[:, q] = 0
    for (b, t) in oracle.pass_plan(bw, tw):
        for (r, k, side) in order_fn(n, b, t):
            oracle.halfstep_band(work, n, b, t, ku, r, k, side)
    return work


def cycle_order(n, b, t):
    """Per-cycle schedule: in cycle T every active sweep r runs step T - lag r.
    Within a cycle the steps are taken in DESCENDING r, the reverse of the
    serial order, so any overlap between them would change the result."""
    lag = _lag_cycle(b, t)
    S = [r for r in range(n) if oracle.sweep_steps(n, b, t, r) > 0]
    K = {r: oracle.sweep_steps(n, b, t, r) for r in S}
    tmax = max(lag * r + K[r] - 1 for r in S) if S else -1
    for T in range(tmax + 1):
        for r in sorted(S, reverse=True):
            k = T - lag * r
            if 0 <= k < K[r]:
                yield (r, k, 0)
                yield (r, k, 1)


def halfstep_protocol_order(seed):
    """A random interleaving allowed by the persistent scheduler's rule: half-
    step h of sweep r may start once sweep r-1 has completed
    min(h + lagh, H_{r-1}) half-steps, and a sweep completes its last
    half-step only after its predecessor has completed all of its own."""
    def gen(n, b, t):
        rng = random.Random(seed * 1000 + n * 7 + b)
        L = _lag_half(b, t)
        S = [r for r in range(n) if oracle.sweep_steps(n, b, t, r) > 0]
        H = {r: 2 * oracle.sweep_steps(n, b, t, r) for r in S}
        done = {r: 0 for r in S}
        while True:
            ready = []
            for r in S:
                h = done[r]
                if h >= H[r]:
                    continue
                if r > 0:
                    need = min(h + L, H[r - 1])
                    if h == H[r] - 1:
                        need = H[r - 1]
                    if done[r - 1] < need:
                        continue
                ready.append(r)
            if not ready:
                break
            # prefer later sweeps, the order most likely to expose a race
            r = max(ready) if rng.random() < 0.7 else rng.choice(ready)
            h = done[r]
            yield (r, h // 2, h % 2)
            done[r] += 1
        assert all(done[r] == H[r] for r in S)
    return gen


@pytest.mark.parametrize("n,bw,tw", [(40, 8, 3), (40, 8, 7), (48, 6, 4), (48, 6, 5), (60, 16, 14),
                                     (33, 5, 2), (64, 16, 8), (50, 3, 2), (50, 3, 1), (70, 24, 7)])
def test_cycle_schedule_reproduces_serial_bitwise(n, bw, tw):
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=n + bw + tw)
    serial = band.copy()
    oracle.reduce_band(serial, n, bw, tw)
    alt = _run_order(band, n, bw, tw, cycle_order)
    assert np.array_equal(alt, serial)


@pytest.mark.parametrize("n,bw,tw", [(40, 8, 3), (40, 8, 7), (48, 6, 4), (48, 6, 5), (60, 16, 14),
                                     (33, 5, 2), (64, 16, 8), (50, 3, 2), (50, 3, 1), (70, 24, 7)])
@pytest.mark.parametrize("seed", [0, 1])
def test_halfstep_protocol_reproduces_serial_bitwise(n, bw, tw, seed):
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=n * 3 + seed)
    serial = band.copy()
    oracle.reduce_band(serial, n, bw, tw)
    alt = _run_order(band, n, bw, tw, halfstep_protocol_order(seed))
    assert np.array_equal(alt, serial)


PIPELINE_CASES = [(40, 8, 3), (40, 8, 7), (48, 6, 4), (48, 6, 5), (60, 16, 14), (33, 5, 2), (64, 16, 8),
                  (50, 3, 2), (50, 3, 1), (70, 24, 7), (2, 1, 1), (3, 2, 1), (5, 3, 2), (300, 40, 12)]


@pytest.mark.parametrize("n,bw,tw", PIPELINE_CASES)
@pytest.mark.parametrize("dt", ["f64", "f32"])
def test_pipelined_threads_reproduce_serial_bitwise(n, bw, tw, dt):
    # the multi-threaded chase (sweep r on thread r mod P, spinning on the
    # predecessor's half-step count) runs the half-step rule concurrently
    band = bi.make_band(n, bw, tw, dt, "normal", seed=n + bw + 5)
    serial = band.copy()
    oracle.reduce_band(serial, n, bw, tw)
    for threads in (1, 2, 3, 8, 16):
        work = band.copy()
        oracle.reduce_band_pipelined(work, n, bw, tw, threads)
        assert np.array_equal(work, serial), threads


@pytest.mark.parametrize("n,bw,tw", [(1000, 32, 8), (600, 9, 8), (800, 12, 10), (512, 64, 16)])
def test_pipelined_threads_larger_bands(n, bw, tw):
    # enough sweeps in flight for real overlap between threads; repeated
    band = bi.make_band(n, bw, tw, "f32", "uniform", seed=n)
    serial = band.copy()
    oracle.reduce_band(serial, n, bw, tw)
    for _ in range(3):
        work = band.copy()
        oracle.reduce_band_pipelined(work, n, bw, tw, 8)
        assert np.array_equal(work, serial)


@pytest.mark.parametrize("dt", ["f32", "f64"])
def test_pipelined_pass_range_equals_serial_pass_range(dt):
    # the multi-threaded chase over a pass range (the CPU baseline times the
    # first pass of the largest workloads this way) is the serial range
    n, bw, tw = 700, 64, 16
    band = bi.make_band(n, bw, tw, dt, "normal", seed=9)
    serial, work = band.copy(), band.copy()
    for lo, hi in ((0, 1), (1, 3), (3, 4)):
        oracle.reduce_band(serial, n, bw, tw, lo, hi)
        oracle.reduce_band_pipelined(work, n, bw, tw, 5, pass_lo=lo, pass_hi=hi)
        assert np.array_equal(work, serial), (lo, hi)
    whole = band.copy()
    oracle.reduce_band(whole, n, bw, tw)
    assert np.array_equal(work, whole)


def test_pipelined_invalid_arguments():
    band = bi.make_band(20, 4, 2, "f64", seed=1)
    for threads, limit in ((0, 10.0), (2000, 10.0), (2, 0.0), (2, -1.0)):
        with pytest.raises(ValueError):
            oracle.reduce_band_pipelined(band.copy(), 20, 4, 2, threads, limit)
    with pytest.raises(ValueError):
        oracle.reduce_band_pipelined(band.copy(), 20, 4, 4, 2)   # tw > bw - 1


def test_a_too_short_lag_is_detected():
    # Sanity of the schedule tests above: running the last pass with a
    # one-cycle lag (steps of consecutive sweeps in the same cycle, taken in
    # reverse order) must change the result.
    n, bw, tw = 40, 8, 7
    band = bi.make_band(n, bw, tw, "f64", "normal", seed=1)
    serial = band.copy()
    oracle.reduce_band(serial, n, bw, tw)

    def bad(n, b, t):
        S = [r for r in range(n) if oracle.sweep_steps(n, b, t, r) > 0]
        K = {r: oracle.sweep_steps(n, b, t, r) for r in S}
        for T in range(max(r + K[r] for r in S)):
            for r in sorted(S, reverse=True):
                k = T - r
                if 0 <= k < K[r]:
                    yield (r, k, 0)
                    yield (r, k, 1)

    alt = _run_order(band, n, bw, tw, bad)
    assert not np.array_equal(alt, serial)


# ---------------------------------------------------------------------------
# Bidiagonal singular values (oracle of bb_singular_values)
# ---------------------------------------------------------------------------

def _dense_bidiag(d, e):
    n = d.size
    B = np.diag(d.astype(np.float64))
    if n > 1:
        B += np.diag(e.astype(np.float64), 1)
    return B


def test_svals_one_by_one():
    assert oracle.bidiagonal_singular_values(np.array([-2.5]), np.zeros(0))[0] == 2.5


def test_svals_two_by_two_closed_form():
    # B = [[a, b], [0, c]]: s1 s2 = |a c|, s1^2 + s2^2 = a^2 + b^2 + c^2
    rng = np.random.default_rng(5)
    for _ in range(20):
        a, b, c = rng.normal(size=3)
        S = a * a + b * b + c * c
        disc = np.sqrt(S * S - 4 * (a * c) ** 2)
        want = np.sqrt(np.array([(S + disc) / 2, max((S - disc) / 2, 0.0)]))
        got = oracle.bidiagonal_singular_values(np.array([a, c]), np.array([b]))
        assert np.allclose(got, want, rtol=1e-12, atol=1e-14)


def test_svals_diagonal_is_sorted_abs():
    d = np.array([0.5, -3.0, 2.0, 0.0, -1.0])
    got = oracle.bidiagonal_singular_values(d, np.zeros(4))
    assert np.array_equal(got, np.array([3.0, 2.0, 1.0, 0.5, 0.0]))


def test_svals_all_ones_path_graph():
    # all d = e = 1: the Golub-Kahan matrix is the path graph on 2n nodes,
    # eigenvalues 2 cos(k pi / (2n + 1)); the positive half are the sigma
    n = 37
    got = oracle.bidiagonal_singular_values(np.ones(n), np.ones(n - 1))
    want = 2 * np.cos(np.arange(1, n + 1) * np.pi / (2 * n + 1))
    assert np.allclose(got, want, rtol=0, atol=1e-13)


def test_svals_match_dense_svd_and_scale():
    rng = np.random.default_rng(6)
    d = rng.normal(size=60)
    e = rng.normal(size=59)
    got = oracle.bidiagonal_singular_values(d, e)
    want = np.linalg.svd(_dense_bidiag(d, e), compute_uv=False)
    assert np.allclose(got, want, rtol=0, atol=1e-13 * want[0])
    got3 = oracle.bidiagonal_singular_values(-3 * d, 3 * e)
    assert np.allclose(got3, 3 * got, rtol=0, atol=1e-13 * got3[0])
    assert np.all(np.diff(got) <= 0)


def test_svals_power_of_two_scaling_exact():
    # sigma(2^k B) = 2^k sigma(B) exactly (the oracle scales internally), from
    # near underflow to near overflow
    rng = np.random.default_rng(7)
    d = rng.normal(size=40)
    e = rng.normal(size=39)
    base = oracle.bidiagonal_singular_values(d, e)
    for k in (-1000, -500, -60, 60, 500, 1000):
        got = oracle.bidiagonal_singular_values(np.ldexp(d, k), np.ldexp(e, k))
        assert np.array_equal(got, np.ldexp(base, k)), k
