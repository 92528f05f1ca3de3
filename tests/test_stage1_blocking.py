"""The blocked (compact WY) schedule of the GPU's stage 1, replayed in numpy
and checked against the oracle's reflector-by-reflector stage 1.

The GPU (bb_dense_to_band) takes a panel's QR reflectors, then its LQ
reflectors, in blocks of at most 16 (fewer where a block must fit shared
memory).  Per block it factorizes the block's columns, forms the upper
triangular T of H_0 H_1 ... = I - V T V^T (LAPACK xLARFT, forward,
columnwise), and updates the rest of the matrix with matrix products:
A -= V T^T (V^T A) after a QR block, A -= (A U) T U^T after an LQ block.
This replay follows the same block boundaries (including the narrowed
widths) and the same T recurrence, so a mistake in the schedule (a block
range, the rows an LQ block updates, T's recurrence) shows up as a
difference from oracle.dense_to_band far above rounding.  No GPU needed.
"""
import numpy as np
import pytest

import oracle


def larfg(alpha, x):
    ss = float(np.dot(x, x))
    if ss == 0.0:
        return alpha, np.zeros_like(x), 0.0
    nrm = np.sqrt(alpha * alpha + ss)
    beta = -nrm if alpha >= 0 else nrm
    return beta, x / (alpha - beta), (beta - alpha) / beta


def panel(P, nq):
    """Factorize the first nq columns of the view P in place; returns V, T."""
    m = P.shape[0]
    V = np.zeros((m, nq))
    T = np.zeros((nq, nq))
    for j in range(nq):
        beta, vt, tau = larfg(P[j, j], P[j + 1:, j].copy())
        v = np.zeros(m)
        v[j] = 1.0
        v[j + 1:] = vt
        V[:, j] = v
        P[j, j] = beta
        P[j + 1:, j] = 0
        if tau != 0:
            P[j:, j + 1:] -= tau * np.outer(v[j:], v[j:] @ P[j:, j + 1:])
        T[:j, j] = -tau * (T[:j, :j] @ (V[:, :j].T @ v))
        T[j, j] = tau
    return V, T


def blocked_stage1(a, bw, block=16, cap=None):
    """The GPU's schedule: blocks of `block` reflectors, narrowed to
    cap // m where a panel of m rows would not fit (cap None: never)."""
    a = a.copy()
    n = a.shape[0]
    bw = min(bw, n)
    width = lambda m: block if cap is None or cap // m < 1 else min(block, cap // m)
    for k in range(0, n, bw):
        kb = min(k + bw, n)
        qend = min(kb, n - 1)  # QR reflectors j < n - 1
        cs = k
        while cs < qend:
            nbs = width(n - cs)
            nq, nc = min(nbs, qend - cs), min(nbs, kb - cs)
            V, T = panel(a[cs:, cs:cs + nc], nq)
            if cs + nc < n:
                At = a[cs:, cs + nc:]
                At -= V @ (T.T @ (V.T @ At))
            cs += nbs
        lend = min(kb, n - 1 - bw)  # LQ reflectors i with i + bw + 1 < n
        rs = k
        while rs < lend:
            nbs = width(n - rs - bw)
            nl = min(nbs, lend - rs)
            U, T = panel(a[rs:rs + nl, rs + bw:].T, nl)  # the rows' transposed view
            if rs + nl < n:
                At = a[rs + nl:, rs + bw:]
                At -= ((At @ U) @ T) @ U.T
            rs += nbs
    return a


CASES = [(1, 1), (2, 1), (5, 2), (9, 8), (40, 1), (64, 16), (100, 7), (130, 40), (200, 32), (257, 64),
         (300, 299), (97, 200), (77, 17)]


@pytest.mark.parametrize("n,bw", CASES)
@pytest.mark.parametrize("block,cap", [(16, None), (5, None), (16, 800), (16, 3000)])
def test_blocked_schedule_equals_the_oracle(n, bw, block, cap):
    rng = np.random.default_rng(7 * n + bw)
    a = rng.standard_normal((n, n))
    ref = oracle.dense_to_band(a, bw)
    got = blocked_stage1(a, bw, block, cap)
    assert np.abs(got - ref).max() <= 1e-13 * max(np.linalg.norm(a), 1e-300)


def test_a_wrong_lq_update_range_is_caught():
    # the replay must be sensitive: updating the LQ block's own rows again
    # (rows rs.. instead of rs+nl..) breaks the agreement
    n, bw = 120, 16
    a = np.random.default_rng(3).standard_normal((n, n))
    ref = oracle.dense_to_band(a, bw)
    b = a.copy()
    for k in range(0, n, bw):
        kb = min(k + bw, n)
        qend = min(kb, n - 1)
        for cs in range(k, qend, 16):
            nq, nc = min(16, qend - cs), min(16, kb - cs)
            V, T = panel(b[cs:, cs:cs + nc], nq)
            if cs + nc < n:
                At = b[cs:, cs + nc:]
                At -= V @ (T.T @ (V.T @ At))
        lend = min(kb, n - 1 - bw)
        for rs in range(k, lend, 16):
            nl = min(16, lend - rs)
            U, T = panel(b[rs:rs + nl, rs + bw:].T, nl)
            At = b[rs:, rs + bw:]  # wrong: includes the block's own rows
            At -= ((At @ U) @ T) @ U.T
    assert np.abs(b - ref).max() > 1e-6 * np.linalg.norm(a)
