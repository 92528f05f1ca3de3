"""The group kernel's schedule and buffer protocol, checked on the host.

1. Lockstep: sweep jj of a group runs half-step tau - L*jj at tick tau, with
   L = 2 (b - t >= 3), 3 (b - t == 2) or 4 (b - t == 1).  At every tick the
   half-steps touch disjoint windows, and any two overlapping half-steps of
   different sweeps run in sweep order, so a tick needs one barrier and the
   result is the serial one.  L is also the least lag that works when b - t
   is 1 or at least 3.
2. Buffer protocol: random interleavings of the loader, the compute warps and
   the storer, as the kernel runs them, with the buffer size the library's
   planner gives (bb_group_plan): every column a tick touches is in its slot,
   no slot is refilled before its column was written back and while a later
   tick still touches it, nothing deadlocks, and the group writes back every
   column it loaded.
"""
import random

import pytest

import banded_svd_stage_gb300 as bb


def lag(b, t):
    return 2 if b - t >= 3 else (3 if b - t == 2 else 4)


def steps(n, b, t, r):
    last = n - 2 - r - (b - t)
    return 0 if last < 0 else last // b + 1


def window(n, b, t, r, h):
    """(rows, cols) ranges of half-step h (right: 2k, left: 2k+1) of sweep r."""
    k = h >> 1
    c = r + (b - t) + k * b
    p = r if k == 0 else c - b
    ce = min(c + t, n - 1)
    cend = min(ce + b, n - 1)
    return ((p, ce), (c, ce)) if (h & 1) == 0 else ((c, ce), (c, cend))


def overlap(x, y):
    (r0, r1), (c0, c1) = x
    (s0, s1), (d0, d1) = y
    return not (r1 < s0 or s1 < r0 or c1 < d0 or d1 < c0)


def lockstep_ok(n, b, t, L):
    sweeps = [r for r in range(n) if steps(n, b, t, r) > 0]
    H = {r: 2 * steps(n, b, t, r) for r in sweeps}
    W = {(r, h): window(n, b, t, r, h) for r in sweeps for h in range(H[r])}
    for (r, h), x in W.items():
        for rp in range(r + 1, min(r + 3 * b + 3, n)):
            if rp not in H:
                continue
            for hp in range(H[rp]):
                if overlap(x, W[(rp, hp)]) and not (h + L * r < hp + L * rp):
                    return False
    return True


CASES = [(b, t) for b in range(2, 12) for t in range(1, b)]


@pytest.mark.parametrize("b,t", CASES)
def test_lockstep_lag_is_valid(b, t):
    for n in (3 * b + 7, 5 * b + 3):
        assert lockstep_ok(n, b, t, lag(b, t)), (n, b, t)


@pytest.mark.parametrize("b,t", [(b, t) for (b, t) in CASES if b - t != 2])
def test_lockstep_lag_is_least(b, t):
    n = 5 * b + 3
    assert not lockstep_ok(n, b, t, lag(b, t) - 1), (n, b, t)


def sym_lag(b, t):
    return 2 if b - t >= 2 else 3


def sym_cols(n, b, t, r, k):
    """Column range p .. ce of step k of sweep r of the symmetric chase."""
    c = r + (b - t) + k * b
    p = r if k == 0 else c - b
    return p, min(c + t, n - 1)


def sym_entries(n, b, t, r, k):
    """Entries (i, j), i >= j, that step k of sweep r of the symmetric chase
    reads or writes: column p and columns p+1..c-1 on rows c..ce, the lower
    triangle of the block c..ce, rows ce+1..cend of columns c..ce."""
    c = r + (b - t) + k * b
    p = r if k == 0 else c - b
    ce = min(c + t, n - 1)
    cend = min(ce + b, n - 1)
    out = {(i, j) for j in range(p, c) for i in range(c, ce + 1)}
    out |= {(i, j) for j in range(c, ce + 1) for i in range(j, cend + 1)}
    return out


def sym_lockstep_ok(n, b, t, L):
    sweeps = [r for r in range(n) if steps(n, b, t, r) > 0]
    E = {(r, k): sym_entries(n, b, t, r, k) for r in sweeps for k in range(steps(n, b, t, r))}
    for (r, k), x in E.items():
        for rp in range(r + 1, min(r + 3 * b + 3, n)):
            for kp in range(steps(n, b, t, rp)):
                if (x & E[(rp, kp)]) and not (k + L * r < kp + L * rp):
                    return False
    return True


@pytest.mark.parametrize("b,t", CASES)
def test_sym_lockstep_lag_is_valid(b, t):
    """The symmetric group kernel's lockstep (sweep jj runs step tau - L jj
    at tick tau) keeps every entry's steps in sweep order."""
    for n in (3 * b + 7, 5 * b + 3):
        assert sym_lockstep_ok(n, b, t, sym_lag(b, t)), (n, b, t)


@pytest.mark.parametrize("b,t", CASES)
def test_sym_lockstep_lag_is_least(b, t):
    n = 5 * b + 3
    assert not sym_lockstep_ok(n, b, t, sym_lag(b, t) - 1), (n, b, t)


def simulate(n, bw, tw, elem, pass_index, r0, seed, sym=False):
    """One group (sweeps r0 .. r0+g-1) under random interleavings of the
    loader, compute and storer; returns None or a description of the fault.
    sym: the symmetric chase (one step per tick, bb_sym_group_plan)."""
    plan_of = bb.bb_sym_group_plan if sym else bb.bb_group_plan
    g, nslot, ahead, _ = plan_of(n, bw, tw, elem, pass_index, 0)
    if g == 0:
        return "no plan"
    b = bw
    plan = []
    while b > 1:
        t = min(tw, b - 1)
        plan.append((b, t))
        b -= t
    b, t = plan[pass_index]
    bp, L = b - t, (sym_lag(b, t) if sym else lag(b, t))
    U = 1 if sym else 2  # units per step
    nsw = n - bp - 1
    ng = min(g, nsw - r0)
    if ng <= 0:
        return None
    ns = [steps(n, b, t, r0 + jj) for jj in range(ng)]
    tend = max(L * jj + U * ns[jj] for jj in range(ng))

    def unit_cols(r, h):
        if sym:
            return sym_cols(n, b, t, r, h)
        (_, _), (c0, c1) = window(n, b, t, r, h)
        return c0, c1

    def cols(u):
        out = set()
        for jj in range(ng):
            h = u - L * jj
            if 0 <= h < U * ns[jj]:
                c0, c1 = unit_cols(r0 + jj, h)
                out.update(range(c0, c1 + 1))
        return out

    def tmax(u):
        return max(cols(u), default=-1)

    def tmin(u):
        a = n
        for jj in range(ng):
            h = u - L * jj
            if h < U * ns[jj]:
                a = min(a, unit_cols(r0 + jj, max(h, 0))[0])
        return a

    live_until = {}
    for u in range(tend):
        for c in cols(u):
            live_until[c] = u
    rng = random.Random(seed)
    slots, stored = {}, set()
    done, lu, sv = -1, 0, 0
    B = A = unit_cols(r0, 0)[0]  # the group's first column
    B -= 1
    freed, retired, xr = A, -1, -1
    while done < tend - 1 or lu < tend or sv < tend:
        acts = []
        if done + 1 < tend and lu > done + 1:
            acts.append("c")
        if lu < tend and (lu - ahead - 1 < 0 or retired >= lu - ahead - 1):
            xn = tmax(lu)
            if xn <= B or freed >= xn - nslot + 1:
                acts.append("l")
        if sv < tend and done >= sv:
            acts.append("s")
        if not acts:
            return f"deadlock done={done} loader={lu} storer={sv}"
        a = rng.choice(acts)
        if a == "c":
            tau = done + 1
            for c in cols(tau):
                if slots.get(c % nslot) != c:
                    return f"column {c} missing at tick {tau}"
            done = tau
        elif a == "l":
            xn = tmax(lu)
            for c in range(B + 1, xn + 1):
                old = slots.get(c % nslot)
                if old is not None and (old not in stored or live_until.get(old, -1) > done):
                    return f"slot of column {old} refilled with {c} too early"
                slots[c % nslot] = c
            B = max(B, xn)
            lu += 1
        else:
            xr = max(xr, tmax(sv))
            an = n if sv == tend - 1 else tmin(sv + 1)
            an = min(an, xr + 1)
            for c in range(A, an):
                if slots.get(c % nslot) != c:
                    return f"column {c} written back but not buffered"
                if live_until.get(c, -1) > sv:
                    return f"column {c} written back while tick {live_until[c]} touches it"
                stored.add(c)
            A = max(A, an)
            freed, retired = A, sv
            sv += 1
    # every column copied in was written back (the symmetric chase never
    # touches the last columns of the matrix in some groups; the kernel then
    # publishes n once its storer is done)
    return None if A == B + 1 else f"ended with A = {A}, last column copied in {B}"


@pytest.mark.parametrize("n,bw,tw,elem", [(200, 16, 8, 4), (150, 9, 8, 8), (300, 24, 7, 4), (160, 12, 5, 8),
                                          (257, 8, 7, 8), (400, 40, 12, 8), (200, 16, 8, 2), (300, 24, 7, 2)])
def test_buffer_protocol_random_interleavings(n, bw, tw, elem):
    npass = bb.bb_num_passes(bw, tw)
    checked = 0
    for pi in range(npass):
        g, _, _, _ = bb.bb_group_plan(n, bw, tw, elem, pi, 0)
        if g == 0:
            continue
        for r0 in (0, g, 3 * g, max(0, n - (bw - tw) - 1 - g)):
            for seed in range(3):
                fault = simulate(n, bw, tw, elem, pi, r0, seed)
                assert fault is None, (pi, r0, seed, fault)
                checked += 1
    assert checked > 0


@pytest.mark.parametrize("n,bw,tw,elem", [(200, 16, 8, 4), (150, 9, 8, 8), (300, 24, 7, 4), (160, 12, 5, 8),
                                          (257, 8, 7, 4), (400, 40, 12, 8), (300, 32, 16, 8)])
def test_sym_buffer_protocol_random_interleavings(n, bw, tw, elem):
    npass = bb.bb_num_passes(bw, tw)
    checked = 0
    for pi in range(npass):
        g, _, _, _ = bb.bb_sym_group_plan(n, bw, tw, elem, pi, 0)
        if g == 0:
            continue
        for r0 in (0, g, 3 * g, max(0, n - (bw - tw) - 1 - g)):
            for seed in range(3):
                fault = simulate(n, bw, tw, elem, pi, r0, seed, sym=True)
                assert fault is None, (pi, r0, seed, fault)
                checked += 1
    assert checked > 0


def test_sym_group_plan():
    # the symmetric chase's plans on the main workload's shape: 13 sweeps per
    # group on both passes (float), rows 0 .. b + t of each column buffered
    for p, lds in ((0, 28), (1, 16)):
        g, nslot, ahead, got_lds = bb.bb_sym_group_plan(4096, 16, 8, 4, p)
        assert g == 13 and got_lds == lds and nslot > 16 + 8 and ahead >= 3
    # reflectors longer than 33 elements stay on the flag kernel
    assert bb.bb_sym_group_plan(4096, 128, 64, 4, 0)[0] == 0
    with pytest.raises(bb.BBError):
        bb.bb_sym_group_plan(100, 16, 8, 4, 9)


def test_group_plan_matches_workloads():
    # the plans the automatic scheduler uses on the benchmark workloads
    assert [bb.bb_group_plan(4096, 16, 8, 4, p)[0] for p in range(2)] == [13, 13]
    assert [bb.bb_group_plan(8192, 64, 16, 4, p)[0] for p in range(4)] == [7, 12, 13, 13]
    assert [bb.bb_group_plan(32768, 256, 32, 4, p)[0] for p in range(8)] == [0, 0, 0, 0, 0, 2, 5, 5]
    with pytest.raises(bb.BBError):
        bb.bb_group_plan(100, 16, 8, 4, 9)


def sym_tiles(n, b, t, r, k):
    """Entries the shared-memory flag kernel of the symmetric chase copies
    for step k of sweep r: the left tile (columns p .. c-1 on rows c .. ce)
    and the right tile (columns c .. ce on rows c .. cend, lower triangle)."""
    c = r + (b - t) + k * b
    p = r if k == 0 else c - b
    ce = min(c + t, n - 1)
    cend = min(ce + b, n - 1)
    left = {(c + m, j) for j in range(p, c) for m in range(ce - c + 1)}
    right = {(c + i, c + q) for q in range(ce - c + 1) for i in range(q, cend - c + 1)}
    assert not (left & right)
    return left | right


@pytest.mark.parametrize("b,t", [(2, 1), (8, 7), (16, 8), (24, 7), (40, 12), (64, 16)])
def test_sym_window_tiles_cover_exactly_the_step(b, t):
    """What the symmetric flag kernel reads into shared memory and writes
    back is exactly the step's window: every entry the step reads or writes,
    and no other (so the write-back of unchanged entries touches nothing
    another sweep may be changing)."""
    for n in (3 * b + 7, 6 * b + 5):
        for r in range(n - (b - t) - 1):
            for k in range(steps(n, b, t, r)):
                assert sym_tiles(n, b, t, r, k) == sym_entries(n, b, t, r, k), (n, r, k)
