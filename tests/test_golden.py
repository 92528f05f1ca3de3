"""Oracle regression fixtures (tests/golden/, written by
tests/golden/make_golden.py from oracle/ alone).

The pages print no worked example, so these are not pins of the oracle:
they freeze its outputs so that any change to its arithmetic is seen here
and has to be made on purpose (regenerate the fixtures and name the passage
that justifies the change).  d and e come from the C oracle's IEEE
operations in a fixed order and are compared bit for bit; the singular
values come from LAPACK (through scipy), whose last bits may differ between
builds, and are compared to a few ulps of the largest.
"""
import os
import sys

import numpy as np
import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)

import make_golden  # noqa: E402


def load(name):
    out = {}
    with open(os.path.join(HERE, name + ".txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            out[key] = np.array([float.fromhex(v) for v in vals])
    return out


@pytest.mark.parametrize("case", make_golden.CASES, ids=[c[0] for c in make_golden.CASES])
def test_oracle_matches_its_fixture(case):
    name, kind, n, bw, tw, dt, dist, seed = case
    want = load(name)
    d, e, sigma = make_golden.compute(kind, n, bw, tw, dt, dist, seed)
    assert np.array_equal(d.astype(np.float64), want["d"])
    assert np.array_equal(e.astype(np.float64), want["e"])
    if sigma is not None:
        assert np.abs(sigma - want["sigma"]).max() <= 8 * np.finfo(np.float64).eps * want["sigma"][0]
