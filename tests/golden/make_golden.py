"""Writes the oracle regression fixtures in this folder (calls only oracle/
and the seeded input generators).

The pages print no worked numerical example, so no fixture here comes from
them.  These files instead freeze the oracle's own outputs, bit for bit (as
hexadecimal floats), on small seeded inputs, so that any change to the
oracle's arithmetic shows up in tests/test_golden.py and has to be made on
purpose: rerun this script and name, in the commit message, the passage (or
the reading of it) that justifies the change.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import band_inputs as bi  # noqa: E402
import oracle  # noqa: E402

# (name, kind, n, bw, tw, dtype, dist, seed)
CASES = [
    ("bidiagonal_n256_bw8_tw7_f64", "bidiagonal", 256, 8, 7, "f64", "normal", 0),
    ("bidiagonal_n64_bw16_tw8_f32", "bidiagonal", 64, 16, 8, "f32", "uniform", 1),
    ("bidiagonal_n40_bw8_tw3_f64", "bidiagonal", 40, 8, 3, "f64", "normal", 2),
    ("tridiagonal_n48_bw12_tw5_f64", "tridiagonal", 48, 12, 5, "f64", "normal", 3),
]


def hexes(a):
    return " ".join(float(x).hex() for x in np.asarray(a, dtype=np.float64))


def compute(kind, n, bw, tw, dt, dist, seed):
    if kind == "bidiagonal":
        band = bi.make_band(n, bw, tw, dt, dist, seed=seed)
        d, e = oracle.bidiagonal(band, n, bw, tw)
        sigma = oracle.bidiagonal_singular_values(d.astype(np.float64), e.astype(np.float64))
        return d, e, sigma
    sb = bi.make_sym_band(n, bw, tw, dt, dist, seed=seed)
    d, e = oracle.tridiagonal(sb, n, bw, tw)
    return d, e, None


def main():
    for name, kind, n, bw, tw, dt, dist, seed in CASES:
        d, e, sigma = compute(kind, n, bw, tw, dt, dist, seed)
        lines = [f"# oracle {kind} of band_inputs.make_{'band' if kind == 'bidiagonal' else 'sym_band'}"
                 f"(n={n}, bw={bw}, tw={tw}, dtype={dt}, dist={dist}, seed={seed}); written by make_golden.py",
                 f"d {hexes(d)}", f"e {hexes(e)}"]
        if sigma is not None:
            lines.append(f"sigma {hexes(sigma)}")
        with open(os.path.join(HERE, name + ".txt"), "w") as f:
            f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
