"""Writes the full-size oracle results of the two largest workloads (calls
only oracle/ and the seeded input generators).

    python tests/golden/make_full_size.py [n16384|n32768 ...]

The two workloads are too large for the serial oracle to run inside a test
(minutes of scalar work each), so their results are computed once here, with
the oracle's multi-thread driver (sweep r on thread r mod P; bitwise equal to
the serial order, which tests/test_oracle_pins.py checks), and stored:

  full_n16384_bw128_tw32_f64_graded.npz   d, e  (float64 oracle), sens
  full_n32768_bw256_tw32_f32.npz          d, e  (float32 oracle), sens,
                                          d64, e64 (float64 oracle run on the
                                          same float32 input, widened exactly)

sens is the oracle's own sensitivity: the largest change of |d|, |e| (over
||A||_F) when the input is perturbed by about one ulp
(band_inputs.perturb_ulp, seeds band_inputs.SENSITIVITY_SEEDS).

The float64 result of the float32 workload is the second reference the
float32 parity tests use to bound the GPU's forward error by the float32
oracle's own.  Each file also stores the input's Frobenius norm and a
SHA-256 of the input band, so that a changed generator shows up as a
mismatch rather than as a parity failure.
"""
import hashlib
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import band_inputs as bi  # noqa: E402
import oracle  # noqa: E402

TARGETS = {
    "n16384": ("n16384_bw128_tw32_f64_graded", False),
    "n32768": ("n32768_bw256_tw32_f32", True),
}


def path_of(name: str) -> str:
    return os.path.join(HERE, f"full_{name}.npz")


def band_digest(band: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(band).tobytes()).hexdigest()


def threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def de_change(d, e, d_ref, e_ref, fro):
    """max | |d|-|d_ref| |, | |e|-|e_ref| | over ||A||_F."""
    def dist(a, b):
        return float(np.abs(np.abs(a.astype(np.float64)) - np.abs(b.astype(np.float64))).max()) if a.size else 0.0
    return max(dist(d, d_ref), dist(e, e_ref)) / fro


def write(key: str) -> None:
    """Compute what the file of workload `key` lacks (an existing file is
    kept when its input digest still matches) and store it."""
    name, widen = TARGETS[key]
    w = bi.by_name(name)
    band = bi.make_workload(w)
    digest = band_digest(band)
    out = {}
    if os.path.exists(path_of(name)):
        with np.load(path_of(name)) as z:
            if str(z["band_sha256"]) == digest:
                out = {k: z[k] for k in z.files}
    out["fro"] = np.float64(np.linalg.norm(band.astype(np.float64)))
    out["band_sha256"] = np.array(digest)
    p = threads()

    def run(b):
        t0 = time.time()
        d, e = oracle.bidiagonal_pipelined(b, w.n, w.bw, w.tw, p, time_limit=7200.0)
        print(f"{name}: {b.dtype} oracle on {p} threads, {time.time() - t0:.1f} s", flush=True)
        return d, e

    if "d" not in out:
        out["d"], out["e"] = run(band)
        np.savez_compressed(path_of(name), **out)
    if widen and "d64" not in out:
        out["d64"], out["e64"] = run(band.astype(np.float64))
        np.savez_compressed(path_of(name), **out)
    if "sens" not in out:
        sens = 0.0
        for sd in bi.SENSITIVITY_SEEDS:
            d2, e2 = run(bi.perturb_ulp(band, sd))
            sens = max(sens, de_change(d2, e2, out["d"], out["e"], float(out["fro"])))
        out["sens"] = np.float64(sens)
    np.savez_compressed(path_of(name), **out)


def main(argv):
    for key in (argv or list(TARGETS)):
        write(key)


if __name__ == "__main__":
    main(sys.argv[1:])
