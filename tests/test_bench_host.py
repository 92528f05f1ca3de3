"""Host-side logic of bench.py (no GPU): the dominant-kernel roofline
bookkeeping and the staleness guard of the committed DRAM traffic."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_dominant_kernel_picks_the_largest_time_share():
    res = {"kernels": [(2, 0), (2, 0), (3, 5), (3, 5)],
           "pass_ms_mean": [10.0, 10.0, 30.0, 5.0],
           "pass_bytes": [100e9, 100e9, 50e9, 10e9]}
    name, ach, nl, by, ms = bench.dominant_kernel(res)
    assert name == "pass_group_kernel" and nl == 2
    assert by == 60e9 and ms == 35.0
    assert ach == pytest.approx(60e9 / 35e-3 / 1e9)


def test_dominant_kernel_per_cycle_has_no_launch_count():
    res = {"kernels": [(1, 0)], "pass_ms_mean": [5.0], "pass_bytes": [1e9]}
    name, ach, nl, _, _ = bench.dominant_kernel(res)
    assert name == "pass_cycle_kernel" and nl == 0
    res = {"kernels": [(4, 0)], "pass_ms_mean": [5.0], "pass_bytes": [1e9]}
    assert bench.dominant_kernel(res)[0] == "pass_cycle_kernel"


def test_dominant_kernel_empty():
    assert bench.dominant_kernel({"kernels": [], "pass_ms_mean": [], "pass_bytes": []})[0] is None


def test_committed_traffic_is_reported_only_for_its_sources():
    """bench reports the DRAM bytes of profiles/traffic.json only while the
    kernel sources are the ones they were taken on."""
    from banded_svd_stage_gb300.buildlib import source_digest
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        data = json.load(f)
    got = bench.traffic_for("pass_group_kernel", "n4096_bw16_tw8_f32")
    if data["source_digest"] == source_digest():
        assert got == data["per_launch"]["pass_group_kernel"]["n4096_bw16_tw8_f32"] > 0
    else:
        assert got is None
    assert bench.traffic_for("pass_group_kernel", "no_such_workload") is None


def test_traffic_is_dropped_when_sources_change(monkeypatch):
    import banded_svd_stage_gb300.buildlib as bl
    monkeypatch.setattr(bl, "source_digest", lambda: "0000000000000000")
    assert bench.traffic_for("pass_group_kernel", "n4096_bw16_tw8_f32") is None


def test_measured_peak_is_read():
    peak, src = bench.measured_peaks()
    assert peak > 1000 and src in ("measured", "fallback")


def test_cpu_legs_report_rates_and_threads():
    import band_inputs as bi
    w = bi.WORKLOADS[0]
    serial = bench.cpu_oracle_rate(w, budget_s=0.3)
    pipe = bench.cpu_pipelined_rate(w, budget_s=0.3)
    assert serial["cores"] == 1 and serial["value"] > 0
    assert pipe["value"] > 0 and 1 <= pipe["cores"] <= max(1, w.n // 256)
    # the thread count follows the limits of the pipelined chase
    big = bi.by_name("n4096_bw16_tw8_f32")
    cores = len(os.sched_getaffinity(0))
    assert min(cores, 16) == max(1, min(cores, 2 * big.n // (3 * big.bw), big.n // 256))


def test_traffic_digest_covers_the_pass_kernels_only():
    import banded_svd_stage_gb300.buildlib as bl
    srcs = set(bl.PASS_KERNEL_SOURCES)
    for f in srcs:
        assert os.path.exists(os.path.join(bl.CSRC, f)), f
    # every file defining one of the bidiagonal pass kernels, and the planner
    # that launches them
    kernels = ("pass_persistent_kernel(", "pass_group_kernel(", "pass_cycle_kernel(")
    for f in os.listdir(bl.CSRC):
        text = open(os.path.join(bl.CSRC, f)).read()
        if f.endswith((".cu", ".cuh")) and any(k in text for k in kernels):
            assert f in srcs, f
    assert "bb_plan.cu" in srcs and "bb_launch.cuh" in srcs
    # the boundary and the other kernels are not part of it
    assert not srcs & {"bb_api.cu", "bb_noalloc.cu", "bb_svals.cu"}
    assert len(bl.source_digest()) == 16


def test_latency_chain_of_the_main_workload():
    # measured pass times of the main workload (n = 4096, bw = 16, tw = 8)
    out = bench.latency_chain(4096, 16, 8, [11.19, 19.89])
    assert [(p["b"], p["t"], p["sweeps"], p["lag"]) for p in out] == [(16, 8, 4087, 2), (8, 7, 4094, 4)]
    assert abs(out[0]["us_per_link"] - 11.19e3 / (4087 * 2)) < 1e-9
    assert abs(out[1]["us_per_link"] - 19.89e3 / (4094 * 4)) < 1e-9
    # every pass of the largest workload, lags 2 except the last (b - t = 1)
    big = bench.latency_chain(32768, 256, 32, [1.0] * 8)
    assert [p["lag"] for p in big] == [2] * 7 + [4] and big[-1]["t"] == 31


def test_cpu_model_is_reported():
    m = bench.cpu_model()
    assert isinstance(m, str) and m.strip()


def test_model_bytes_without_the_gpu_library():
    """The reference arm's vectorised count equals the plain step-by-step
    definition (and, through tests/test_abi.py, the library's)."""
    import band_inputs as bi
    for (n, bw, tw, dt) in ((300, 20, 7, "f32"), (257, 8, 7, "f64"), (100, 33, 32, "f32"), (64, 1, 1, "f64"),
                            (50, 30, 4, "f64")):
        w = bi.Workload("x", n, bw, tw, dt, "normal", False, 0)
        elem = 4 if dt == "f32" else 8
        assert bench.model_bytes_np(n, bw, tw, elem) == bench._model_bytes_py(w)
        npass = len(__import__("oracle").pass_plan(bw, tw))
        assert sum(bench.model_bytes_np(n, bw, tw, elem, p) for p in range(npass)) == bench._model_bytes_py(w)


def test_cpu_baseline_for_both_kinds():
    import band_inputs as bi
    w = bi.Workload("small", 600, 24, 8, "f32", "normal", False, 0)
    serial = bench.cpu_baseline_for(w, budget_s=0.2)
    assert serial["kind"] == "oracle" and serial["cores"] == 1 and serial["value"] > 0
    pipe = bench.cpu_baseline_for(w, budget_s=0.2, serial_limit_bytes=0)
    assert pipe["kind"].startswith("oracle, pipelined") and pipe["cores"] >= 1 and pipe["value"] > 0
    assert "first pass (24->16)" in pipe["sample"]


def test_stage1_flop_model():
    # n = 5, bw = 2: QR reflectors j = 0..3 act on (5 - j) x (4 - j) entries,
    # LQ reflectors of panel 0 (i = 0, 1; c0 = 2, 3) on (4 - i) x (5 - c0),
    # of panel 1 (i = 2; c0 = 4 -> none)
    want = 4.0 * (5 * 4 + 4 * 3 + 3 * 2 + 2 * 1) + 4.0 * (4 * 3 + 3 * 2)
    assert bench.stage1_flops(5, 2) == want
