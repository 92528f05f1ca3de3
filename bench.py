"""Benchmark of the band -> bidiagonal reduction on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--scheduler 0|1|2|3|4] [--group-size G]
                    [--no-sweep] [--no-cpu] [--no-e2e]
    python bench.py --profile-pass WORKLOAD:N:PASS:SCHEDULER:DTYPE[:MAX_CTAS]

One step is one whole reduction (every pass down to bidiagonal form, plus the
fill-row zeroing and the d/e extraction) of one synthetic band.  Before each
step the pristine band is copied into the work buffer and L2 is flushed by
writing a 256 MiB buffer, both outside the timed events, so every timed step
starts with its input resident in HBM and not in L2.

metric: effective GB/s = algorithmic bytes of the reduction (each step's
right and left blocks read once and written once; bb_model_bytes) / device
time per reduction.  ms_per_step is the device time of one reduction.

With --gpus N (under torchrun) every rank reduces its own band (seed offset
by the rank): independent replicas, no collective on the data path; the value
is all ranks' bytes over the slowest rank's time.

--impl reference times the CPU oracle (the plain serial implementation the
tests check the GPU against) on the host, on the same workload and metric.

Besides the contract's keys the line carries: roofline (the dominant pass
kernel against the measured HBM copy rate, and against the nominal ~8 TB/s,
on which the 40% target is judged; with its ncu DRAM traffic), cpu_baseline
(the serial oracle on one host core), cpu_pipelined (the oracle's
multi-thread pipelined chase, context only), e2e (host buffers in, d and e
out, copies timed), latency_chain (per pass: sweeps, half-step lag and the
measured time per dependent link, the quantity that bounds these latency
chains), median_ms / min_ms (of this rank's timed steps), per_scheduler (the
main workload under each scheduler: per-cycle launches, their CUDA-graph
replay, the flag and the group kernel), per_workload (each other workload,
5 timed steps after 2 warm-up steps: its own roofline, e2e and CPU baseline
-- the serial oracle where a reduction takes seconds, else the oracle's
multi-thread driver on the first pass), singular_values (bb_singular_values
on the reduction's output), symmetric (the symmetric band variant),
half_storage (the main workload's band in binary16 storage, BB_F16) and
stage1 (bb_dense_to_band on a dense matrix of the main workload's order,
bandwidth and dtype).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import band_inputs as bi  # noqa: E402

METRIC = "band→bidiagonal ms/reduction and effective GB/s (% of HBM peak), N=4k–32k"
MAIN_WORKLOAD = bi.WORKLOADS[1].name
SWEEP_WORKLOADS = [w.name for w in bi.WORKLOADS[1:]]
HBM_FALLBACK_GBS = 6800.0
# GB300 HBM3e nominal bandwidth (about 8 TB/s).  The 40% target is judged
# against this figure, the stricter of the two; fractions of the measured
# copy rate (MEASURED_PEAKS.json) are reported beside it.
NOMINAL_HBM_GBS = 7900.0
L2_FLUSH_BYTES = 256 << 20


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return HBM_FALLBACK_GBS, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_seed(w: bi.Workload, rank: int) -> int:
    """Seed of rank `rank`'s band: every replica reduces a different matrix."""
    return w.seed + 1000 * rank


def aggregate(values_per_rank_ms: float, units: float, group=None):
    """Max over ranks of the time and sum over ranks of the units."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return values_per_rank_ms, units
    dev = "cpu" if dist.get_backend(group) == "gloo" else torch.device("cuda", torch.cuda.current_device())
    t = torch.tensor([values_per_rank_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"bb_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    mhz.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, flag in zip(names, parts[5:9]):
                    if flag.lower() == "active":
                        reasons.add(nm)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


def run_ours(w: bi.Workload, steps: int, warmup: int, scheduler: int, rank: int, with_e2e: bool,
             group_size: int = 0):
    import torch

    import banded_svd_stage_gb300 as bb
    from banded_svd_stage_gb300.tensor import Reducer

    dev = torch.device("cuda", torch.cuda.current_device())
    tdt = torch.float32 if w.dtype == "f32" else torch.float64
    esz = 4 if w.dtype == "f32" else 8
    band_np = bi.make_band(w.n, w.bw, w.tw, w.dtype, w.dist, w.graded, replica_seed(w, rank))
    pristine = torch.from_numpy(band_np).to(dev)
    work = torch.empty_like(pristine)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    red = Reducer(w.n, w.bw, tdt, scheduler=scheduler)
    if group_size:
        bb.bb_set_param(red.h, bb.BB_PARAM_GROUP_SIZE, group_size)
    red.enable_timing(True)
    d = torch.empty(w.n, dtype=tdt, device=dev)
    e = torch.empty(w.n, dtype=tdt, device=dev)
    stream = torch.cuda.current_stream(dev)
    model_bytes = bb.bb_model_bytes(w.n, w.bw, w.tw, esz)
    npass = bb.bb_num_passes(w.bw, w.tw)
    pass_bytes = [bb.bb_model_bytes(w.n, w.bw, w.tw, esz, i) for i in range(npass)]

    def one(timed_events):
        work.copy_(pristine)
        flush.fill_(rank + 1)
        if timed_events:
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
        red.reduce_(work, w.tw, d, e, stream)
        if timed_events:
            ev1.record(stream)
            return ev0, ev1
        return None

    for _ in range(warmup):
        one(False)
    red.check(stream)
    torch.cuda.synchronize()
    events, pass_ms, launches = [], [], 0
    for _ in range(steps):
        events.append(one(True))
        launches += bb.bb_last_launches(red.h)
        torch.cuda.synchronize()
        pass_ms.append(red.pass_ms())
    red.check(stream)
    ms = [a.elapsed_time(b) for a, b in events]
    kernels = red.pass_kernels()
    # dominant kernel: the pass kernel, one launch per pass (persistent scheduler)
    per_pass_ms = np.array(pass_ms)  # steps x passes
    e2e = None
    if with_e2e:
        e2e = run_e2e(w, band_np, steps, warmup, scheduler, model_bytes)
    red.close()
    return {
        "ms": ms, "model_bytes": model_bytes, "pass_bytes": pass_bytes,
        "pass_ms_mean": per_pass_ms.mean(axis=0).tolist(), "launches": launches,
        "e2e": e2e, "band_bytes": band_np.nbytes, "esz": esz, "kernels": kernels,
    }


def run_svals(w: bi.Workload, steps: int, warmup: int):
    """Device time of bb_singular_values on the bidiagonal the library
    produces for workload w (the step after the reduction), CUDA events on
    the launching stream."""
    import torch

    import banded_svd_stage_gb300 as bb
    dev = torch.device("cuda", torch.cuda.current_device())
    band = torch.from_numpy(bi.make_workload(w)).to(dev)
    d = torch.empty(w.n, dtype=band.dtype, device=dev)
    e = torch.empty(max(w.n - 1, 1), dtype=band.dtype, device=dev)
    sig = torch.empty(w.n, dtype=band.dtype, device=dev)
    h = bb.bb_create(w.n, w.bw, bb.dtype_code(w.dtype))
    stream = torch.cuda.current_stream(dev)
    try:
        bb.bb_reduce(h, band, band.shape[1], w.tw, d, e, stream)
        if bb.bb_status_sync(h, stream) != bb.BB_OK:
            raise RuntimeError("reduction failed")
    finally:
        bb.bb_destroy(h)
    code = bb.dtype_code(w.dtype)
    for _ in range(warmup):
        bb.bb_singular_values(code, w.n, d, e, sig, stream)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        bb.bb_singular_values(code, w.n, d, e, sig, stream)
        ev1.record(stream)
        torch.cuda.synchronize()
        times.append(ev0.elapsed_time(ev1))
    ms = statistics.median(times)
    return {"ms": ms, "n": w.n, "values_per_s": w.n / (ms * 1e-3), "kernel": "bidiag_svals_kernel",
            "launches": 1, "method": "multisection on Sturm counts of the 2n Golub-Kahan tridiagonal, "
                                     "a group of lanes per singular value"}


def run_sym(w: bi.Workload, steps: int, warmup: int):
    """Symmetric variant: device time of bb_sym_reduce on a symmetric band of
    the workload's n, bandwidth, tw, entry distribution and dtype (L2
    flushed and the band restored before each step, outside the events),
    beside the oracle's pipelined multi-thread chase on the host."""
    import torch

    import banded_svd_stage_gb300 as bb
    dev = torch.device("cuda", torch.cuda.current_device())
    sb_np = bi.make_sym_band(w.n, w.bw, w.tw, w.dtype, w.dist, seed=w.seed)
    pristine = torch.from_numpy(sb_np).to(dev)
    band = pristine.clone()
    d = torch.empty(w.n, dtype=band.dtype, device=dev)
    e = torch.empty(max(w.n - 1, 1), dtype=band.dtype, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    h = bb.bb_create(w.n, w.bw, bb.dtype_code(w.dtype))
    stream = torch.cuda.current_stream(dev)
    times = []
    try:
        for i in range(warmup + steps):
            band.copy_(pristine)
            flush.fill_(i & 0xFF)
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            bb.bb_sym_reduce(h, band, band.shape[1], w.tw, d, e, stream)
            ev1.record(stream)
            if bb.bb_status_sync(h, stream) != bb.BB_OK:
                raise RuntimeError("symmetric reduction failed: " + bb.bb_last_error())
            if i >= warmup:
                times.append(ev0.elapsed_time(ev1))
        # per pass: the group kernel (its sweeps per CTA) or the flag kernel
        names = {2: "sym_pass_kernel", 3: "pass_group_kernel<SymChase>"}
        kernels = [f"{names.get(bb.bb_last_pass_kernel(h, i), '?')}"
                   + (f" g={bb.bb_last_pass_group(h, i)}" if bb.bb_last_pass_kernel(h, i) == 3 else "")
                   for i in range(bb.bb_last_num_passes(h))]
        launches = int(bb.bb_last_launches(h))
    finally:
        bb.bb_destroy(h)
    out = {"ms": statistics.median(times), "n": w.n, "bw": w.bw, "tw": w.tw, "dtype": w.dtype,
           "kernels": kernels, "launches": launches}
    try:
        import oracle
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        P = max(1, min(cores, 2 * w.n // (3 * max(w.bw, 1)), w.n // 256))
        t0 = time.perf_counter()
        work = sb_np.copy()
        oracle.sym_reduce_band_pipelined(work, w.n, w.bw, w.tw, P, time_limit=60.0)
        out["cpu_pipelined_ms"] = (time.perf_counter() - t0) * 1e3
        out["cpu_threads"] = P
    except Exception as ex:  # context only
        out["cpu_pipelined_error"] = f"{type(ex).__name__}: {ex}"
    return out


def run_half(w: bi.Workload, steps: int, warmup: int):
    """Binary16 storage (BB_F16): device time of bb_reduce on the workload's
    band rounded to binary16 (L2 flushed and the band restored before each
    step, outside the events), with its algorithmic bytes at 2 bytes an
    entry."""
    import torch

    import banded_svd_stage_gb300 as bb
    dev = torch.device("cuda", torch.cuda.current_device())
    band_np = bi.make_band(w.n, w.bw, w.tw, "f64", w.dist, w.graded, w.seed).astype(np.float16)
    pristine = torch.from_numpy(band_np).to(dev)
    band = pristine.clone()
    d = torch.empty(w.n, dtype=torch.float16, device=dev)
    e = torch.empty(max(w.n - 1, 1), dtype=torch.float16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    h = bb.bb_create(w.n, w.bw, bb.BB_F16)
    stream = torch.cuda.current_stream(dev)
    times = []
    try:
        for i in range(warmup + steps):
            band.copy_(pristine)
            flush.fill_(i & 0xFF)
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            bb.bb_reduce(h, band, band.shape[1], w.tw, d, e, stream)
            ev1.record(stream)
            if bb.bb_status_sync(h, stream) != bb.BB_OK:
                raise RuntimeError("binary16 reduction failed: " + bb.bb_last_error())
            if i >= warmup:
                times.append(ev0.elapsed_time(ev1))
        # per pass: the group kernel on binary16 columns or the binary16 flag kernel
        names = {3: "pass_group_kernel<float, W, BidiagChase, __half>", 5: "pass_half_kernel"}
        kernels = [names.get(bb.bb_last_pass_kernel(h, i), "?")
                   + (f" g={bb.bb_last_pass_group(h, i)}" if bb.bb_last_pass_kernel(h, i) == 3 else "")
                   for i in range(bb.bb_last_num_passes(h))]
        launches = int(bb.bb_last_launches(h))
    finally:
        bb.bb_destroy(h)
    ms = statistics.median(times)
    mb = model_bytes_np(w.n, w.bw, w.tw, 2)
    return {"ms": ms, "n": w.n, "bw": w.bw, "tw": w.tw, "dtype": "f16 storage, f32 arithmetic",
            "effective_gbs": mb / (ms * 1e-3) / 1e9, "kernels": kernels, "launches": launches}


def stage1_flops(n: int, bw: int) -> float:
    """Flops of stage 1's rank-one applications (a dot product and an update,
    4 flops an entry): every QR reflector j on rows j.. of columns j+1..,
    every LQ reflector i on rows i+1.. of columns i+bw.."""
    tot = 0.0
    for k in range(0, n, bw):
        for j in range(k, min(k + bw, n)):
            if j + 1 < n:
                tot += 4.0 * (n - j) * (n - j - 1)
        for i in range(k, min(k + bw, n)):
            c0 = i + bw
            if c0 + 1 < n:
                tot += 4.0 * (n - i - 1) * (n - c0)
    return tot


def run_stage1(w: bi.Workload, steps: int, warmup: int):
    """Stage 1 (bb_dense_to_band) on a seeded dense n x n matrix of the
    workload's dtype, to the workload's bandwidth: device time per call."""
    import torch

    import banded_svd_stage_gb300 as bb
    dev = torch.device("cuda", torch.cuda.current_device())
    rng = np.random.default_rng(w.seed)
    a_np = rng.standard_normal((w.n, w.n)).astype(np.float32 if w.dtype == "f32" else np.float64)
    pristine = torch.from_numpy(a_np).to(dev)
    a = pristine.clone()
    code = bb.dtype_code(w.dtype)
    nbytes = bb.bb_dense_to_band_workspace(w.n, w.bw, code)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    times = []
    for i in range(warmup + steps):
        a.copy_(pristine)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        bb.bb_dense_to_band(code, w.n, w.bw, a, w.n, ws, nbytes, stream)
        ev1.record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            times.append(ev0.elapsed_time(ev1))
    ms = statistics.median(times)
    fl = stage1_flops(w.n, w.bw)
    return {"ms": ms, "n": w.n, "bw": w.bw, "dtype": w.dtype, "gflops": fl / (ms * 1e-3) / 1e9,
            "flops_model": "4 flops per entry of every rank-one application",
            "kernels": "s1_panel_smem_kernel (s1_panel_kernel for panels too tall for shared memory), "
                       "s1_gemm_kernel, s1_reduce_tri_kernel"}


def run_e2e(w, band_np, steps, warmup, scheduler, model_bytes):
    """bb_reduce_host from pinned host memory: H2D of the band, reduction, D2H
    of d and e, inside the timed region (host wall clock around the call,
    which synchronizes)."""
    import torch

    import banded_svd_stage_gb300 as bb
    h = bb.bb_create(w.n, w.bw, bb.dtype_code(w.dtype))
    bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, scheduler)
    src = torch.from_numpy(band_np).pin_memory()
    tdt = torch.float32 if w.dtype == "f32" else torch.float64
    d = torch.empty(w.n, dtype=tdt).pin_memory()
    e = torch.empty(w.n, dtype=tdt).pin_memory()
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    times = []
    for i in range(warmup + steps):
        flush.fill_(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        bb.bb_reduce_host(h, src, band_np.shape[1], w.tw, d, e, stream)
        t1 = time.perf_counter()
        if i >= warmup:
            times.append((t1 - t0) * 1e3)
    bb.bb_destroy(h)
    ms = statistics.median(times)
    return {"value": model_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(band_np.nbytes),
            "d2h_bytes_per_step": int((2 * w.n - 1) * (4 if w.dtype == "f32" else 8))}


def cpu_model() -> str:
    """The host CPU's model name (Linux: lscpu's "Model name", else
    /proc/cpuinfo), for the CPU timings' context."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(line.split(":", 1) for line in out.splitlines() if ":" in line)
        name = fields.get("Model name", "").strip()
        vendor = fields.get("Vendor ID", "").strip()
        if name and name != "-":
            return f"{vendor} {name}".strip() if vendor and vendor not in name else name
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_rate(w: bi.Workload, budget_s: float = 12.0):
    """The oracle, as it stands, on one host core: whole reductions of the
    workload repeated until about budget_s seconds have elapsed (one at least)."""
    import oracle
    band = bi.make_workload(w)
    model_bytes = None
    try:
        import banded_svd_stage_gb300 as bb
        model_bytes = bb.bb_model_bytes(w.n, w.bw, w.tw, 4 if w.dtype == "f32" else 8)
    except Exception:
        model_bytes = _model_bytes_py(w)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.bidiagonal(band, w.n, w.bw, w.tw)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el / reps * (reps + 1) > 2.5 * budget_s:
            break
    sec = el / reps
    return {"value": model_bytes / sec / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
            "ms_per_reduction": sec * 1e3,
            "sample": f"{reps} whole serial reductions of {w.name} ({el:.1f} s)"}


def cpu_pipelined_rate(w: bi.Workload, budget_s: float = 6.0):
    """The oracle's pipelined driver on the host cores: sweep r on thread
    r mod P, each sweep spinning on its predecessor's count of finished
    half-steps (the multi-threaded chase of "A two-stage reduction on an Apple
    M5 Pro", Section 6), bitwise equal to the serial oracle.  P follows that
    section's limits: at most the usable cores, 2n / (3 bw) and n / 256."""
    import oracle
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    P = max(1, min(cores, 2 * w.n // (3 * max(w.bw, 1)), w.n // 256))
    band = bi.make_workload(w)
    try:
        import banded_svd_stage_gb300 as bb
        model_bytes = bb.bb_model_bytes(w.n, w.bw, w.tw, 4 if w.dtype == "f32" else 8)
    except Exception:
        model_bytes = _model_bytes_py(w)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.bidiagonal_pipelined(band, w.n, w.bw, w.tw, P, time_limit=60.0)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el / reps * (reps + 1) > 2.5 * budget_s:
            break
    sec = el / reps
    return {"value": model_bytes / sec / 1e9, "unit": "GB/s", "cores": P, "kind": "oracle, pipelined sweeps",
            "cpu": cpu_model(),
            "ms_per_reduction": sec * 1e3,
            "sample": f"{reps} whole reductions of {w.name} on {P} threads ({el:.1f} s)"}


def cpu_baseline_for(w: bi.Workload, budget_s: float = 12.0, serial_limit_bytes: float = 60e9):
    """CPU baseline of workload w, on the host cores, as the oracle stands:
    the serial oracle on one core (whole reductions, repeated for about
    budget_s) where one reduction takes seconds, otherwise a bounded sample:
    the oracle's multi-thread driver on the first pass only (its bytes over
    its time; the thread count follows that driver's limits).  Workloads of
    more than serial_limit_bytes algorithmic bytes take the second form."""
    import oracle
    elem = 4 if w.dtype == "f32" else 8
    total = model_bytes_np(w.n, w.bw, w.tw, elem)
    if total <= serial_limit_bytes:
        out = cpu_oracle_rate(w, budget_s)
        out["model_bytes"] = total
        return out
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    P = max(1, min(cores, 2 * w.n // (3 * max(w.bw, 1)), w.n // 256))
    band = bi.make_workload(w)
    pass_bytes = model_bytes_np(w.n, w.bw, w.tw, elem, 0)
    t0 = time.perf_counter()
    oracle.reduce_band_pipelined(band, w.n, w.bw, w.tw, P, time_limit=300.0, pass_lo=0, pass_hi=1)
    sec = time.perf_counter() - t0
    t = min(w.tw, w.bw - 1)
    return {"value": pass_bytes / sec / 1e9, "unit": "GB/s", "cores": P, "kind": "oracle, pipelined sweeps",
            "cpu": cpu_model(), "ms_per_pass": sec * 1e3,
            "sample": f"first pass ({w.bw}->{w.bw - t}) of {w.name} on {P} threads ({sec:.1f} s, "
                      f"{pass_bytes / 1e9:.1f} GB of the reduction's {total / 1e9:.1f} GB)"}


def roofline_of(res, hbm: float, peak_src: str, workload: str):
    """Roofline entry of the dominant pass kernel of one run (run_ours)."""
    kname, achieved, nl, kbytes, kms = dominant_kernel(res)
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": (achieved / hbm) if achieved else None,
            "frac_of_nominal": (achieved / NOMINAL_HBM_GBS) if achieved else None,
            "nominal_peak": NOMINAL_HBM_GBS, "traffic": traffic_for(kname, workload),
            "kernel": kname, "peak_source": peak_src, "launches_per_step": nl,
            "algorithmic_bytes_per_launch": kbytes / nl if nl else None,
            "ms_per_launch": kms / nl if nl else None,
            "achieved_def": "algorithmic bytes of the kernel's passes / their CUDA-event time "
                            "(events on the launching stream around each pass launch)"}


def _model_bytes_py(w):
    """Algorithmic bytes of workload w, step by step (plain Python; the
    definition, kept for the tests)."""
    s = 4 if w.dtype == "f32" else 8
    tot, b = 0, w.bw
    while b > 1:
        t = min(w.tw, b - 1)
        bp = b - t
        for r in range(0, w.n - bp - 1):
            c = r + bp
            k = 0
            while c + 1 <= w.n - 1:
                p = r if k == 0 else c - b
                ce = min(c + t, w.n - 1)
                cend = min(ce + b, w.n - 1)
                ww = ce - c + 1
                tot += 2 * s * ((ce - p + 1) * ww + ww * (cend - c + 1))
                k += 1
                c += b
        b -= t
    return tot


def model_bytes_np(n: int, bw: int, tw: int, elem: int, pass_index: int = -1) -> float:
    """The same count as _model_bytes_py (and bb_model_bytes), vectorised over
    the sweeps with numpy, one step index at a time: every step's right block
    (rows p..ce x cols c..ce) and left block (rows c..ce x cols c..cend) read
    once and written once.  Needs no GPU library (the reference arm uses it)."""
    import numpy as np
    tot, b, pi = 0, bw, 0
    while b > 1:
        t = min(tw, b - 1)
        bp = b - t
        if pass_index < 0 or pi == pass_index:
            r = np.arange(max(0, n - bp - 1), dtype=np.int64)
            k = 0
            while r.size:
                c = r + bp + k * b
                r = r[c + 1 <= n - 1]
                c = c[c + 1 <= n - 1]
                if not r.size:
                    break
                p = r if k == 0 else c - b
                ce = np.minimum(c + t, n - 1)
                cend = np.minimum(ce + b, n - 1)
                ww = ce - c + 1
                tot += int((2 * elem * ((ce - p + 1) * ww + ww * (cend - c + 1))).sum())
                k += 1
        b -= t
        pi += 1
    return float(tot)


def latency_chain(n: int, bw: int, tw: int, pass_ms):
    """Per pass of the plan: the sweeps, the half-step lag L between
    consecutive sweeps (2 when b - t >= 3, 3 when b - t == 2, 4 when
    b - t == 1) and the measured time per lag unit, pass_ms / (sweeps * L).
    A pass is a chain of about sweeps * L dependent half-steps, so this is
    the effective latency of one link, the quantity the kernels must lower
    (the bytes a link moves are fixed by the method)."""
    out = []
    b, i = bw, 0
    while b > 1 and i < len(pass_ms):
        t = min(tw, b - 1)
        bp = b - t
        lag = 2 if bp >= 3 else (3 if bp == 2 else 4)
        sweeps = max(0, n - bp - 1)
        us = (pass_ms[i] * 1e3 / (sweeps * lag)) if sweeps and pass_ms[i] is not None else None
        out.append({"b": b, "t": t, "sweeps": sweeps, "lag": lag, "us_per_link": us})
        b -= t
        i += 1
    return out


KERNEL_NAMES = {1: "pass_cycle_kernel", 2: "pass_persistent_kernel", 3: "pass_group_kernel",
                4: "pass_cycle_kernel"}
SCHEDULER_NAMES = {0: "auto", 1: "per-cycle", 2: "flags", 3: "group", 4: "per-cycle-graph"}


def dominant_kernel(res):
    """(name, achieved GB/s, launches, bytes, ms) of the pass kernel with the
    largest share of the step's pass time."""
    tot = {}
    for (kind, _g), ms, by in zip(res["kernels"], res["pass_ms_mean"], res["pass_bytes"]):
        t = tot.setdefault(kind, [0.0, 0.0, 0])
        t[0] += ms
        t[1] += by
        t[2] += 1
    if not tot:
        return None, None, 0, 0.0, 0.0
    kind = max(tot, key=lambda k: tot[k][0])
    ms, by, nl = tot[kind]
    if kind in (1, 4):
        nl = None  # one launch per cycle: many launches per pass
    ach = by / (ms * 1e-3) / 1e9 if ms > 0 else None
    return KERNEL_NAMES.get(kind, str(kind)), ach, nl if nl else 0, by, ms


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if that summary was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            data = json.load(f)
        from banded_svd_stage_gb300.buildlib import source_digest
        if data.get("source_digest") != source_digest():
            return None
        return data.get("per_launch", {}).get(kernel, {}).get(workload)
    except Exception:
        return None


# Bound of one device-side wait in the profiling modes: a profiler's
# instrumented replay can run a pass far slower than normal, and a CTA then
# waits on its predecessor for longer than the library's default 4 s.
PROFILE_WAIT_MS = 60000


def profile_pass(spec: str) -> int:
    """--profile-pass WORKLOAD:N:PASS:SCHEDULER:DTYPE[:MAX_CTAS] -- one run of
    one pass of the workload's recipe at order N (DTYPE f32, f64 or f16), for
    an ncu capture of that pass's kernel; prints one line, no timing."""
    import torch

    import banded_svd_stage_gb300 as bb
    parts = spec.split(":")
    name, n, p, sched, dt = parts[0], int(parts[1]), int(parts[2]), int(parts[3]), parts[4]
    ctas = int(parts[5]) if len(parts) > 5 else 0
    w = bi.by_name(name)
    if dt == "f16":
        band_np = bi.make_band(n, w.bw, w.tw, "f64", w.dist, w.graded, w.seed).astype(np.float16)
    else:
        band_np = bi.make_band(n, w.bw, w.tw, dt, w.dist, w.graded, w.seed)
    torch.cuda.set_device(0)
    band = torch.from_numpy(band_np).cuda()
    d = torch.empty(n, dtype=band.dtype, device="cuda")
    e = torch.empty(n, dtype=band.dtype, device="cuda")
    h = bb.bb_create(n, w.bw, bb.dtype_code(dt))
    try:
        bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, sched)
        bb.bb_set_param(h, bb.BB_PARAM_WAIT_BUDGET_MS, PROFILE_WAIT_MS)
        bb.bb_set_param(h, bb.BB_PARAM_MAX_CTAS, ctas)
        bb.bb_set_param(h, bb.BB_PARAM_PASS_LO, p)
        bb.bb_set_param(h, bb.BB_PARAM_PASS_HI, p + 1)
        s = torch.cuda.current_stream()
        bb.bb_reduce(h, band, band.shape[1], w.tw, d, e, s)
        st = bb.bb_status_sync(h, s)
    finally:
        bb.bb_destroy(h)
    print(f"profile pass: {name} n={n} pass={p} scheduler={sched} dtype={dt} max_ctas={ctas} status={st}")
    return 0 if st == 0 else 1


def profile_stage1(spec: str) -> int:
    """--profile-stage1 N:BW:DTYPE -- one bb_dense_to_band call on a seeded
    dense N x N matrix (DTYPE f32 or f64) to bandwidth BW, for an ncu launch
    list of stage 1; prints one line, no timing."""
    import torch

    import banded_svd_stage_gb300 as bb
    n_s, bw_s, dt = spec.split(":")
    n, bw = int(n_s), int(bw_s)
    torch.cuda.set_device(0)
    rng = np.random.default_rng(n + bw)
    a = torch.from_numpy(rng.standard_normal((n, n)).astype(np.float32 if dt == "f32" else np.float64)).cuda()
    code = bb.dtype_code(dt)
    nbytes = bb.bb_dense_to_band_workspace(n, bw, code)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    bb.bb_dense_to_band(code, n, bw, a, n, ws, nbytes, torch.cuda.current_stream())
    torch.cuda.synchronize()
    print(f"profile stage1: n={n} bw={bw} dtype={dt}")
    return 0


def profile_sym(spec: str) -> int:
    """--profile-sym N:BW:TW:DTYPE:SCHEDULER -- one bb_sym_reduce on a seeded
    symmetric band (uniform entries, DTYPE f32 or f64), for an ncu capture of
    the symmetric chase's kernels; prints one line, no timing."""
    import torch

    import banded_svd_stage_gb300 as bb
    n_s, bw_s, tw_s, dt, sched_s = spec.split(":")
    n, bw, tw, sched = int(n_s), int(bw_s), int(tw_s), int(sched_s)
    torch.cuda.set_device(0)
    sb = torch.from_numpy(bi.make_sym_band(n, bw, tw, dt, "uniform", seed=n + bw)).cuda()
    d = torch.empty(n, dtype=sb.dtype, device="cuda")
    e = torch.empty(max(n - 1, 1), dtype=sb.dtype, device="cuda")
    h = bb.bb_create(n, bw, bb.dtype_code(dt))
    try:
        bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, sched)
        bb.bb_set_param(h, bb.BB_PARAM_WAIT_BUDGET_MS, PROFILE_WAIT_MS)
        s = torch.cuda.current_stream()
        bb.bb_sym_reduce(h, sb, sb.shape[1], tw, d, e, s)
        st = bb.bb_status_sync(h, s)
        ks = [bb.bb_last_pass_kernel(h, i) for i in range(bb.bb_last_num_passes(h))]
    finally:
        bb.bb_destroy(h)
    print(f"profile sym: n={n} bw={bw} tw={tw} dtype={dt} scheduler={sched} kernels={ks} status={st}")
    return 0 if st == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=MAIN_WORKLOAD)
    ap.add_argument("--scheduler", type=int, default=0)
    ap.add_argument("--group-size", type=int, default=0,
                    help="sweeps per CTA of the group kernel (0: the planner's choice)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer (e2e) leg")
    ap.add_argument("--profile-sym", default=None, metavar="N:BW:TW:DTYPE:SCHEDULER",
                    help="one symmetric reduction, for an ncu capture")
    ap.add_argument("--profile-stage1", default=None, metavar="N:BW:DTYPE",
                    help="one stage-1 call (dense -> band), for an ncu launch list")
    ap.add_argument("--profile-pass", default=None, metavar="WORKLOAD:N:PASS:SCHEDULER:DTYPE[:MAX_CTAS]",
                    help="run one pass once for a profiler capture and exit (no measurement)")
    args = ap.parse_args()
    if args.profile_pass:
        return profile_pass(args.profile_pass)
    if args.profile_stage1:
        return profile_stage1(args.profile_stage1)
    if args.profile_sym:
        return profile_sym(args.profile_sym)
    rank, world, local = dist_env()
    w = bi.by_name(args.workload)

    if args.impl == "reference":
        if rank != 0:
            return 0
        times = []
        import oracle
        band = bi.make_workload(w)
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.bidiagonal(band, w.n, w.bw, w.tw)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        mb = model_bytes_np(w.n, w.bw, w.tw, 4 if w.dtype == "f32" else 8)
        sec = sum(times) / len(times)
        val = mb / sec / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
                "data": "synthetic", "config": {"workload": w.name, "n": w.n, "bw": w.bw, "tw": w.tw},
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
                                 "sample": f"whole serial reductions of {w.name}, one per step"},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    hbm, peak_src = measured_peaks()

    sampler = ClockSampler(local) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t_wall0 = time.perf_counter()
    res = run_ours(w, args.steps, args.warmup, args.scheduler, rank, with_e2e=(world == 1 and not args.no_e2e),
                   group_size=args.group_size)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall0
    clocks = sampler.stop() if sampler else None
    ms_step = sum(res["ms"]) / len(res["ms"])
    ms_max, bytes_all = aggregate(ms_step, res["model_bytes"])
    value = bytes_all / (ms_max * 1e-3) / 1e9
    # roofline of the dominant kernel: the pass kernel (one launch a pass for
    # the flag and group kernels) that takes the most time in a step
    roof = roofline_of(res, hbm, peak_src, w.name)

    sweep = []
    if rank == 0 and world == 1 and not args.no_sweep:
        for ww in bi.WORKLOADS:
            if ww.name == w.name:
                continue
            r2 = run_ours(ww, 5, 2, args.scheduler, rank, with_e2e=not args.no_e2e, group_size=args.group_size)
            m2 = statistics.median(r2["ms"])
            g2 = r2["model_bytes"] / (m2 * 1e-3) / 1e9
            entry = {"workload": ww.name, "config": ww.describe(), "dtype": ww.dtype, "steps": 5, "warmup": 2,
                     "ms_per_reduction": m2, "min_ms": min(r2["ms"]), "effective_gbs": g2,
                     "frac_of_hbm": g2 / hbm, "frac_of_nominal_hbm": g2 / NOMINAL_HBM_GBS,
                     "model_bytes": r2["model_bytes"], "roofline": roofline_of(r2, hbm, peak_src, ww.name),
                     "e2e": r2["e2e"], "pass_ms": r2["pass_ms_mean"], "pass_kernels": r2["kernels"],
                     "latency_chain": latency_chain(ww.n, ww.bw, ww.tw, r2["pass_ms_mean"])}
            if not args.no_cpu:
                try:
                    entry["cpu_baseline"] = cpu_baseline_for(ww)
                except Exception as ex:  # a side measurement never loses the line
                    entry["cpu_baseline"] = {"error": f"{type(ex).__name__}: {ex}"}
            sweep.append(entry)

    # both scheduler families on the main workload, measured in the same run:
    # per-cycle launches (plain and replayed from a CUDA graph) and the
    # persistent kernels (flag, group); the headline uses the automatic choice
    per_sched = None
    if rank == 0 and world == 1 and not args.no_sweep:
        per_sched = {}
        for sc in (1, 4, 2, 3):
            try:
                rs = run_ours(w, max(2, min(args.steps, 3)), 1, sc, rank, with_e2e=False)
                per_sched[SCHEDULER_NAMES[sc]] = {"median_ms": statistics.median(rs["ms"]), "min_ms": min(rs["ms"]),
                                                  "launches": rs["launches"], "pass_ms": rs["pass_ms_mean"]}
            except Exception as ex:  # a side measurement never loses the line
                per_sched[SCHEDULER_NAMES[sc]] = {"error": f"{type(ex).__name__}: {ex}"}

    svals = None
    if rank == 0 and world == 1 and not args.no_sweep:
        svals = run_svals(w, args.steps, args.warmup)
    sym = None
    if rank == 0 and world == 1 and not args.no_sweep:
        try:
            sym = run_sym(w, args.steps, args.warmup)
        except Exception as ex:  # a side measurement never loses the line
            sym = {"error": f"{type(ex).__name__}: {ex}"}

    stage1 = None
    if rank == 0 and world == 1 and not args.no_sweep:
        try:
            stage1 = run_stage1(w, 3, 1)
        except Exception as ex:  # a side measurement never loses the line
            stage1 = {"error": f"{type(ex).__name__}: {ex}"}
    half = None
    if rank == 0 and world == 1 and not args.no_sweep:
        try:
            half = run_half(w, args.steps, args.warmup)
        except Exception as ex:  # a side measurement never loses the line
            half = {"error": f"{type(ex).__name__}: {ex}"}

    cpu = cpu_pipe = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_oracle_rate(w)
        try:
            cpu_pipe = cpu_pipelined_rate(w)
        except Exception as ex:  # context only: never lose the line for it
            cpu_pipe = {"error": f"{type(ex).__name__}: {ex}"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "n": w.n, "bw": w.bw, "tw": w.tw, "dist": w.dist,
                       "graded": w.graded, "scheduler": SCHEDULER_NAMES.get(args.scheduler, str(args.scheduler)),
                       "group_size": args.group_size or "planner",
                       "l2": "flushed between steps (256 MiB write); band restored before each step",
                       "parallelism": f"replicas x{world}"},
            "frac_of_hbm": value / hbm,
            "frac_of_nominal_hbm": value / NOMINAL_HBM_GBS,
            "roofline": roof,
            "cpu_baseline": cpu,
            "cpu_pipelined": cpu_pipe,
            "e2e": res["e2e"],
            "gpu_launches": res["launches"] * world,
            "clocks": clocks,
            "wall_s": wall,
            "pass_kernels": res["kernels"],
            "pass_ms": res["pass_ms_mean"],
            "latency_chain": latency_chain(w.n, w.bw, w.tw, res["pass_ms_mean"]),
            "median_ms": statistics.median(res["ms"]), "min_ms": min(res["ms"]),
            "per_scheduler": per_sched,
            "per_workload": sweep,
            "singular_values": svals,
            "symmetric": sym,
            "half_storage": half,
            "stage1": stage1,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
