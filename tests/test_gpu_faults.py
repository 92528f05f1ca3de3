"""Failure detection on the GPU without faulting it.

A CTA told not to report its progress (BB_PARAM_STALL_SWEEP) leaves the sweeps
after it waiting on a flag that nothing sets; every such wait is bounded
(BB_PARAM_WAIT_BUDGET_MS), latches BB_ERR_TIMEOUT in the device status word
and returns, so the kernel ends and the context stays usable.
"""
import numpy as np
import pytest
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb
import oracle
from gpu_helpers import TOL, fro_of_band, sigma_bidiagonal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sched", [0, 2, 3])
def test_stalled_sweep_times_out_and_context_survives(sched):
    n, bw, tw = 2000, 32, 8
    band = bi.make_band(n, bw, tw, "f32", "normal", seed=1)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(band).to(dev)
    d = torch.empty(n, dtype=torch.float32, device=dev)
    e = torch.empty(n - 1, dtype=torch.float32, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F32)
    try:
        bb.bb_set_param(h, bb.BB_PARAM_SCHEDULER, sched)
        bb.bb_set_param(h, bb.BB_PARAM_WAIT_BUDGET_MS, 50)
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, 5)
        s = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_ERR_TIMEOUT
        # the status word was cleared and the same handle works again
        bb.bb_set_param(h, bb.BB_PARAM_STALL_SWEEP, -1)
        x.copy_(torch.from_numpy(band).to(dev))
        bb.bb_reduce(h, x, band.shape[1], tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK
    finally:
        bb.bb_destroy(h)
    d_ref, e_ref = oracle.bidiagonal(band, n, bw, tw)
    s = sigma_bidiagonal(d.cpu().numpy(), e.cpu().numpy())
    s_ref = sigma_bidiagonal(d_ref, e_ref)
    assert np.abs(s - s_ref).max() <= TOL["f32"] * fro_of_band(band)


def test_argument_errors_are_reported_not_launched():
    n, bw, tw = 100, 10, 3
    dev = torch.device("cuda:0")
    x = torch.zeros((n, bw + 2 * tw + 1), dtype=torch.float64, device=dev)
    d = torch.empty(n, dtype=torch.float64, device=dev)
    e = torch.empty(n - 1, dtype=torch.float64, device=dev)
    h = bb.bb_create(n, bw, bb.BB_F64)
    try:
        with pytest.raises(bb.BBError) as ex:
            bb.bb_reduce(h, x, bw + 2 * tw, tw, d, e)       # ldab too small
        assert ex.value.status == bb.BB_ERR_LDAB
        with pytest.raises(bb.BBError) as ex:
            bb.bb_reduce(h, x, x.shape[1], bw, d, e)         # tw > bw - 1
        assert ex.value.status == bb.BB_ERR_INVALID_ARG
        with pytest.raises(bb.BBError) as ex:
            bb.bb_reduce(h, 0, x.shape[1], tw, d, e)         # null band
        assert ex.value.status == bb.BB_ERR_INVALID_ARG
        host = np.zeros((n, x.shape[1]))
        with pytest.raises(bb.BBError) as ex:
            bb.bb_reduce(h, host, x.shape[1], tw, d, e)      # host pointer
        assert ex.value.status == bb.BB_ERR_INVALID_ARG
        with pytest.raises(bb.BBError):
            bb.bb_set_param(h, bb.BB_PARAM_TPB, 100)
    finally:
        bb.bb_destroy(h)
    with pytest.raises(bb.BBError):
        bb.bb_create(10, 10, bb.BB_F32)                      # bw >= n
    with pytest.raises(bb.BBError):
        bb.bb_create(10, 3, 7)                               # dtype


def test_timing_and_launch_counts():
    w = bi.WORKLOADS[1]
    band = bi.make_workload(w)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(band).to(dev)
    d = torch.empty(w.n, dtype=torch.float32, device=dev)
    e = torch.empty(w.n - 1, dtype=torch.float32, device=dev)
    h = bb.bb_create(w.n, w.bw, bb.BB_F32)
    try:
        bb.bb_set_param(h, bb.BB_PARAM_TIMING, 1)
        s = torch.cuda.current_stream(dev)
        bb.bb_reduce(h, x, band.shape[1], w.tw, d, e, s)
        assert bb.bb_status_sync(h, s) == bb.BB_OK
        npass = bb.bb_num_passes(w.bw, w.tw)
        assert bb.bb_last_num_passes(h) == npass
        assert bb.bb_last_launches(h) == npass + 2
        ms = [bb.bb_last_pass_ms(h, i) for i in range(npass)]
        assert all(m > 0 for m in ms)
    finally:
        bb.bb_destroy(h)
