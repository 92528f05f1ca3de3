"""bb_reduce_noalloc: the entry point for callers that cannot allocate device
memory (their memory belongs to a pool or another allocator, or cudaMalloc /
cudaFree, which can synchronize the device, are not acceptable where they
call).  It takes its scratch from a fixed array inside the library, so these
tests check that it computes the same d and e as bb_reduce, on two calls in a
row (the second call finds the first call's leftovers in that array), and
that sizes beyond its fixed scratch are refused.

This file is named to be collected last, so that a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import band_inputs as bi
import banded_svd_stage_gb300 as bb
import oracle
from gpu_helpers import TOL, fro_of_band, gpu_reduce
from test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("idx", [1, 0])
def test_noalloc_matches_bb_reduce_on_two_calls(idx):
    w = bi.WORKLOADS[idx]
    band = bi.make_workload(w)
    d_ref, e_ref = gpu_reduce(band, w.n, w.bw, w.tw, w.dtype, 0)
    fro = fro_of_band(band)
    dev = torch.device("cuda:0")
    tdt = torch.float32 if w.dtype == "f32" else torch.float64
    for _ in range(2):
        x = torch.from_numpy(band).to(dev)
        d = torch.full((w.n,), float("nan"), dtype=tdt, device=dev)
        e = torch.full((w.n - 1,), float("nan"), dtype=tdt, device=dev)
        bb.bb_reduce_noalloc(x, w.n, w.bw, band.shape[1], w.tw, bb.dtype_code(w.dtype), d, e,
                             torch.cuda.current_stream(dev))
        dn, en = d.cpu().numpy(), e.cpu().numpy()
        err = max(np.abs(dn.astype(np.float64) - d_ref).max(), np.abs(en.astype(np.float64) - e_ref).max())
        assert err <= TOL[w.dtype] * fro, f"no-alloc result differs from bb_reduce by {err / fro:.3e}"


def run_noalloc(band, n, bw, tw, dt):
    dev = torch.device("cuda:0")
    tdt = torch.float32 if dt == "f32" else torch.float64
    x = torch.from_numpy(band).to(dev)
    d = torch.full((n,), float("nan"), dtype=tdt, device=dev)
    e = torch.full((n - 1,), float("nan"), dtype=tdt, device=dev)
    bb.bb_reduce_noalloc(x, n, bw, band.shape[1], tw, bb.dtype_code(dt), d, e, torch.cuda.current_stream(dev))
    return d.cpu().numpy(), e.cpu().numpy()


# (n, bw, tw, dtype, ldab):
#   * the n = 4096 workload with its column stride padded to 144 bytes, so
#     that its passes run on the group kernel (watermarks in the fixed array);
#   * a column stride of 264 bytes (ldab = bw + 2 tw + 2), not a multiple of
#     16: every pass falls back to the flag kernel, in place;
#   * the n = 32768 recipe at n = 2111 with a 16-byte column stride: the wide
#     passes run on the flag kernel and the narrow ones on the group kernel.
LAYOUTS = [(4096, 16, 8, "f32", 36), (1000, 40, 12, "f32", 66), (2111, 256, 32, "f32", 324)]


@pytest.mark.parametrize("n,bw,tw,dt,ldab", LAYOUTS)
def test_noalloc_kernel_paths_match_oracle_and_bb_reduce(n, bw, tw, dt, ldab):
    w = bi.WORKLOADS[1] if n == 4096 else bi.WORKLOADS[4]
    band = bi.make_band(n, bw, tw, dt, w.dist, False, seed=n + ldab, ldab=ldab)
    inner = np.ascontiguousarray(band[:, : bw + 2 * tw + 1])
    d_ref, e_ref = oracle.bidiagonal(inner, n, bw, tw)
    d_dev, e_dev = gpu_reduce(band, n, bw, tw, dt, 0)
    for _ in range(2):
        d, e = run_noalloc(band, n, bw, tw, dt)
        # the same kernels as bb_reduce in the same launch shapes: equal bitwise
        assert np.array_equal(d, d_dev) and np.array_equal(e, e_dev)
        assert_parity(d, e, d_ref, e_ref, inner, n, bw, tw, dt)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    n, bw, tw = 65537, 2, 1
    dev = torch.device("cuda:0")
    x = torch.zeros((n, bw + 2 * tw + 1), dtype=torch.float32, device=dev)
    d = torch.empty(n, dtype=torch.float32, device=dev)
    e = torch.empty(n - 1, dtype=torch.float32, device=dev)
    with pytest.raises(bb.BBError) as ex:
        bb.bb_reduce_noalloc(x, n, bw, x.shape[1], tw, bb.BB_F32, d, e)
    assert ex.value.status == bb.BB_ERR_INVALID_ARG
    assert "65536" in str(ex.value)
