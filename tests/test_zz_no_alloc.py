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
from gpu_helpers import TOL, fro_of_band, gpu_reduce

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
