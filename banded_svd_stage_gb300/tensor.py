"""Torch-tensor conveniences over the C ABI (allocation and marshalling only).

``Reducer`` owns one library handle and reduces CUDA tensors in band storage
(shape (n, ldab), row j = column j of the matrix, as produced by
``band_inputs``).  Torch supplies device memory and the current stream; all
arithmetic runs in libbb.so.
"""
from __future__ import annotations

import torch

from . import (BB_PARAM_SCHEDULER, BB_PARAM_TIMING, bb_create, bb_destroy, bb_last_num_passes,
               bb_last_pass_ms, bb_reduce, bb_set_param, bb_status_sync, BBError, dtype_code)


class Reducer:
    def __init__(self, n: int, bw: int, dtype: torch.dtype, scheduler: int = 0, **params):
        self.n, self.bw, self.dtype = n, bw, dtype
        self.h = bb_create(n, bw, dtype_code(dtype))
        bb_set_param(self.h, BB_PARAM_SCHEDULER, scheduler)
        for k, v in params.items():
            bb_set_param(self.h, k, v)

    def close(self):
        if self.h:
            bb_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reduce_(self, band: torch.Tensor, tw: int, d: torch.Tensor | None = None,
                e: torch.Tensor | None = None, stream=None):
        """Reduce band (CUDA, (n, ldab), contiguous) in place; returns (d, e)."""
        if not (band.is_cuda and band.is_contiguous() and band.dtype == self.dtype):
            raise ValueError("band must be a contiguous CUDA tensor of the reducer's dtype")
        if band.dim() != 2 or band.shape[0] != self.n:
            raise ValueError(f"band must have shape ({self.n}, ldab)")
        if d is None:
            d = torch.empty(self.n, dtype=self.dtype, device=band.device)
        if e is None:
            e = torch.empty(max(self.n - 1, 1), dtype=self.dtype, device=band.device)
        s = stream if stream is not None else torch.cuda.current_stream(band.device)
        bb_reduce(self.h, band, band.shape[1], tw, d, e, s)
        return d, e[: max(self.n - 1, 0)]

    def sync_status(self, stream=None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream()
        return bb_status_sync(self.h, s)

    def check(self, stream=None) -> None:
        st = self.sync_status(stream)
        if st != 0:
            raise BBError(st, "device-side failure")

    def enable_timing(self, on: bool = True) -> None:
        bb_set_param(self.h, BB_PARAM_TIMING, 1 if on else 0)

    def pass_ms(self):
        return [bb_last_pass_ms(self.h, i) for i in range(bb_last_num_passes(self.h))]

    def pass_kernels(self):
        """[(kernel, group size), ...] of the last reduction: 1 per-cycle, 2 flags, 3 group,
        4 per-cycle launches replayed from a CUDA graph."""
        from . import bb_last_pass_group, bb_last_pass_kernel
        return [(bb_last_pass_kernel(self.h, i), bb_last_pass_group(self.h, i))
                for i in range(bb_last_num_passes(self.h))]
