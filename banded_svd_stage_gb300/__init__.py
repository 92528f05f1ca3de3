"""Python binding of libbb.so, the GB300 band -> bidiagonal reduction.

Thin ctypes marshalling over the C ABI declared in include/bb.h; every step of
the reduction runs in the library's CUDA kernels.  Function names and
argument order are those of the C ABI.  Device buffers may be passed as raw
integer addresses or as CUDA tensors (their ``data_ptr()`` is used); streams as
raw ``cudaStream_t`` integers or ``torch.cuda.Stream`` objects.

There is no fallback: if libbb.so has not been built (``build()``), importing
this package succeeds but every call raises ``BBError``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbb.so")

BB_F32, BB_F64, BB_F16 = 0, 1, 2
BB_OK, BB_ERR_INVALID_ARG, BB_ERR_LDAB, BB_ERR_DTYPE, BB_ERR_CUDA, BB_ERR_TIMEOUT, BB_ERR_NOMEM = range(7)
STATUS_NAMES = {0: "BB_OK", 1: "BB_ERR_INVALID_ARG", 2: "BB_ERR_LDAB", 3: "BB_ERR_DTYPE",
                4: "BB_ERR_CUDA", 5: "BB_ERR_TIMEOUT", 6: "BB_ERR_NOMEM"}
(BB_PARAM_SCHEDULER, BB_PARAM_TPB, BB_PARAM_MAX_CTAS, BB_PARAM_WAIT_BUDGET_MS, BB_PARAM_PASS_LO,
 BB_PARAM_PASS_HI, BB_PARAM_STALL_SWEEP, BB_PARAM_TIMING, BB_PARAM_GROUP_SIZE, BB_PARAM_RECORD) = range(10)
BB_ERR_INTERNAL = 7
STATUS_NAMES[7] = "BB_ERR_INTERNAL"
# scheduler values
SCHED_AUTO, SCHED_CYCLE, SCHED_FLAGS, SCHED_GROUP, SCHED_CYCLE_GRAPH = 0, 1, 2, 3, 4


class BBError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def build(force: bool = False) -> str:
    """Compile libbb.so in-tree (nvcc, sm_103a)."""
    from . import buildlib
    return buildlib.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded libbb.so (raises BBError if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise BBError(BB_ERR_CUDA, f"CUDA library not built: {LIB_PATH} is missing "
                                       "(run banded_svd_stage_gb300.build())")
        L = ctypes.CDLL(LIB_PATH)
        i64, p, ci, cd = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        sig = {
            "bb_create": ([i64, i64, ci], p),
            "bb_reduce": ([p, p, i64, i64, p, p, p], ci),
            "bb_reduce_host": ([p, p, i64, i64, p, p, p], ci),
            "bb_destroy": ([p], None),
            "bb_required_ldab": ([i64, i64], i64),
            "bb_status_sync": ([p, p], ci),
            "bb_set_param": ([p, ci, i64], ci),
            "bb_get_param": ([p, ci], i64),
            "bb_num_passes": ([i64, i64], i64),
            "bb_pass_info": ([i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)], ci),
            "bb_model_bytes": ([i64, i64, i64, i64, i64], cd),
            "bb_model_steps": ([i64, i64, i64, i64], i64),
            "bb_last_launches": ([p], i64),
            "bb_last_num_passes": ([p], i64),
            "bb_last_pass_ms": ([p, i64, ctypes.POINTER(cd)], ci),
            "bb_last_error": ([], ctypes.c_char_p),
            "bb_reduce_noalloc": ([p, i64, i64, i64, i64, ci, p, p, p], ci),
            "bb_last_pass_kernel": ([p, i64], i64),
            "bb_last_pass_group": ([p, i64], i64),
            "bb_singular_values": ([ci, i64, p, p, p, p], ci),
            "bb_singular_values_lanes": ([ci, i64, p, p, p, i64, p], ci),
            "bb_group_plan": ([i64, i64, i64, i64, i64, i64] + [ctypes.POINTER(i64)] * 4, ci),
            "bb_sym_group_plan": ([i64, i64, i64, i64, i64, i64] + [ctypes.POINTER(i64)] * 4, ci),
            "bb_sym_reduce": ([p, p, i64, i64, p, p, p], ci),
            "bb_dense_to_band_workspace": ([i64, i64, ci], i64),
            "bb_dense_to_band": ([ci, i64, i64, p, i64, p, i64, p], ci),
            "bb_pack_band": ([ci, i64, i64, i64, p, i64, p, i64, p], ci),
            "bb_sym_required_ldab": ([i64, i64], i64),
            "bb_back_transform": ([p, p, i64, p, i64, p], ci),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):  # numpy array (host buffers)
        return int(x.ctypes.data)
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s) -> int | None:
    if s is None or isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError(f"not a stream: {type(s)}")


def _check(st: int) -> None:
    if st != BB_OK:
        raise BBError(st, bb_last_error())


def bb_last_error() -> str:
    return lib().bb_last_error().decode()


def bb_create(n: int, bw: int, dtype: int) -> int:
    h = lib().bb_create(n, bw, dtype)
    if not h:
        raise BBError(BB_ERR_INVALID_ARG, bb_last_error())
    return h


def bb_destroy(h) -> None:
    lib().bb_destroy(h)


def bb_reduce(h, band, ldab: int, tw: int, d_out, e_out, stream=None) -> None:
    _check(lib().bb_reduce(h, _addr(band), ldab, tw, _addr(d_out), _addr(e_out), _stream(stream)))


def bb_reduce_host(h, band_host, ldab: int, tw: int, d_host, e_host, stream=None) -> None:
    _check(lib().bb_reduce_host(h, _addr(band_host), ldab, tw, _addr(d_host), _addr(e_host),
                                _stream(stream)))


def bb_status_sync(h, stream=None) -> int:
    """Synchronize and return the device status (0 or BB_ERR_TIMEOUT); does not raise."""
    return int(lib().bb_status_sync(h, _stream(stream)))


def bb_set_param(h, param: int, value: int) -> None:
    _check(lib().bb_set_param(h, param, value))


def bb_get_param(h, param: int) -> int:
    return int(lib().bb_get_param(h, param))


def bb_required_ldab(bw: int, tw: int) -> int:
    return int(lib().bb_required_ldab(bw, tw))


def bb_num_passes(bw: int, tw: int) -> int:
    return int(lib().bb_num_passes(bw, tw))


def bb_pass_info(bw: int, tw: int, i: int):
    b, t = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().bb_pass_info(bw, tw, i, ctypes.byref(b), ctypes.byref(t)))
    return b.value, t.value


def bb_model_bytes(n: int, bw: int, tw: int, elem_bytes: int, pass_index: int = -1) -> float:
    return float(lib().bb_model_bytes(n, bw, tw, elem_bytes, pass_index))


def bb_model_steps(n: int, bw: int, tw: int, pass_index: int = -1) -> int:
    return int(lib().bb_model_steps(n, bw, tw, pass_index))


def bb_last_launches(h) -> int:
    return int(lib().bb_last_launches(h))


def bb_last_num_passes(h) -> int:
    return int(lib().bb_last_num_passes(h))


def bb_last_pass_kernel(h, i: int) -> int:
    return int(lib().bb_last_pass_kernel(h, i))


def bb_last_pass_group(h, i: int) -> int:
    return int(lib().bb_last_pass_group(h, i))


def bb_last_pass_ms(h, i: int) -> float:
    ms = ctypes.c_double()
    _check(lib().bb_last_pass_ms(h, i, ctypes.byref(ms)))
    return ms.value


def bb_reduce_noalloc(band, n: int, bw: int, ldab: int, tw: int, dtype: int, d_out, e_out,
                      stream=None) -> None:
    """Reduction with no device allocation (fixed in-library scratch, n <= 65536);
    synchronizes the stream before returning."""
    _check(lib().bb_reduce_noalloc(_addr(band), n, bw, ldab, tw, dtype, _addr(d_out), _addr(e_out),
                                   _stream(stream)))


def bb_singular_values_lanes(dtype: int, n: int, d, e, sigma_out, lanes: int, stream=None) -> None:
    """bb_singular_values with the lanes per value fixed (0: the default rule)."""
    _check(lib().bb_singular_values_lanes(dtype, n, _addr(d), _addr(e), _addr(sigma_out), lanes, _stream(stream)))


def bb_group_plan(n: int, bw: int, tw: int, elem_bytes: int, pass_index: int, group_size: int = 0):
    """(g, nslot, ahead, lds) of the group kernel's plan for one pass; g = 0
    when the group kernel cannot take it.  Host-only."""
    vals = [ctypes.c_int64() for _ in range(4)]
    _check(lib().bb_group_plan(n, bw, tw, elem_bytes, pass_index, group_size, *[ctypes.byref(v) for v in vals]))
    return tuple(v.value for v in vals)


def bb_sym_group_plan(n: int, bw: int, tw: int, elem_bytes: int, pass_index: int, group_size: int = 0):
    """(g, nslot, ahead, lds) of the symmetric chase's group-kernel plan for
    one pass; g = 0 when its group kernel cannot take it.  Host-only."""
    vals = [ctypes.c_int64() for _ in range(4)]
    _check(lib().bb_sym_group_plan(n, bw, tw, elem_bytes, pass_index, group_size,
                                   *[ctypes.byref(v) for v in vals]))
    return tuple(v.value for v in vals)


def bb_singular_values(dtype: int, n: int, d, e, sigma_out, stream=None) -> None:
    """Singular values of the bidiagonal (d, e), descending, into sigma_out
    (device buffers; asynchronous on `stream`)."""
    _check(lib().bb_singular_values(dtype, n, _addr(d), _addr(e), _addr(sigma_out), _stream(stream)))


def bb_sym_reduce(h, band, ldab: int, tw: int, d, e, stream=None) -> None:
    """Symmetric band (lower band storage, device) -> tridiagonal (d, e)."""
    _check(lib().bb_sym_reduce(h, _addr(band), ldab, tw, _addr(d), _addr(e), _stream(stream)))


def bb_dense_to_band_workspace(n: int, bw: int, dtype: int) -> int:
    """Bytes of device workspace bb_dense_to_band needs (-1: invalid)."""
    return lib().bb_dense_to_band_workspace(n, bw, dtype)


def bb_dense_to_band(dtype: int, n: int, bw: int, a, lda: int, workspace, workspace_bytes: int, stream=None) -> None:
    """Stage 1: dense column-major a (device) -> upper band of bandwidth bw, in place."""
    _check(lib().bb_dense_to_band(dtype, n, bw, _addr(a), lda, _addr(workspace), workspace_bytes, _stream(stream)))


def bb_pack_band(dtype: int, n: int, bw: int, tw: int, a, lda: int, band, ldab: int, stream=None) -> None:
    """The upper band of dense column-major a (device) into bb_reduce's band storage."""
    _check(lib().bb_pack_band(dtype, n, bw, tw, _addr(a), lda, _addr(band), ldab, _stream(stream)))


def bb_sym_required_ldab(bw: int, tw: int) -> int:
    return lib().bb_sym_required_ldab(bw, tw)
def bb_back_transform(h, U, ldu: int, V, ldv: int, stream=None) -> None:
    """U, V (device, column-major n x n; either may be None) of the last
    reduction recorded with BB_PARAM_RECORD, so that A = U B V^T."""
    _check(lib().bb_back_transform(h, _addr(U), ldu, _addr(V), ldv, _stream(stream)))


def dtype_code(dtype) -> int:
    """BB_F32 / BB_F64 / BB_F16 from a torch or numpy dtype or the strings
    'f32' / 'f64' / 'f16'."""
    s = str(dtype)
    if s in ("f32", "float32", "torch.float32"):
        return BB_F32
    if s in ("f64", "float64", "torch.float64"):
        return BB_F64
    if s in ("f16", "float16", "torch.float16"):
        return BB_F16
    raise ValueError(f"unsupported dtype {dtype}")
