"""C-ABI checks that need no GPU: the library loads, exports every function
include/bb.h declares, and its host-side planner and traffic model agree with
an enumeration written here from the definition of the windows."""
import os
import re

import pytest

import banded_svd_stage_gb300 as bb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bb.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(bb_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    bb.build()
    return bb.lib()


def test_header_declares_the_core_entry_points():
    names = declared_functions()
    for core in ("bb_create", "bb_reduce", "bb_destroy"):
        assert core in names


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(bb.BBError):
        bb.bb_create(100, 8, bb.BB_F32)
    assert bb.bb_last_error()


def test_null_handle_and_bad_params(lib):
    assert lib.bb_reduce(None, None, 10, 1, None, None, None) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_set_param(None, 0, 0) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_status_sync(None, None) == bb.BB_ERR_INVALID_ARG
    bb.bb_destroy(None)


def _plan(bw, tw):
    out, b = [], bw
    while b > 1:
        t = min(tw, b - 1)
        out.append((b, t))
        b -= t
    return out


def _enumerate(n, bw, tw, s):
    """Steps and modeled bytes from the windows: right block rows p..ce x cols
    c..ce, left block rows c..ce x cols c..cend, each element read + written."""
    steps, byts = 0, 0
    for (b, t) in _plan(bw, tw):
        bp = b - t
        for r in range(0, n - bp - 1):
            k = 0
            while True:
                c = r + bp + k * b
                if c + 1 > n - 1:
                    break
                p = r if k == 0 else c - b
                ce = min(c + t, n - 1)
                cend = min(ce + b, n - 1)
                w = ce - c + 1
                steps += 1
                byts += 2 * s * ((ce - p + 1) * w + w * (cend - c + 1))
                k += 1
    return steps, byts


@pytest.mark.parametrize("n,bw,tw", [(2, 1, 1), (10, 3, 1), (64, 16, 8), (100, 17, 5), (257, 64, 16),
                                     (300, 40, 39)])
def test_planner_and_traffic_model(lib, n, bw, tw):
    plan = _plan(bw, tw)
    assert bb.bb_num_passes(bw, tw) == len(plan)
    for i, bt in enumerate(plan):
        assert bb.bb_pass_info(bw, tw, i) == bt
    steps, byts = _enumerate(n, bw, tw, 4)
    assert bb.bb_model_steps(n, bw, tw) == steps
    assert bb.bb_model_bytes(n, bw, tw, 4) == pytest.approx(byts, rel=1e-12)
    per_pass = sum(bb.bb_model_bytes(n, bw, tw, 4, i) for i in range(len(plan)))
    assert per_pass == pytest.approx(byts, rel=1e-12)


def test_required_ldab(lib):
    assert bb.bb_required_ldab(256, 32) == 321
    assert bb.bb_required_ldab(8, 7) == 23


def test_singular_values_argument_errors_need_no_gpu(lib):
    # the entry point validates its arguments before any CUDA call
    fake = 0x1000  # never dereferenced: every call below is rejected first
    assert lib.bb_singular_values(bb.BB_F32, 0, fake, fake, fake, None) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_singular_values(bb.BB_F32, -5, fake, fake, fake, None) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_singular_values(bb.BB_F64, (1 << 29) + 1, fake, fake, fake, None) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_singular_values(bb.BB_F32, 4, None, fake, fake, None) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_singular_values(bb.BB_F32, 4, fake, None, fake, None) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_singular_values(bb.BB_F32, 4, fake, fake, None, None) == bb.BB_ERR_INVALID_ARG
    assert lib.bb_singular_values(7, 4, fake, fake, fake, None) == bb.BB_ERR_DTYPE
    assert "bb_singular_values" in bb.bb_last_error()


def test_pass_count_is_arithmetic_and_bounded(lib):
    # the plan is never materialised for these: a huge bandwidth costs nothing
    assert bb.bb_num_passes((1 << 30) - 1, 1) == (1 << 30) - 2
    assert bb.bb_num_passes((1 << 30) + 1, 1) == 0          # beyond any accepted order
    assert bb.bb_pass_info((1 << 30) - 1, 1, (1 << 30) - 3) == (2, 1)
    for bw in range(0, 70):
        for tw in range(1, 12):
            assert bb.bb_num_passes(bw, tw) == len(_plan(bw, tw))
    assert bb.bb_num_passes(16, 0) == 0 and bb.bb_num_passes(-3, 2) == 0


def test_group_plan_rejects_inconsistent_shapes(lib):
    for args in ((100, 100, 8, 4, 0), (100, 16, 0, 4, 0), (100, 16, 16, 4, 0), (100, 16, 8, 3, 0),
                 (0, 0, 1, 4, 0), (100, 16, 8, 4, -1)):
        with pytest.raises(bb.BBError):
            bb.bb_group_plan(*args)


def test_group_plan_of_binary16_storage(lib):
    # elem_bytes 2: binary16 columns (rows rounded to 8 elements = 16 bytes),
    # float scratch; reflectors of more than 33 elements have no group kernel
    g, nslot, ahead, lds = bb.bb_group_plan(4096, 16, 8, 2, 0)
    assert g == 13 and lds % 8 == 0 and lds >= 2 * 8 + 16 + 1
    assert bb.bb_group_plan(4096, 16, 8, 4, 0)[1] == nslot
    assert bb.bb_group_plan(4096, 128, 64, 2, 0)[0] == 0


def test_singular_value_lanes_are_validated_without_a_gpu(lib):
    fake = 0x1000  # never dereferenced: rejected before any CUDA call
    for lanes in (-1, 3, 6, 33, 64):
        assert lib.bb_singular_values_lanes(bb.BB_F64, 8, fake, fake, fake, lanes, None) == bb.BB_ERR_INVALID_ARG


def test_header_is_c99_and_links_against_the_library(lib, tmp_path):
    # the boundary is a C ABI: a C99 translation unit includes the header with
    # every warning an error, takes the address of every declared function,
    # and links against libbb.so (nothing runs: that would need a GPU)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    names = declared_functions()
    src = ["#include <stdio.h>", '#include "bb.h"', "int main(void) {", "    void* fns[] = {"]
    src += [f"        (void*){n}," for n in names]
    src += ["    };", "    unsigned long long s = 0;",
            "    for (unsigned i = 0; i < sizeof fns / sizeof fns[0]; ++i) s += (unsigned long long)fns[i] != 0;",
            '    printf("%llu\\n", s);', "    return 0;", "}"]
    c = tmp_path / "uses_bb.c"
    c.write_text("\n".join(src) + "\n")
    libdir = os.path.dirname(bb.LIB_PATH)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), str(c), "-o", str(tmp_path / "uses_bb"),
           "-L", libdir, "-l:libbb.so", f"-Wl,-rpath-link,{libdir}",
           "-Wl,--unresolved-symbols=ignore-in-shared-libs"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_back_transform_rejects_a_null_handle(lib):
    assert lib.bb_back_transform(None, None, 1, None, 1, None) == bb.BB_ERR_INVALID_ARG


def test_noalloc_argument_errors_need_no_gpu(lib):
    # bb_reduce_noalloc checks every argument before its first CUDA call
    fake = 0x1000  # never dereferenced: every call below is rejected first
    f = lib.bb_reduce_noalloc
    assert f(fake, 100, 8, 23, 7, 7, fake, fake, None) == bb.BB_ERR_DTYPE           # dtype
    assert f(fake, 0, 0, 2, 1, bb.BB_F32, fake, fake, None) == bb.BB_ERR_INVALID_ARG  # n < 1
    assert f(fake, 10, 10, 31, 1, bb.BB_F32, fake, fake, None) == bb.BB_ERR_INVALID_ARG  # bw >= n
    assert f(fake, 65537, 8, 23, 7, bb.BB_F32, fake, fake, None) == bb.BB_ERR_INVALID_ARG  # beyond scratch
    assert f(fake, 100, 8, 23, 8, bb.BB_F32, fake, fake, None) == bb.BB_ERR_INVALID_ARG  # tw > bw - 1
    assert f(fake, 100, 8, 22, 7, bb.BB_F32, fake, fake, None) == bb.BB_ERR_LDAB          # ldab too small
    assert f(None, 100, 8, 23, 7, bb.BB_F32, fake, fake, None) == bb.BB_ERR_INVALID_ARG  # null band
    assert f(fake, 100, 8, 23, 7, bb.BB_F32, fake, None, None) == bb.BB_ERR_INVALID_ARG  # null e
    # a band too wide for the flag kernel's shared-memory tile
    assert f(fake, 20000, 9000, 9001 + 2 * 64, 64, bb.BB_F64, fake, fake, None) == bb.BB_ERR_INVALID_ARG
