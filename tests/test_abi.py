"""CPU checks of the C ABI: the library loads, exports every entry point
include/rr.h declares, and rejects bad arguments before touching CUDA.  The
work partition the kernels use is compiled for the host and checked for
exact coverage.  No compute call is made here."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rr.h")


@pytest.fixture(scope="module")
def rr():
    from allgather_rr_allreduce_gb300 import build
    build.build()
    import allgather_rr_allreduce_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rr_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("rr_allreduce_oneshot", "rr_allreduce_twoshot", "rr_allgather",
                 "rr_allgather_param_contiguous", "rr_allgather_list", "rr_signal_pad_create"):
        assert must in names


def test_library_exports_every_declared_function(rr):
    lib = ctypes.CDLL(rr.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(rr):
    lib = rr.lib()
    for code, name in [(0, b"RR_OK"), (3, b"RR_ERR_ALIGNMENT"), (7, b"RR_ERR_TIMEOUT")]:
        assert lib.rr_status_string(code) == name


def _raw_status(fn, *args):
    return fn(*args)


def test_host_argument_checks_without_a_gpu(rr):
    lib = rr.lib()
    h = ctypes.c_void_p()
    assert lib.rr_signal_pad_create(0, 0, 0, ctypes.byref(h)) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_signal_pad_create(17, 0, 0, ctypes.byref(h)) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_signal_pad_create(4, -1, 0, ctypes.byref(h)) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_signal_pad_create(4, 0, 0, None) == rr.RR_ERR_INVALID_ARG
    arr = rr.pointer_array([16, 32])
    # NULL pad is rejected first, for every entry point
    assert lib.rr_allreduce_oneshot(None, arr, arr, 2, 8, 0, 0, None, None) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_allreduce_twoshot(None, arr, arr, 2, 8, 0, 0, None, None) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_allgather(arr, arr, 2, 8, 0, None, None) == rr.RR_ERR_INVALID_ARG
    sp = (ctypes.c_int64 * 1)(8)
    assert lib.rr_allgather_param_contiguous(arr, arr, 2, sp, 1, 0, None, None) == rr.RR_ERR_INVALID_ARG
    lists = rr.pointer_array([16, 32, 48, 64])
    assert lib.rr_allgather_list(arr, lists, 2, 8, 0, None, None) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_signal_pad_status(None, None) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_signal_pad_set_option(None, 0, 1) == rr.RR_ERR_INVALID_ARG
    assert lib.rr_signal_pad_destroy(None) == rr.RR_OK
    assert b"pad" in lib.rr_last_error() or lib.rr_last_error() == b""


def test_pad_creation_fails_cleanly_or_succeeds(rr):
    """Without a GPU the CUDA runtime call fails and the status says so; with
    one, the pad is made and destroyed."""
    lib = rr.lib()
    h = ctypes.c_void_p()
    st = lib.rr_signal_pad_create(2, 4, 0, ctypes.byref(h))
    assert st in (rr.RR_OK, rr.RR_ERR_CUDA)
    if st == rr.RR_OK:
        assert lib.rr_signal_pad_destroy(h) == rr.RR_OK
    else:
        assert h.value is None
        assert lib.rr_last_error()


def test_binding_raises_rrerror(rr):
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather([16, 32], [16, 32], 2, 8, "bf16", None, 0)
    assert e.value.status == rr.RR_ERR_INVALID_ARG


def test_partition_covers_exactly_once(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    cuda_inc = None
    for cand in ("/usr/local/cuda/include", os.path.join(os.environ.get("CUDA_HOME", ""), "include")):
        if cand and os.path.exists(os.path.join(cand, "cuda_runtime.h")):
            cuda_inc = cand
            break
    if cuda_inc is None:
        pytest.skip("CUDA headers not found")
    exe = tmp_path / "partition_check"
    src = os.path.join(ROOT, "tests", "native", "partition_check.cpp")
    subprocess.run([gxx, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "allgather_rr_allreduce_gb300", "csrc"), "-I", cuda_inc,
                    src, "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
