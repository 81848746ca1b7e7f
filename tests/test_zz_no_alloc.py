"""The allocation-free one-shot allreduce (rr_allreduce_oneshot_noalloc).

Some callers cannot call cudaMalloc: engine plugins whose enqueue runs inside
a memory budget fixed ahead of time, frameworks that own all device memory
through their own pool, latency-critical code that cannot afford the device
synchronisation an allocation brings.  They cannot make a signal pad, so this
entry point keeps its pad in a static device array inside the library.

The test calls it through the C ABI twice in a row (the second call reuses
the array the first one left behind, with new inputs) and compares each
output bit for bit with the pad-based rr_allreduce_oneshot on the same
inputs: the tolerance of every allreduce test here is bit-exactness.  It is
meant to pass alone in a fresh process (the first call on the device does
the one-time set-up) and after every other test; its file name makes pytest
collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import GuardedOutputs, RankBuffers, assert_bitwise

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    from allgather_rr_allreduce_gb300 import build
    build.build()
    import allgather_rr_allreduce_gb300 as rr
    l = ctypes.CDLL(rr.LIB_PATH)
    f = l.rr_allreduce_oneshot_noalloc
    vp = ctypes.POINTER(ctypes.c_void_p)
    f.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    l.rr_last_error.restype = ctypes.c_char_p
    return l, rr


@pytest.mark.parametrize("copy_mode", [0, 1])
def test_noalloc_matches_pad_oneshot_on_two_calls(lib, copy_mode):
    l, rr = lib
    W, N, dtype = 8, (1 << 20) + 5, "bf16"
    stream = torch.cuda.current_stream().cuda_stream
    pad = rr.rr_signal_pad_create(W)
    for call in range(2):
        ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=6100 + 10 * call + copy_mode)
        bufs_a, bufs_b = RankBuffers(W, N, dtype), RankBuffers(W, N, dtype)
        src = RankBuffers(W, N, dtype)
        if copy_mode:
            src.fill(ins)
        else:
            bufs_a.fill(ins)
            bufs_b.fill(ins)
        ref = GuardedOutputs(W, N, dtype)
        got = GuardedOutputs(W, N, dtype, materialise=(0, 3))
        rr.rr_allreduce_oneshot(src.ptrs if copy_mode else None, bufs_a.ptrs, ref.ptrs, W, N, dtype,
                                copy_mode, pad, stream)
        st = l.rr_allreduce_oneshot_noalloc(rr.pointer_array(src.ptrs) if copy_mode else None,
                                            rr.pointer_array(bufs_b.ptrs), rr.pointer_array(got.ptrs),
                                            W, N, rr.RR_BF16, copy_mode, stream)
        assert st == rr.RR_OK, l.rr_last_error()
        pad.status(stream)
        torch.cuda.synchronize()
        for r in (0, 3):
            assert_bitwise(got.host(r), ref.host(0), f"call {call}, output {r}")
        got.check_guards()
    pad.close()


def test_noalloc_rejects_more_ranks_than_its_pad_holds(lib):
    l, rr = lib
    W, N = 9, 64
    bufs = RankBuffers(W, N, "fp32")
    outs = GuardedOutputs(W, N, "fp32", materialise=(0,))
    st = l.rr_allreduce_oneshot_noalloc(None, rr.pointer_array(bufs.ptrs), rr.pointer_array(outs.ptrs),
                                        W, N, rr.RR_FP32, 0, None)
    assert st == rr.RR_ERR_INVALID_ARG
    assert b"1..8" in l.rr_last_error()
