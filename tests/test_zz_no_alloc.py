"""The allocation-free one-shot allreduce (rr_allreduce_oneshot_noalloc).

Some callers cannot call cudaMalloc: engine plugins whose enqueue runs inside
a memory budget fixed ahead of time, frameworks that own all device memory
through their own pool, latency-critical code that cannot afford the device
synchronisation an allocation brings.  They cannot make a signal pad, so this
entry point keeps its pad in a static device array inside the library.

The tests call it through the C ABI.  Two calls in a row (the second reuses
the array the first one left behind, with new inputs) are compared bit for
bit with the pad-based rr_allreduce_oneshot on the same inputs and with the
CPU oracle: the tolerance of every allreduce test here is bit-exactness.  A
sequence of calls that changes the world size, the dtype, the ragged length
and copy_mode is compared with the oracle call by call (flags left in the
array by a call with another W must never let a later call pass a barrier
early).  A second call leaves the device's free memory unchanged, a call
made while its stream is being captured into a CUDA graph is refused, and
the allocation-free status read reports no timeout.  The file is meant to
pass alone in a fresh process (the first call on the device does the
one-time set-up) and after every other test; its name makes pytest collect
it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GuardedOutputs, RankBuffers, assert_bitwise

pytestmark = pytest.mark.gpu

DTYPE_CODE = {"bf16": 0, "fp16": 1, "fp32": 2, "int32": 3}


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
    l.rr_allreduce_oneshot_noalloc_status.argtypes = [ctypes.c_void_p]
    l.rr_allreduce_oneshot_noalloc_status.restype = ctypes.c_int
    l.rr_last_error.restype = ctypes.c_char_p
    oracle.lib()
    return l, rr


def _call(l, rr, src, bufs, outs, W, N, dtype, copy_mode, stream):
    return l.rr_allreduce_oneshot_noalloc(rr.pointer_array(src.ptrs) if copy_mode else None,
                                          rr.pointer_array(bufs.ptrs), rr.pointer_array(outs.ptrs),
                                          W, N, DTYPE_CODE[dtype], copy_mode, stream)


@pytest.mark.parametrize("copy_mode", [0, 1])
def test_noalloc_matches_pad_oneshot_and_oracle_on_two_calls(lib, copy_mode):
    l, rr = lib
    W, N, dtype = 8, (1 << 20) + 5, "bf16"
    stream = torch.cuda.current_stream().cuda_stream
    pad = rr.rr_signal_pad_create(W)
    for call in range(2):
        ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=6100 + 10 * call + copy_mode)
        want = oracle.allreduce(ins, dtype)
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
        st = _call(l, rr, src, bufs_b, got, W, N, dtype, copy_mode, stream)
        assert st == rr.RR_OK, l.rr_last_error()
        pad.status(stream)
        assert l.rr_allreduce_oneshot_noalloc_status(stream) == rr.RR_OK, l.rr_last_error()
        torch.cuda.synchronize()
        for r in (0, 3):
            assert_bitwise(got.host(r), ref.host(0), f"call {call}, output {r} against the pad-based one-shot")
            assert_bitwise(got.host(r), want, f"call {call}, output {r} against the oracle")
        got.check_guards()
    pad.close()


# W changes between calls (the array is re-indexed for each call's W), with
# ragged lengths, every dtype and both copy modes.
SEQUENCE = [(8, "bf16", 1_000_003, 0), (2, "fp32", 77_777, 1), (5, "int32", 300_001, 0),
            (8, "fp16", 65_539, 1), (1, "bf16", 4097, 0), (8, "fp32", 2_000_017, 0),
            (3, "bf16", 9, 1), (8, "int32", 1_048_579, 1)]


def test_noalloc_sequence_of_world_sizes_matches_oracle(lib):
    l, rr = lib
    stream = torch.cuda.current_stream().cuda_stream
    for k, (W, dtype, N, copy_mode) in enumerate(SEQUENCE):
        dist = "int" if dtype == "int32" else "normal"
        ins = workloads.rank_buffers(W, N, dtype, dist, seed_base=6500 + 31 * k)
        want = oracle.allreduce(ins, dtype)
        bufs, src = RankBuffers(W, N, dtype), RankBuffers(W, N, dtype)
        (src if copy_mode else bufs).fill(ins)
        keep = tuple(range(W)) if k % 2 else (W - 1,)
        outs = GuardedOutputs(W, N, dtype, materialise=keep)
        st = _call(l, rr, src, bufs, outs, W, N, dtype, copy_mode, stream)
        assert st == rr.RR_OK, l.rr_last_error()
        assert l.rr_allreduce_oneshot_noalloc_status(stream) == rr.RR_OK, l.rr_last_error()
        for r in keep:
            assert_bitwise(outs.host(r), want, f"call {k} (W={W}, {dtype}, N={N}, copy_mode={copy_mode}) output {r}")
        outs.check_guards()
        if copy_mode:
            for r in range(W):
                assert_bitwise(bufs.host(r), ins[r], f"call {k}: staged buffer {r}")


def test_noalloc_second_call_allocates_nothing(lib):
    l, rr = lib
    W, N, dtype = 8, (1 << 22) + 3, "bf16"
    stream = torch.cuda.current_stream().cuda_stream
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=6900)
    bufs, src = RankBuffers(W, N, dtype), RankBuffers(W, N, dtype)
    bufs.fill(ins)
    src.fill(ins)
    outs = GuardedOutputs(W, N, dtype, materialise=(0,))
    for copy_mode in (0, 1):
        assert _call(l, rr, src, bufs, outs, W, N, dtype, copy_mode, stream) == rr.RR_OK, l.rr_last_error()
        torch.cuda.synchronize()
        free_before, _ = torch.cuda.mem_get_info()
        assert _call(l, rr, src, bufs, outs, W, N, dtype, copy_mode, stream) == rr.RR_OK, l.rr_last_error()
        assert l.rr_allreduce_oneshot_noalloc_status(stream) == rr.RR_OK
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
        assert free_after == free_before, f"copy_mode={copy_mode}: free device memory changed by {free_before - free_after} bytes"
    assert_bitwise(outs.host(0), oracle.allreduce(ins, dtype))


def test_noalloc_refuses_a_call_during_stream_capture(lib):
    l, rr = lib
    W, N, dtype = 2, 4096, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "uniform", seed_base=6950)
    bufs = RankBuffers(W, N, dtype)
    bufs.fill(ins)
    outs = GuardedOutputs(W, N, dtype, materialise=(0,))
    side = torch.cuda.Stream()
    x = torch.zeros(16, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        x.add_(1)
        st = _call(l, rr, bufs, bufs, outs, W, N, dtype, 0, side.cuda_stream)
    assert st == rr.RR_ERR_INVALID_ARG
    assert b"captur" in l.rr_last_error()
    graph.replay()
    torch.cuda.synchronize()
    # outside the capture the same call runs
    st = _call(l, rr, bufs, bufs, outs, W, N, dtype, 0, side.cuda_stream)
    assert st == rr.RR_OK, l.rr_last_error()
    assert l.rr_allreduce_oneshot_noalloc_status(side.cuda_stream) == rr.RR_OK
    assert_bitwise(outs.host(0), oracle.allreduce(ins, dtype))


def test_noalloc_rejects_more_ranks_than_its_pad_holds(lib):
    l, rr = lib
    W, N = 9, 64
    bufs = RankBuffers(W, N, "fp32")
    outs = GuardedOutputs(W, N, "fp32", materialise=(0,))
    st = l.rr_allreduce_oneshot_noalloc(None, rr.pointer_array(bufs.ptrs), rr.pointer_array(outs.ptrs),
                                        W, N, rr.RR_FP32, 0, None)
    assert st == rr.RR_ERR_INVALID_ARG
    assert b"1..8" in l.rr_last_error()
