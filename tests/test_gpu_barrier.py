"""The signal-pad barrier: generation flags, bounded waits, sticky timeouts.

Failure is made on purpose only through the pad's fault-injection option:
one rank never emits one barrier's flags, so its peers' waits run out after
a short limit (20 ms here), the kernel records RR_ERR_TIMEOUT in the pad and
returns, and the context stays usable.  Nothing here faults or traps the GPU.
"""
import pytest
import torch

import oracle
import workloads
from gpu_util import GuardedOutputs, RankBuffers, assert_bitwise

pytestmark = pytest.mark.gpu

SHORT_NS = 20_000_000


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    from allgather_rr_allreduce_gb300 import build
    build.build()
    import allgather_rr_allreduce_gb300 as m
    m.lib()
    return m


def _inputs(W, N):
    ins = workloads.rank_buffers(W, N, "bf16", "uniform", seed_base=77)
    return ins, oracle.allreduce(ins, "bf16")


def _call(rr, algo, pad, W, N, ins, copy_mode):
    bufs = RankBuffers(W, N, "bf16")
    src = RankBuffers(W, N, "bf16")
    (src if copy_mode else bufs).fill(ins)
    outs = GuardedOutputs(W, N, "bf16")
    fn = rr.rr_allreduce_oneshot if algo == "oneshot" else rr.rr_allreduce_twoshot
    pad.set_option("twoshot_mode", 1 if algo == "twoshot_pull" else 0)
    fn(src.ptrs if copy_mode else None, bufs.ptrs, outs.ptrs, W, N, "bf16", copy_mode, pad)
    pad.set_option("twoshot_mode", 0)
    return outs


CASES = [
    ("oneshot", 0, 1, "ARRIVE"), ("oneshot", 1, 2, "STAGE"), ("oneshot", 0, 3, "END"),
    ("twoshot_pull", 0, 0, "MID"), ("twoshot_pull", 1, 1, "STAGE"), ("twoshot_pull", 1, 2, "END"),
]


@pytest.mark.parametrize("algo,copy_mode,rank,barrier", CASES)
def test_skipped_flag_times_out_and_recovers(rr, algo, copy_mode, rank, barrier):
    W, N = 4, 50_000
    ins, want = _inputs(W, N)
    bar = getattr(rr, f"RR_BARRIER_{barrier}")
    pad = rr.rr_signal_pad_create(W, 0, SHORT_NS)
    pad.set_option("inject_skip", rank * 4 + bar)
    outs = _call(rr, algo, pad, W, N, ins, copy_mode)
    with pytest.raises(rr.RRError) as e:
        pad.status()
    assert e.value.status == rr.RR_ERR_TIMEOUT
    info = pad.timeout_info()
    assert info["barrier"] == bar
    assert info["generation"] == pad.get_option("generation")
    outs.check_guards()
    # the status was cleared by reading it; the pad and the GPU work again
    pad.set_option("inject_skip", -1)
    outs = _call(rr, algo, pad, W, N, ins, copy_mode)
    pad.status()
    for r in range(W):
        assert_bitwise(outs.host(r), want, f"after recovery, output {r}")
    pad.close()


def test_tma_oneshot_times_out_and_recovers(rr):
    W, N = 4, 200_000
    ins, want = _inputs(W, N)
    pad = rr.rr_signal_pad_create(W, 0, SHORT_NS)
    pad.set_option("reduce_engine", 2)
    for rank, barrier in ((2, "ARRIVE"), (1, "END")):
        pad.set_option("inject_skip", rank * 4 + getattr(rr, f"RR_BARRIER_{barrier}"))
        _call(rr, "oneshot", pad, W, N, ins, 0)
        with pytest.raises(rr.RRError) as e:
            pad.status()
        assert e.value.status == rr.RR_ERR_TIMEOUT
        pad.set_option("inject_skip", -1)
        outs = _call(rr, "oneshot", pad, W, N, ins, 0)
        pad.status()
        for r in range(W):
            assert_bitwise(outs.host(r), want)
    pad.close()


@pytest.mark.parametrize("copy_mode,barrier", [(0, "END"), (1, "STAGE"), (0, "ARRIVE")])
def test_twoshot_push_times_out_and_recovers(rr, copy_mode, barrier):
    W, N = 4, 60_000
    ins, want = _inputs(W, N)
    pad = rr.rr_signal_pad_create(W, 0, SHORT_NS)
    pad.set_option("twoshot_mode", 2)
    pad.set_option("inject_skip", 3 * 4 + getattr(rr, f"RR_BARRIER_{barrier}"))
    _call(rr, "twoshot", pad, W, N, ins, copy_mode)
    with pytest.raises(rr.RRError) as e:
        pad.status()
    assert e.value.status == rr.RR_ERR_TIMEOUT
    pad.set_option("inject_skip", -1)
    outs = _call(rr, "twoshot", pad, W, N, ins, copy_mode)
    pad.status()
    for r in range(W):
        assert_bitwise(outs.host(r), want)
    pad.close()


@pytest.mark.parametrize("algo,barrier", [("oneshot", "STAGE"), ("twoshot", "STAGE"), ("oneshot", "END")])
def test_staged_copy_mode_times_out_and_recovers(rr, algo, barrier):
    W, N = 4, 300_000
    ins, want = _inputs(W, N)
    pad = rr.rr_signal_pad_create(W, 0, SHORT_NS)
    pad.set_option("reduce_engine", 2)
    pad.set_option("inject_skip", 1 * 4 + getattr(rr, f"RR_BARRIER_{barrier}"))
    _call(rr, algo, pad, W, N, ins, 1)
    with pytest.raises(rr.RRError) as e:
        pad.status()
    assert e.value.status == rr.RR_ERR_TIMEOUT
    pad.set_option("inject_skip", -1)
    outs = _call(rr, algo, pad, W, N, ins, 1)
    pad.status()
    for r in range(W):
        assert_bitwise(outs.host(r), want)
    pad.close()


def test_pending_timeout_blocks_later_calls(rr):
    """While a timeout is recorded and not yet read, later calls on the pad
    stop at their first barrier and leave their outputs untouched."""
    W, N = 2, 4096
    ins, want = _inputs(W, N)
    pad = rr.rr_signal_pad_create(W, 0, SHORT_NS)
    pad.set_option("inject_skip", 1 * 4 + rr.RR_BARRIER_ARRIVE)
    _call(rr, "oneshot", pad, W, N, ins, 0)
    pad.set_option("inject_skip", -1)
    outs = _call(rr, "oneshot", pad, W, N, ins, 0)
    torch.cuda.synchronize()
    untouched = outs.host(0)
    assert (untouched.view("u1") == 0xA5).all()
    with pytest.raises(rr.RRError):
        pad.status()
    outs = _call(rr, "oneshot", pad, W, N, ins, 0)
    pad.status()
    assert_bitwise(outs.host(0), want)
    pad.close()


def test_gather_timeout(rr):
    W, N = 3, 10_000
    pad = rr.rr_signal_pad_create(W, 0, SHORT_NS)
    ins = workloads.rank_buffers(W, N, "int32", "int", seed_base=1)
    bufs = RankBuffers(W, N, "int32")
    bufs.fill(ins)
    for engine in (1, 2):
        pad.set_option("gather_engine", engine)
        pad.set_option("inject_skip", 2 * 4 + rr.RR_BARRIER_END)
        outs = GuardedOutputs(W, W * N, "int32")
        rr.rr_allgather(bufs.ptrs, outs.ptrs, W, N, "int32", pad)
        with pytest.raises(rr.RRError) as e:
            pad.status()
        assert e.value.status == rr.RR_ERR_TIMEOUT
        assert pad.timeout_info()["barrier"] == rr.RR_BARRIER_END
        pad.set_option("inject_skip", -1)
        rr.rr_allgather(bufs.ptrs, outs.ptrs, W, N, "int32", pad)
        pad.status()
        assert_bitwise(outs.host(0), oracle.allgather_rank_major(ins, "int32"))
    pad.close()


def test_generation_advances_and_keeps_parity(rr):
    W, N = 2, 1024
    ins, want = _inputs(W, N)
    pad = rr.rr_signal_pad_create(W)
    g0 = pad.get_option("generation")
    for k in range(6):
        outs = _call(rr, ("twoshot", "twoshot_pull", "oneshot")[k % 3], pad, W, N, ins, k % 2)
        assert pad.get_option("generation") == g0 + k + 1
    pad.status()
    assert_bitwise(outs.host(1), want)
    pad.close()


def test_pads_on_two_streams(rr):
    """Concurrent collectives on two streams, each with its own pad."""
    W, N = 4, 1 << 18
    ins, want = _inputs(W, N)
    pads = [rr.rr_signal_pad_create(W) for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    bufs = RankBuffers(W, N, "bf16")
    bufs.fill(ins)
    outs = [GuardedOutputs(W, N, "bf16") for _ in range(2)]
    torch.cuda.synchronize()
    for it in range(20):
        for k in range(2):
            fn = rr.rr_allreduce_oneshot if k == 0 else rr.rr_allreduce_twoshot
            fn(None, bufs.ptrs, outs[k].ptrs, W, N, "bf16", 0, pads[k], streams[k])
    for k in range(2):
        pads[k].status(streams[k])
        for r in range(W):
            assert_bitwise(outs[k].host(r), want)
        pads[k].close()
