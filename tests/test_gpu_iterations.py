"""GPU tests of the in-launch iteration mode (pad options debug_iterations and
debug_skew_ns): several complete calls run inside one launch, so that the
barriers separating one call from the next are crossed with no kernel
boundary in between, as they are between GPUs.  Ranks are put out of step
by a per-rank sleep before every iteration.  Every iteration works on its
own seeded inputs and writes its own output slice, which must equal the
oracle's result for that iteration bit for bit.  With copy_mode on, every
iteration stages into the same rank buffers: a rank that restaged before a
peer had finished reading its previous iteration would corrupt that peer's
result (the write-after-read case the end barrier exists for)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import CANARY, GUARD, assert_bitwise

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    from allgather_rr_allreduce_gb300 import build
    build.build()
    import allgather_rr_allreduce_gb300 as m
    m.lib()
    return m


def stride_of(nbytes):
    return (nbytes + 15) // 16 * 16


class Slices:
    """W device buffers (None where not materialised), each holding `iters`
    slices of `nbytes` at a 16-byte-rounded stride, with canary bytes before,
    between and after the slices."""

    def __init__(self, W, iters, nbytes, materialise=None):
        self.W, self.iters, self.nbytes = W, iters, nbytes
        self.stride = stride_of(nbytes)
        size = 2 * GUARD + self.stride * (iters - 1) + nbytes
        keep = range(W) if materialise is None else materialise
        self.bufs = [torch.full((size,), CANARY, dtype=torch.uint8, device="cuda") if r in keep else None
                     for r in range(W)]
        self.ptrs = [None if t is None else t.data_ptr() + GUARD for t in self.bufs]

    def view(self, r, k):
        o = GUARD + k * self.stride
        return self.bufs[r][o:o + self.nbytes]

    def fill(self, k, arrays):
        for r, a in enumerate(arrays):
            if self.bufs[r] is not None and a.size:
                self.view(r, k).copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8)).cuda())

    def host(self, r, k, dtype):
        return self.view(r, k).cpu().numpy().view(workloads.STORAGE[dtype])

    def check_guards(self):
        for r, t in enumerate(self.bufs):
            if t is None:
                continue
            a = t.cpu().numpy()
            used = np.zeros(a.size, dtype=bool)
            for k in range(self.iters):
                o = GUARD + k * self.stride
                used[o:o + self.nbytes] = True
            assert (a[~used] == CANARY).all(), f"buffer {r}: a byte outside the slices was written"


def iteration_inputs(W, N, iters, seed):
    return [workloads.rank_buffers(W, N, "bf16", "normal", seed_base=seed + 100 * k) for k in range(iters)]


def make_pad(rr, W, iters, skew_ns, round_bytes=0):
    pad = rr.rr_signal_pad_create(W)
    pad.set_option("debug_iterations", iters)
    pad.set_option("debug_skew_ns", skew_ns)
    pad.set_option("round_bytes", round_bytes)
    return pad


AR_CASES = [
    # W, N, iterations, skew ns, round bytes (0 = automatic)
    (2, 4096, 4, 0, 0),
    (8, 8195, 6, 20_000, 0),
    (8, 300_001, 5, 30_000, 4096),
    (5, 77_777, 4, 20_000, 2048),
    (16, 2048, 3, 5_000, 0),
]


@pytest.mark.parametrize("algo", ["oneshot", "twoshot"])
@pytest.mark.parametrize("copy_mode", [0, 1])
@pytest.mark.parametrize("W,N,iters,skew,rb", AR_CASES, ids=[f"W{c[0]}_N{c[1]}_it{c[2]}_sk{c[3]}" for c in AR_CASES])
def test_iterations_allreduce(rr, algo, copy_mode, W, N, iters, skew, rb):
    nbytes = N * 2
    ins = iteration_inputs(W, N, iters, seed=7000 + W * 10 + copy_mode)
    pad = make_pad(rr, W, iters, skew, rb)
    g0 = pad.get_option("generation")
    outs = Slices(W, iters, nbytes)
    if copy_mode:
        src = Slices(W, iters, nbytes)
        for k in range(iters):
            src.fill(k, ins[k])
        regs = Slices(W, 1, nbytes)
        fn = getattr(rr, f"rr_allreduce_{algo}")
        fn(src.ptrs, regs.ptrs, outs.ptrs, W, N, "bf16", 1, pad)
    else:
        regs = Slices(W, iters, nbytes)
        for k in range(iters):
            regs.fill(k, ins[k])
        fn = getattr(rr, f"rr_allreduce_{algo}")
        fn(None, regs.ptrs, outs.ptrs, W, N, "bf16", 0, pad)
    pad.status()
    assert pad.get_option("generation") - g0 == iters
    for k in range(iters):
        want = oracle.allreduce(ins[k], "bf16")
        for q in range(W):
            assert_bitwise(outs.host(q, k, "bf16"), want, f"iteration {k} output {q}")
    if copy_mode:
        for r in range(W):
            assert_bitwise(regs.host(r, 0, "bf16"), ins[-1][r], f"rank buffer {r} after the last iteration")
    outs.check_guards()
    regs.check_guards()
    pad.close()


def test_iterations_oneshot_subset_of_outputs(rr):
    W, N, iters = 8, 65_536 + 24, 4
    ins = iteration_inputs(W, N, iters, seed=9100)
    pad = make_pad(rr, W, iters, 25_000)
    regs = Slices(W, iters, 2 * N)
    for k in range(iters):
        regs.fill(k, ins[k])
    outs = Slices(W, iters, 2 * N, materialise=(1, 6))
    rr.rr_allreduce_oneshot(None, regs.ptrs, outs.ptrs, W, N, "bf16", 0, pad)
    pad.status()
    for k in range(iters):
        want = oracle.allreduce(ins[k], "bf16")
        for q in (1, 6):
            assert_bitwise(outs.host(q, k, "bf16"), want, f"iteration {k} output {q}")
    outs.check_guards()
    pad.close()


@pytest.mark.parametrize("engine", [1, 2])
@pytest.mark.parametrize("kind", ["rank_major", "param_contiguous", "list"])
@pytest.mark.parametrize("skew", [0, 20_000])
def test_iterations_allgather(rr, engine, kind, skew):
    W, iters, dtype = 8, 5, "fp16"
    splits = [4096, 7, 512, 0, 1023, 8 * 300 + 3] if kind == "param_contiguous" else [20_001]
    S = sum(splits)
    eb = 2
    ins = [workloads.rank_buffers(W, S, dtype, "bits", seed_base=8000 + 50 * k) for k in range(iters)]
    pad = make_pad(rr, W, iters, skew)
    pad.set_option("gather_engine", engine)
    src = Slices(W, iters, S * eb)
    for k in range(iters):
        src.fill(k, ins[k])
    if kind == "list":
        # output list q entry r: one Slices per (q, r) for q in {0, 3}
        lists = {q: [Slices(1, iters, S * eb) for _ in range(W)] for q in (0, 3)}
        rows = [[lists[q][r].ptrs[0] for r in range(W)] if q in lists else None for q in range(W)]
        rr.rr_allgather_list(src.ptrs, rows, W, S, dtype, pad)
        pad.status()
        for k in range(iters):
            for q in lists:
                for r in range(W):
                    assert_bitwise(lists[q][r].host(0, k, dtype), ins[k][r], f"iteration {k} list {q} entry {r}")
        for q in lists:
            for t in lists[q]:
                t.check_guards()
    else:
        outs = Slices(W, iters, W * S * eb, materialise=(0, 3))
        if kind == "rank_major":
            rr.rr_allgather(src.ptrs, outs.ptrs, W, S, dtype, pad)
        else:
            rr.rr_allgather_param_contiguous(src.ptrs, outs.ptrs, W, splits, dtype, pad)
        pad.status()
        for k in range(iters):
            want = (oracle.allgather_rank_major(ins[k], dtype) if kind == "rank_major"
                    else oracle.allgather_param_contiguous(ins[k], splits, dtype))
            for q in (0, 3):
                assert_bitwise(outs.host(q, k, dtype), want, f"iteration {k} output {q}")
        outs.check_guards()
    pad.close()


def test_iterations_timeout_stops_and_recovers(rr):
    """Rank 2 never emits its END flags: the first iteration's END wait runs
    out, later iterations do not start, and the pad works again afterwards."""
    W, N, iters = 4, 4096, 4
    ins = iteration_inputs(W, N, iters, seed=9300)
    pad = make_pad(rr, W, iters, 0)
    pad.set_option("timeout_ns", 50_000_000)
    regs = Slices(W, iters, 2 * N)
    for k in range(iters):
        regs.fill(k, ins[k])
    outs = Slices(W, iters, 2 * N)
    pad.set_option("inject_skip", 2 * 4 + rr.RR_BARRIER_END)
    rr.rr_allreduce_twoshot(None, regs.ptrs, outs.ptrs, W, N, "bf16", 0, pad)
    with pytest.raises(rr.RRError) as e:
        pad.status()
    assert e.value.status == rr.RR_ERR_TIMEOUT
    info = pad.timeout_info()
    assert info["barrier"] == rr.RR_BARRIER_END
    # later iterations never ran: their output slices still hold the canary
    for k in range(1, iters):
        for q in range(W):
            assert (outs.view(q, k).cpu().numpy() == CANARY).all(), f"iteration {k} ran after the timeout"
    pad.set_option("inject_skip", -1)
    rr.rr_allreduce_twoshot(None, regs.ptrs, outs.ptrs, W, N, "bf16", 0, pad)
    pad.status()
    for k in range(iters):
        want = oracle.allreduce(ins[k], "bf16")
        for q in range(W):
            assert_bitwise(outs.host(q, k, "bf16"), want, f"iteration {k} output {q} after recovery")
    pad.close()


def test_iterations_then_plain_calls(rr):
    """Plain calls after an iterated call on the same pad take fresh
    generations (the iterated call reserved one per iteration)."""
    W, N = 8, 40_000
    ins = iteration_inputs(W, N, 3, seed=9400)
    pad = make_pad(rr, W, 3, 10_000)
    regs = Slices(W, 3, 2 * N)
    for k in range(3):
        regs.fill(k, ins[k])
    outs = Slices(W, 3, 2 * N)
    rr.rr_allreduce_oneshot(None, regs.ptrs, outs.ptrs, W, N, "bf16", 0, pad)
    pad.set_option("debug_iterations", 1)
    pad.set_option("debug_skew_ns", 0)
    for k in (2, 0, 1, 2):
        outs1 = Slices(W, 1, 2 * N)
        rr.rr_allreduce_twoshot(None, [p + k * regs.stride for p in regs.ptrs], outs1.ptrs, W, N, "bf16", 0, pad)
        pad.status()
        want = oracle.allreduce(ins[k], "bf16")
        for q in range(W):
            assert_bitwise(outs1.host(q, 0, "bf16"), want, f"plain call on iteration {k}'s data, output {q}")
    for k in range(3):
        want = oracle.allreduce(ins[k], "bf16")
        assert_bitwise(outs.host(0, k, "bf16"), want, f"iteration {k}")
    pad.close()


def test_iterations_argument_errors(rr):
    W, N = 4, 1024
    pad = make_pad(rr, W, 3, 0)
    regs = Slices(W, 3, 2 * N)
    outs = Slices(W, 3, 2 * N)
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, regs.ptrs, outs.ptrs, W, N, "fp16", 0, pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    pad.set_option("twoshot_mode", 1)
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_twoshot(None, regs.ptrs, outs.ptrs, W, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    pad.set_option("twoshot_mode", 0)
    pad.set_option("gather_engine", 3)
    gout = Slices(W, 3, W * 2 * N)
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather(regs.ptrs, gout.ptrs, W, N, "bf16", pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    pad.set_option("gather_engine", 0)
    # rank buffers one slice apart overlap once three iterations are asked for
    packed = torch.empty(W * 2 * N + 64, dtype=torch.uint8, device="cuda")
    close = [packed.data_ptr() + r * 2 * N for r in range(W)]
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, close, outs.ptrs, W, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    pad.set_option("device_generation", 1)
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, regs.ptrs, outs.ptrs, W, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    pad.set_option("device_generation", 0)
    with pytest.raises(rr.RRError):
        pad.set_option("debug_iterations", 0)
    with pytest.raises(rr.RRError):
        pad.set_option("debug_skew_ns", 2_000_000)
    pad.status()
    pad.close()
