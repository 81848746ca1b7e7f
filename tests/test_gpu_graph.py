"""Device-resident generation counter: calls captured in a CUDA graph.

With the pad's device_generation option on, each call takes its generation
from a counter in device memory that the previous call's last block
advanced, so a graph of captured calls replays with fresh flag values every
time.  The inputs change between replays and alternate inside a replay: a
call that passed a barrier on a stale flag would hand back the other input
set's (or the previous replay's) data."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GuardedOutputs, RankBuffers, assert_bitwise, to_device

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


def _call(rr, algo, pad, W, N, src, bufs, outs, stream):
    if algo.startswith("allgather"):
        rr.rr_allgather(src.ptrs, outs, W, N, "bf16", pad, stream)
        return
    copy = algo.endswith("_copy")
    fn = rr.rr_allreduce_oneshot if algo.startswith("oneshot") else rr.rr_allreduce_twoshot
    if copy:
        fn(src.ptrs, bufs.ptrs, outs, W, N, "bf16", 1, pad, stream)
    else:
        fn(None, src.ptrs, outs, W, N, "bf16", 0, pad, stream)


def _want(algo, ins):
    if algo.startswith("allgather"):
        return oracle.allgather_rank_major(ins, "bf16")
    return oracle.allreduce(ins, "bf16")


def test_device_generation_on_a_stream_and_back(rr):
    W, N = 8, 100_003
    pad = rr.rr_signal_pad_create(W)
    sets = [workloads.rank_buffers(W, N, "bf16", "uniform", seed_base=8000 + 10 * k) for k in range(2)]
    srcs = []
    for s in sets:
        rb = RankBuffers(W, N, "bf16")
        rb.fill(s)
        srcs.append(rb)
    staging = RankBuffers(W, N, "bf16")
    stream = torch.cuda.current_stream()
    algos = ["oneshot", "oneshot_copy", "twoshot", "twoshot_copy", "twoshot_pull", "allgather"]
    calls = 0
    for mode in (0, 1, 0, 1):
        pad.set_option("device_generation", mode)
        g0 = pad.get_option("generation")
        for i, algo in enumerate(algos):
            k = (i + mode) % 2
            pad.set_option("twoshot_mode", 1 if algo == "twoshot_pull" else 0)
            n_out = W * N if algo == "allgather" else N
            outs = GuardedOutputs(W, n_out, "bf16")
            _call(rr, algo, pad, W, N, srcs[k], staging, outs.ptrs, stream)
            pad.status(stream)
            want = _want(algo, sets[k])
            for r in range(W):
                assert_bitwise(outs.host(r), want, f"mode {mode} {algo} output {r}")
            calls += 1
        pad.set_option("twoshot_mode", 0)
        assert pad.get_option("generation") == g0 + len(algos)
    pad.close()


@pytest.mark.parametrize("algo", ["oneshot", "oneshot_copy", "twoshot", "twoshot_copy", "twoshot_pull",
                                  "allgather"])
def test_graph_replays_stay_correct(rr, algo):
    W, N, K, replays = 8, 65536 + 5, 6, 4
    pad = rr.rr_signal_pad_create(W)
    pad.set_option("device_generation", 1)
    pad.set_option("twoshot_mode", 1 if algo == "twoshot_pull" else 0)
    # host input sets: replay j, call i uses set (j, i % 2)
    hsets = [[workloads.rank_buffers(W, N, "bf16", "uniform", seed_base=9000 + 100 * j + 10 * k)
              for k in range(2)] for j in range(replays)]
    srcs = [RankBuffers(W, N, "bf16") for _ in range(2)]
    staging = RankBuffers(W, N, "bf16")
    n_out = W * N if algo == "allgather" else N
    outs = [GuardedOutputs(W, n_out, "bf16") for _ in range(K)]
    stream = torch.cuda.Stream()
    for k in range(2):
        srcs[k].fill(hsets[0][k])
    torch.cuda.synchronize()
    # a call outside the capture fills the library's per-kernel caches
    with torch.cuda.stream(stream):
        _call(rr, algo, pad, W, N, srcs[0], staging, outs[0].ptrs, stream)
    pad.status(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        cs = torch.cuda.current_stream()
        for i in range(K):
            _call(rr, algo, pad, W, N, srcs[i % 2], staging, outs[i].ptrs, cs)
    for j in range(replays):
        for k in range(2):
            srcs[k].fill(hsets[j][k])
        torch.cuda.synchronize()
        for o in outs:
            o.poison()
        graph.replay()
        torch.cuda.synchronize()
        pad.status(stream)
        for i in range(K):
            want = _want(algo, hsets[j][i % 2])
            for r in range(W):
                assert_bitwise(outs[i].host(r), want, f"replay {j} call {i} output {r}")
            outs[i].check_guards()
    # a fresh pad: one call before the capture, then K calls per replay
    assert pad.get_option("generation") == 1 + K * replays
    pad.close()


@pytest.mark.parametrize("engine", [1, 2])
def test_graph_replays_param_contiguous_and_list(rr, engine):
    """Param-contiguous and list-output gathers captured together in one
    graph (alternating), replayed with new shards each time."""
    W, replays = 8, 3
    splits = [20_000, 5, 0, 45_539]
    S = sum(splits)
    pad = rr.rr_signal_pad_create(W)
    pad.set_option("device_generation", 1)
    pad.set_option("gather_engine", engine)
    src = RankBuffers(W, S, "bf16")
    pc_out = [GuardedOutputs(W, W * S, "bf16", materialise=(0, 7)) for _ in range(2)]
    lists = [[GuardedOutputs(W, S, "bf16") for _ in range(2)] for _ in range(2)]  # [call][row q in (2, 5)]

    def rows(i):
        return [lists[i][0].ptrs if q == 2 else lists[i][1].ptrs if q == 5 else None for q in range(W)]

    stream = torch.cuda.Stream()
    src.fill(workloads.rank_buffers(W, S, "bf16", "bits", seed_base=9500))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        rr.rr_allgather_param_contiguous(src.ptrs, pc_out[0].ptrs, W, splits, "bf16", pad, stream)
        rr.rr_allgather_list(src.ptrs, rows(0), W, S, "bf16", pad, stream)
    pad.status(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        cs = torch.cuda.current_stream()
        for i in range(2):
            rr.rr_allgather_param_contiguous(src.ptrs, pc_out[i].ptrs, W, splits, "bf16", pad, cs)
            rr.rr_allgather_list(src.ptrs, rows(i), W, S, "bf16", pad, cs)
    for j in range(replays):
        ins = workloads.rank_buffers(W, S, "bf16", "bits", seed_base=9600 + 10 * j)
        src.fill(ins)
        for o in pc_out + [x for row in lists for x in row]:
            o.poison()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        pad.status(stream)
        want_pc = oracle.allgather_param_contiguous(ins, splits, "bf16")
        for i in range(2):
            for q in (0, 7):
                assert_bitwise(pc_out[i].host(q), want_pc, f"replay {j} call {i} param-contiguous output {q}")
            for row in lists[i]:
                for r in range(W):
                    assert_bitwise(row.host(r), ins[r], f"replay {j} call {i} list entry {r}")
                row.check_guards()
            pc_out[i].check_guards()
    pad.close()
