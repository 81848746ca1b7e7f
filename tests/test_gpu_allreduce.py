"""GPU parity: one-shot and two-shot allreduce through the C ABI against the
CPU oracle, element by element, bit for bit (binary32 rank-order rule).

Sizes span several blocks' chunks and a ragged tail; the W=8, 2^24-element
bf16 case is the launch configuration the benchmark times, compared in full.
"""
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


_pads = {}


def pad_for(rr, W):
    if W not in _pads:
        _pads[W] = rr.rr_signal_pad_create(W)
    return _pads[W]


def dist_for(dtype):
    return "int" if dtype == "int32" else "normal"


def run_allreduce(rr, algo, W, N, dtype, copy_mode, ins, materialise=None, layout="packed",
                  blocks_per_rank=0):
    pad = pad_for(rr, W)
    pad.set_option("blocks_per_rank", blocks_per_rank)
    bufs = RankBuffers(W, N, dtype, layout=layout)
    src = None
    if copy_mode:
        src = RankBuffers(W, N, dtype, layout=layout)
        src.fill(ins)
        # stale contents in the registered buffers: a missed staging shows
        bufs.fill([np.full_like(a, 0x3C) for a in ins])
    else:
        bufs.fill(ins)
    outs = GuardedOutputs(W, N, dtype, materialise=materialise)
    fn = rr.rr_allreduce_oneshot if algo == "oneshot" else rr.rr_allreduce_twoshot
    if algo == "twoshot_pull":
        pad.set_option("twoshot_mode", 1)
    try:
        fn(src.ptrs if copy_mode else None, bufs.ptrs, outs.ptrs, W, N, dtype, copy_mode, pad)
        pad.status()
    finally:
        pad.set_option("twoshot_mode", 0)
        pad.set_option("blocks_per_rank", 0)
    return bufs, src, outs


SHAPES = [(2, 4096), (1, 100), (2, 4099), (3, 12345), (4, 1), (5, 8 * 16 * 33 + 5), (8, 65536 + 7),
          (16, 10000), (7, 3)]


@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull"])
@pytest.mark.parametrize("copy_mode", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", SHAPES, ids=[f"W{w}_N{n}" for w, n in SHAPES])
def test_allreduce_matches_oracle(rr, algo, copy_mode, dtype, W, N):
    ins = workloads.rank_buffers(W, N, dtype, dist_for(dtype), seed_base=100 * W + N % 97)
    want = oracle.allreduce(ins, dtype)
    bufs, src, outs = run_allreduce(rr, algo, W, N, dtype, copy_mode, ins)
    for r in range(W):
        assert_bitwise(outs.host(r), want, f"{algo} output {r}")
    outs.check_guards()
    for r in range(W):
        assert_bitwise(bufs.host(r), ins[r], f"rank buffer {r} after the call")
        if copy_mode:
            assert_bitwise(src.host(r), ins[r], f"input {r} after the call")


def test_small_workload_uniform(rr):
    """W=2 bf16, 4096 elements per rank, uniform[-1, 1]."""
    cfg = workloads.SMALL
    ins = workloads.rank_buffers(cfg["W"], cfg["N"], "bf16", "uniform", cfg["seed_base"])
    want = oracle.allreduce(ins, "bf16")
    for algo in ("oneshot", "twoshot"):
        for copy_mode in (0, 1):
            _, _, outs = run_allreduce(rr, algo, 2, cfg["N"], "bf16", copy_mode, ins)
            for r in range(2):
                assert_bitwise(outs.host(r), want, f"{algo} copy={copy_mode} rank {r}")


@pytest.mark.parametrize("materialise", [(0,), (1, 3), (0, 1, 2, 3, 4), (7,)])
@pytest.mark.parametrize("copy_mode", [0, 1])
def test_oneshot_subset_of_outputs(rr, materialise, copy_mode):
    W, N, dtype = 8, 3 * 4096 * 16 + 3, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=7)
    want = oracle.allreduce(ins, dtype)
    _, _, outs = run_allreduce(rr, "oneshot", W, N, dtype, copy_mode, ins, materialise=materialise)
    for r in materialise:
        assert_bitwise(outs.host(r), want, f"output {r}")
    outs.check_guards()


@pytest.mark.parametrize("blocks", [1, 2, 7, 32])
@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull"])
def test_fixed_blocks_per_rank(rr, blocks, algo):
    """The result does not depend on how many blocks each rank runs,
    including the single-block degenerate case."""
    W, N, dtype = 4, 200_003, "fp16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=11)
    want = oracle.allreduce(ins, dtype)
    for copy_mode in (0, 1):
        _, _, outs = run_allreduce(rr, algo, W, N, dtype, copy_mode, ins, blocks_per_rank=blocks)
        for r in range(W):
            assert_bitwise(outs.host(r), want, f"{algo} blocks={blocks} output {r}")


@pytest.mark.parametrize("round_bytes", [256, 4096, 1 << 20])
@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull"])
@pytest.mark.parametrize("copy_mode", [0, 1])
def test_round_sizes(rr, round_bytes, algo, copy_mode):
    """The pipelined chunk gives the same bits with 16-vector rounds (many
    rounds per block), the default, and one round per block."""
    W, N, dtype = 8, 3 * (1 << 17) + 11, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=21)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("round_bytes", round_bytes)
    try:
        _, _, outs = run_allreduce(rr, algo, W, N, dtype, copy_mode, ins,
                                   materialise=None if algo != "oneshot" else (0, 6))
    finally:
        pad.set_option("round_bytes", 0)
    for r in (range(W) if algo != "oneshot" else (0, 6)):
        assert_bitwise(outs.host(r), want, f"{algo} round_bytes={round_bytes} output {r}")
    outs.check_guards()


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", SHAPES + [(8, (1 << 20) + 3)], ids=[f"W{w}_N{n}" for w, n in SHAPES + [(8, (1 << 20) + 3)]])
def test_oneshot_tma_engine_matches_oracle(rr, dtype, W, N):
    """The one-shot with bulk-copy (TMA) loads, every output kept and rank 0
    only: same bits as the oracle."""
    ins = workloads.rank_buffers(W, N, dtype, dist_for(dtype), seed_base=300 * W + N % 89)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 2)
    try:
        for materialise in (None, (0,)):
            _, _, outs = run_allreduce(rr, "oneshot", W, N, dtype, 0, ins, materialise=materialise)
            assert pad.get_option("last_engine") == 2
            for r in (range(W) if materialise is None else materialise):
                assert_bitwise(outs.host(r), want, f"tma engine output {r}")
            outs.check_guards()
    finally:
        pad.set_option("reduce_engine", 0)


@pytest.mark.parametrize("blocks", [1, 3, 16])
def test_oneshot_tma_engine_fixed_blocks(rr, blocks):
    W, N, dtype = 4, 300_001, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=19)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 2)
    try:
        _, _, outs = run_allreduce(rr, "oneshot", W, N, dtype, 0, ins, materialise=(1, 2),
                                   blocks_per_rank=blocks)
    finally:
        pad.set_option("reduce_engine", 0)
    for r in (1, 2):
        assert_bitwise(outs.host(r), want)


@pytest.mark.parametrize("copy_mode", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", SHAPES + [(8, (1 << 20) + 3)], ids=[f"W{w}_N{n}" for w, n in SHAPES + [(8, (1 << 20) + 3)]])
def test_twoshot_push_mode_matches_oracle(rr, copy_mode, dtype, W, N):
    """Two-shot whose allgather is a broadcast by each chunk's owner."""
    ins = workloads.rank_buffers(W, N, dtype, dist_for(dtype), seed_base=700 * W + N % 83)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("twoshot_mode", 2)
    try:
        bufs, src, outs = run_allreduce(rr, "twoshot", W, N, dtype, copy_mode, ins)
    finally:
        pad.set_option("twoshot_mode", 0)
    for r in range(W):
        assert_bitwise(outs.host(r), want, f"push output {r}")
    outs.check_guards()
    for r in range(W):
        assert_bitwise(bufs.host(r), ins[r])


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("blocks", [1, 5])
def test_twoshot_modes_fixed_blocks(rr, mode, blocks):
    W, N, dtype = 8, 500_009, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=23)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("twoshot_mode", mode)
    try:
        for copy_mode in (0, 1):
            _, _, outs = run_allreduce(rr, "twoshot", W, N, dtype, copy_mode, ins, blocks_per_rank=blocks)
            for r in range(W):
                assert_bitwise(outs.host(r), want)
    finally:
        pad.set_option("twoshot_mode", 0)


@pytest.mark.parametrize("algo", ["oneshot", "twoshot"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", SHAPES + [(8, (1 << 20) + 3)], ids=[f"W{w}_N{n}" for w, n in SHAPES + [(8, (1 << 20) + 3)]])
def test_staged_copy_mode_matches_oracle(rr, algo, dtype, W, N):
    """copy_mode with the staging done by a bulk-copy producer warp."""
    ins = workloads.rank_buffers(W, N, dtype, dist_for(dtype), seed_base=900 * W + N % 79)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 2)
    try:
        for materialise in ((None,) if algo == "twoshot" else (None, (0,))):
            bufs, src, outs = run_allreduce(rr, algo, W, N, dtype, 1, ins, materialise=materialise)
            assert pad.get_option("last_engine") == 2
            for r in (range(W) if materialise is None else materialise):
                assert_bitwise(outs.host(r), want, f"staged {algo} output {r}")
            outs.check_guards()
            for r in range(W):
                assert_bitwise(bufs.host(r), ins[r], f"staged rank buffer {r}")
    finally:
        pad.set_option("reduce_engine", 0)


@pytest.mark.parametrize("round_bytes", [0, 256, 16384, 1 << 22])  # 0: pieces balanced over the blocks
@pytest.mark.parametrize("blocks", [1, 3, 19])
@pytest.mark.parametrize("algo", ["oneshot", "twoshot"])
def test_staged_rounds_and_blocks(rr, round_bytes, blocks, algo):
    W, N, dtype = 8, 3 * (1 << 18) + 5, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=29)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 2)
    pad.set_option("round_bytes", round_bytes)
    try:
        _, _, outs = run_allreduce(rr, algo, W, N, dtype, 1, ins, blocks_per_rank=blocks)
    finally:
        pad.set_option("reduce_engine", 0)
        pad.set_option("round_bytes", 0)
    for r in range(W):
        assert_bitwise(outs.host(r), want, f"{algo} round_bytes={round_bytes} blocks={blocks} output {r}")


@pytest.mark.parametrize("mode", ["twoshot", "twoshot_pull"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", [(2, 4099), (3, 12345), (8, (1 << 20) + 3), (16, 10000), (5, 7)])
def test_twoshot_in_place(rr, mode, dtype, W, N):
    """outputs[r] == rank_bufs[r]: the sum replaces every rank buffer."""
    ins = workloads.rank_buffers(W, N, dtype, dist_for(dtype), seed_base=1100 * W + N % 71)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    bufs = RankBuffers(W, N, dtype)
    bufs.fill(ins)
    pad.set_option("twoshot_mode", 1 if mode == "twoshot_pull" else 2)
    try:
        rr.rr_allreduce_twoshot(None, bufs.ptrs, bufs.ptrs, W, N, dtype, 0, pad)
        pad.status()
    finally:
        pad.set_option("twoshot_mode", 0)
    for r in range(W):
        assert_bitwise(bufs.host(r), want, f"{mode} in place, rank {r}")


def test_in_place_refused_where_it_would_race(rr):
    W, N = 4, 4096
    pad = pad_for(rr, W)
    bufs = RankBuffers(W, N, "bf16")
    src = RankBuffers(W, N, "bf16")
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, bufs.ptrs, bufs.ptrs, W, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_twoshot(src.ptrs, bufs.ptrs, bufs.ptrs, W, N, "bf16", 1, pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    with pytest.raises(rr.RRError) as e:  # a partial overlap is never in place
        rr.rr_allreduce_twoshot(None, bufs.ptrs, [p + 16 for p in bufs.ptrs], W, N - 8, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    pad.status()


@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", SHAPES, ids=[f"W{w}_N{n}" for w, n in SHAPES])
def test_ldst_copy_mode_matches_oracle(rr, algo, dtype, W, N):
    """copy_mode on the load/store kernels (staging by every thread, rounds)."""
    ins = workloads.rank_buffers(W, N, dtype, dist_for(dtype), seed_base=1300 * W + N % 61)
    want = oracle.allreduce(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 1)
    try:
        bufs, src, outs = run_allreduce(rr, algo, W, N, dtype, 1, ins)
        assert pad.get_option("last_engine") == 1
    finally:
        pad.set_option("reduce_engine", 0)
    for r in range(W):
        assert_bitwise(outs.host(r), want, f"ldst {algo} output {r}")
        assert_bitwise(bufs.host(r), ins[r])
    outs.check_guards()


def test_separate_allocations(rr):
    W, N, dtype = 6, 77_777, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=12)
    want = oracle.allreduce(ins, dtype)
    for algo in ("oneshot", "twoshot"):
        _, _, outs = run_allreduce(rr, algo, W, N, dtype, 1, ins, layout="separate")
        for r in range(W):
            assert_bitwise(outs.host(r), want)


def test_special_values(rr):
    """Infinities, signed zeros, subnormals and NaN inputs.  NaN results are
    compared as a class (the NaN payload after binary32 arithmetic is not
    part of the rule); every other result bit for bit."""
    W, dtype = 3, "bf16"
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x7F7F, 0xFF7F,
                         0x3F80, 0xBF80, 0x0080], dtype=np.uint16)
    n = specials.size
    grid = np.stack(np.meshgrid(*([np.arange(n)] * W), indexing="ij"), -1).reshape(-1, W)
    ins = [specials[grid[:, r]] for r in range(W)]
    want = oracle.allreduce(ins, dtype)
    for algo in ("oneshot", "twoshot"):
        _, _, outs = run_allreduce(rr, algo, W, grid.shape[0], dtype, 0, ins)
        got = outs.host(0)
        wf = oracle.to_f32("bf16", want)
        gf = oracle.to_f32("bf16", got)
        nan = np.isnan(wf)
        assert np.array_equal(np.isnan(gf), nan)
        assert_bitwise(got[~nan], want[~nan], algo)


def test_twoshot_equals_oneshot_repeated(rr):
    W, N, dtype = 8, 1 << 20, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "normal", seed_base=13)
    _, _, a = run_allreduce(rr, "oneshot", W, N, dtype, 0, ins)
    first = a.host(0)
    for algo in ("twoshot", "oneshot", "twoshot_pull"):
        for copy_mode in (0, 1):
            _, _, o = run_allreduce(rr, algo, W, N, dtype, copy_mode, ins)
            for r in range(W):
                assert_bitwise(o.host(r), first, f"{algo} copy={copy_mode} rank {r}")


@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull"])
@pytest.mark.parametrize("copy_mode", [0, 1])
def test_large_workload_full(rr, algo, copy_mode):
    """W=8, bf16, 2^24 elements (32 MiB) per rank, N(0, 1): every output
    element of every rank against the oracle."""
    cfg = workloads.LARGE
    W, N = cfg["W"], cfg["N"]
    ins = workloads.rank_buffers(W, N, "bf16", cfg["dist"], cfg["seed_base"])
    want = oracle.allreduce(ins, "bf16")
    _, _, outs = run_allreduce(rr, algo, W, N, "bf16", copy_mode, ins)
    for r in range(W):
        assert_bitwise(outs.host(r), want, f"{algo} copy={copy_mode} output {r}")
    outs.check_guards()


@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull"])
@pytest.mark.parametrize("copy_mode", [0, 1])
@pytest.mark.parametrize("kib", [8, 16, 32, 64, 128, 256])
def test_back_to_back_alternating_inputs(rr, algo, copy_mode, kib):
    """1000 back-to-back calls on one pad (generation parity alternates),
    inputs alternating between two sets, each call into its own outputs: a
    barrier that let a block read a peer's chunk before it was staged (or
    reduced, for two-shot) would hand back the other set's data."""
    W, dtype, calls = 8, "bf16", 1000
    N = kib * 1024 // 2
    sets = [workloads.rank_buffers(W, N, dtype, "uniform", seed_base=5000 + 17 * k) for k in range(2)]
    wants = [to_device(oracle.allreduce(s, dtype), dtype) for s in sets]
    pad = pad_for(rr, W)
    srcs = []
    for s in sets:
        rb = RankBuffers(W, N, dtype)
        rb.fill(s)
        srcs.append(rb)
    staging = RankBuffers(W, N, dtype)
    outs = torch.empty((calls, W, N), dtype=torch.bfloat16, device="cuda")
    fn = rr.rr_allreduce_oneshot if algo == "oneshot" else rr.rr_allreduce_twoshot
    stream = torch.cuda.current_stream()
    pad.set_option("twoshot_mode", 1 if algo == "twoshot_pull" else 0)
    for i in range(calls):
        s = srcs[i % 2]
        optrs = [outs[i, r].data_ptr() for r in range(W)]
        if copy_mode:
            fn(s.ptrs, staging.ptrs, optrs, W, N, dtype, 1, pad, stream)
        else:
            fn(None, s.ptrs, optrs, W, N, dtype, 0, pad, stream)
    pad.status(stream)
    pad.set_option("twoshot_mode", 0)
    o16 = outs.view(torch.int16)
    for k in range(2):
        bad = (o16[k::2] != wants[k].view(torch.int16)).any(dim=2)   # [calls / 2, W]
        if bad.any():
            i, r = [int(x) for x in bad.nonzero()[0]]
            raise AssertionError(f"call {2 * i + k} rank {r} holds the wrong sum")


def test_zero_elements_is_a_no_op(rr):
    pad = pad_for(rr, 2)
    g0 = pad.get_option("generation")
    bufs = RankBuffers(2, 16, "bf16")
    outs = GuardedOutputs(2, 16, "bf16")
    rr.rr_allreduce_oneshot(None, bufs.ptrs, outs.ptrs, 2, 0, "bf16", 0, pad)
    rr.rr_allreduce_twoshot(None, bufs.ptrs, outs.ptrs, 2, 0, "bf16", 0, pad)
    pad.status()
    assert pad.get_option("generation") == g0
    outs.check_guards()


def test_argument_errors(rr):
    W, N = 4, 1024
    pad = pad_for(rr, W)
    bufs = RankBuffers(W, N, "bf16")
    outs = GuardedOutputs(W, N, "bf16")
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, bufs.ptrs, [bufs.ptrs[0], None, None, None], W, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, [p + 2 for p in bufs.ptrs], outs.ptrs, W, N - 8, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_ALIGNMENT
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_twoshot(None, bufs.ptrs, [outs.ptrs[0], None, outs.ptrs[2], outs.ptrs[3]],
                                W, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, bufs.ptrs[:3], outs.ptrs[:3], 3, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, bufs.ptrs, outs.ptrs, W, N, 9, 0, pad)
    assert e.value.status == rr.RR_ERR_UNSUPPORTED_DTYPE
    with pytest.raises(rr.RRError) as e:
        rr.rr_allreduce_oneshot(None, bufs.ptrs, [None] * W, W, N, "bf16", 0, pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    pad.status()
    outs.check_guards()


AUTO_COPY_CASES = {
    # (algo, W, bf16 elements per rank, engine expected); 2 = staged bulk-copy kernel, 1 = loads/stores
    "oneshot_W2_16MiB": ("oneshot", 2, 8 << 20, 1),
    "oneshot_W4_8MiB": ("oneshot", 4, 4 << 20, 1),
    "oneshot_W4_16MiB": ("oneshot", 4, 8 << 20, 2),
    "oneshot_W8_8MiB": ("oneshot", 8, 4 << 20, 2),
    "oneshot_W16_2MiB": ("oneshot", 16, 1 << 20, 1),
    "twoshot_W2_1MiB": ("twoshot", 2, 1 << 19, 2),
    "twoshot_W8_4MiB": ("twoshot", 8, 2 << 20, 1),
    "twoshot_W8_8MiB": ("twoshot", 8, 4 << 20, 2),
    "twoshot_pull_W8_8MiB": ("twoshot_pull", 8, 4 << 20, 1),
    "oneshot_W16_4MiB": ("oneshot", 16, 2 << 20, 2),
    "twoshot_W16_8MiB_ragged": ("twoshot", 16, (4 << 20) + 13, 2),
    "twoshot_W2_ragged": ("twoshot", 2, 300_007, 2),
}


@pytest.mark.parametrize("case", list(AUTO_COPY_CASES))
def test_automatic_copy_mode_engine(rr, case):
    """copy_mode on the automatic engine: the staged kernel for the one-shot
    when W >= 4 and W x bytes per rank >= 64 MiB, for the push two-shot when
    W = 2 or from 8 MiB per rank; the load/store kernels otherwise.  The sums
    equal the oracle's either way."""
    algo, W, N, expect = AUTO_COPY_CASES[case]
    ins = workloads.rank_buffers(W, N, "bf16", "normal", seed_base=4100 + W)
    want = oracle.allreduce(ins, "bf16")
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 0)
    _, _, outs = run_allreduce(rr, algo, W, N, "bf16", 1, ins, materialise=(0,) if algo == "oneshot" else None)
    assert pad.get_option("last_engine") == expect
    for r in ((0,) if algo == "oneshot" else range(W)):
        assert_bitwise(outs.host(r), want, f"{case} output {r}")
    outs.check_guards()


AUTO_OFF_CASES = {
    # (W, bf16 elements per rank, engine expected) for the one-shot with copy_mode off
    "W16_8MiB": (16, 4 << 20, 2),
    "W16_4MiB": (16, 2 << 20, 1),
    "W10_16MiB": (10, 8 << 20, 2),
    "W8_32MiB": (8, 16 << 20, 1),
    "W12_11MiB_ragged": (12, (11 << 19) + 5, 2),
}


@pytest.mark.parametrize("case", list(AUTO_OFF_CASES))
def test_automatic_oneshot_engine_copy_off(rr, case):
    """The one-shot with copy_mode off on the automatic engine: bulk-copy
    loads when W > 8 and W x bytes per rank >= 128 MiB, loads/stores
    otherwise; the sums equal the oracle's either way."""
    W, N, expect = AUTO_OFF_CASES[case]
    ins = workloads.rank_buffers(W, N, "bf16", "normal", seed_base=4300 + W)
    want = oracle.allreduce(ins, "bf16")
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 0)
    _, _, outs = run_allreduce(rr, "oneshot", W, N, "bf16", 0, ins, materialise=(0, W - 1))
    assert pad.get_option("last_engine") == expect
    for r in (0, W - 1):
        assert_bitwise(outs.host(r), want, f"{case} output {r}")
    outs.check_guards()


AUTO_ALL_OUTPUT_CASES = {
    # (copy_mode, W, bf16 elements per rank, engine expected) for the one-shot with every output kept
    "copy_W4_32MiB": (1, 4, 16 << 20, 1),
    "copy_W8_8MiB": (1, 8, 4 << 20, 1),
    "off_W16_8MiB": (0, 16, 4 << 20, 1),
    "off_W16_32MiB": (0, 16, 16 << 20, 2),
}


@pytest.mark.parametrize("case", list(AUTO_ALL_OUTPUT_CASES))
def test_automatic_oneshot_engine_all_outputs(rr, case):
    """The one-shot's automatic engines count the kept outputs: with every
    output kept the staged kernel gives way to the load/store one, and the
    copy-off bulk-copy kernel needs 512 MiB read per output."""
    copy, W, N, expect = AUTO_ALL_OUTPUT_CASES[case]
    ins = workloads.rank_buffers(W, N, "bf16", "normal", seed_base=4500 + W)
    want = oracle.allreduce(ins, "bf16")
    pad = pad_for(rr, W)
    pad.set_option("reduce_engine", 0)
    _, _, outs = run_allreduce(rr, "oneshot", W, N, "bf16", copy, ins)
    assert pad.get_option("last_engine") == expect
    for r in (0, W // 2, W - 1):
        assert_bitwise(outs.host(r), want, f"{case} output {r}")
    outs.check_guards()
