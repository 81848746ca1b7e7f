"""GPU parity on seeded random configurations: world size, element count,
dtype, algorithm, copy_mode, engine, blocks per rank, kept outputs and
split tables drawn at random (fixed seed, so every run tests the same
cases), each result compared with the oracle.  Covers combinations the
hand-picked parity cases do not list one by one."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GuardedOutputs, RankBuffers, assert_bitwise

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16", "fp32", "int32"]


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    from allgather_rr_allreduce_gb300 import build
    build.build()
    import allgather_rr_allreduce_gb300 as m
    m.lib()
    return m


def _size(rng):
    # mostly small and ragged, sometimes several hundred thousand elements
    kind = rng.integers(0, 4)
    if kind == 0:
        return int(rng.integers(1, 64))
    if kind == 1:
        return int(rng.integers(64, 8192))
    if kind == 2:
        return int(rng.integers(8192, 200_000))
    return int(rng.integers(200_000, 700_000))


def _allreduce_case(i):
    rng = np.random.default_rng(4242 + i)
    W = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 11, 16]))
    return dict(
        W=W, N=_size(rng), dtype=DTYPES[int(rng.integers(0, 4))],
        algo=["oneshot", "twoshot"][int(rng.integers(0, 2))], copy_mode=int(rng.integers(0, 2)),
        reduce_engine=int(rng.integers(0, 3)), twoshot_mode=int(rng.integers(0, 3)),
        blocks=int(rng.choice([0, 0, 1, 2, 5, 13])), round_bytes=int(rng.choice([0, 0, 4096, 65536])),
        keep=sorted(set(int(q) for q in rng.integers(0, W, size=int(rng.integers(1, W + 1))))),
        layout=["packed", "separate"][int(rng.integers(0, 2))], seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("i", range(48))
def test_fuzz_allreduce(rr, i):
    c = _allreduce_case(i)
    W, N, dtype = c["W"], c["N"], c["dtype"]
    dist = "int" if dtype == "int32" else "normal"
    ins = workloads.rank_buffers(W, N, dtype, dist, seed_base=c["seed"])
    want = oracle.allreduce(ins, dtype)
    pad = rr.rr_signal_pad_create(W)
    pad.set_option("reduce_engine", c["reduce_engine"])
    pad.set_option("twoshot_mode", c["twoshot_mode"])
    pad.set_option("round_bytes", c["round_bytes"])
    if c["blocks"] and c["blocks"] * W <= 152:
        pad.set_option("blocks_per_rank", c["blocks"])
    keep = None if c["algo"] == "twoshot" else c["keep"]
    src = RankBuffers(W, N, dtype, layout=c["layout"])
    src.fill(ins)
    outs = GuardedOutputs(W, N, dtype, materialise=keep)
    fn = getattr(rr, f"rr_allreduce_{c['algo']}")
    if c["copy_mode"]:
        staging = RankBuffers(W, N, dtype, layout=c["layout"])
        fn(src.ptrs, staging.ptrs, outs.ptrs, W, N, dtype, 1, pad)
    else:
        fn(None, src.ptrs, outs.ptrs, W, N, dtype, 0, pad)
    pad.status()
    for q in (range(W) if keep is None else keep):
        assert_bitwise(outs.host(q), want, f"case {c}: output {q}")
    outs.check_guards()
    if c["copy_mode"]:
        for r in range(W):
            assert_bitwise(staging.host(r), ins[r], f"case {c}: staged buffer {r}")
    pad.close()


def _gather_case(i):
    rng = np.random.default_rng(777 + i)
    W = int(rng.choice([1, 2, 3, 4, 5, 8, 9, 16]))
    nsplit = int(rng.choice([1, 1, 2, 7, 30, 256]))
    splits = [int(x) for x in rng.integers(0, 4000 if nsplit < 30 else 300, size=nsplit)]
    if rng.integers(0, 3) == 0:
        splits = [s - s % 8 for s in splits]          # 16-byte multiples for 2-byte types
    if sum(splits) == 0:
        splits[0] = 5
    return dict(W=W, splits=splits, dtype=DTYPES[int(rng.integers(0, 4))],
                kind=["rank_major", "param_contiguous", "list"][int(rng.integers(0, 3))],
                engine=int(rng.integers(0, 4)), blocks=int(rng.choice([0, 0, 1, 3, 40])),
                keep=sorted(set(int(q) for q in rng.integers(0, W, size=int(rng.integers(1, W + 1))))),
                seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("i", range(48))
def test_fuzz_allgather(rr, i):
    c = _gather_case(i)
    W, dtype = c["W"], c["dtype"]
    splits = c["splits"] if c["kind"] == "param_contiguous" else [sum(c["splits"])]
    S = sum(splits)
    ins = workloads.rank_buffers(W, S, dtype, "bits", seed_base=c["seed"])
    pad = rr.rr_signal_pad_create(W)
    pad.set_option("gather_engine", c["engine"])
    if c["blocks"] and c["blocks"] * W <= 152:
        pad.set_option("blocks_per_rank", c["blocks"])
    src = RankBuffers(W, S, dtype)
    src.fill(ins)
    if c["kind"] == "list":
        rows = {q: GuardedOutputs(W, S, dtype) for q in c["keep"]}
        rr.rr_allgather_list(src.ptrs, [rows[q].ptrs if q in rows else None for q in range(W)], W, S, dtype,
                             pad)
        pad.status()
        for q, row in rows.items():
            for r in range(W):
                assert_bitwise(row.host(r), ins[r], f"case {c}: list {q} entry {r}")
            row.check_guards()
    else:
        outs = GuardedOutputs(W, W * S, dtype, materialise=c["keep"])
        if c["kind"] == "rank_major":
            rr.rr_allgather(src.ptrs, outs.ptrs, W, S, dtype, pad)
            want = oracle.allgather_rank_major(ins, dtype)
        else:
            rr.rr_allgather_param_contiguous(src.ptrs, outs.ptrs, W, splits, dtype, pad)
            want = oracle.allgather_param_contiguous(ins, splits, dtype)
        pad.status()
        for q in c["keep"]:
            assert_bitwise(outs.host(q), want, f"case {c}: output {q}")
        outs.check_guards()
    for r in range(W):
        assert_bitwise(src.host(r), ins[r], f"case {c}: shard {r} after the call")
    pad.close()
