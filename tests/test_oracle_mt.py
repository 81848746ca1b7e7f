"""The oracle's multi-threaded entry points (used only to time the CPU
baseline on every host core) give the same bits as the single-threaded
definitions for every dtype, world size, thread count and layout, including
NaN, infinity, -0 and subnormal inputs: only the element range is split over
threads, never the per-element order."""
import numpy as np
import pytest

import workloads


def _u(a):
    a = np.asarray(a)
    return a.view({2: np.uint16, 4: np.uint32}[a.dtype.itemsize])


def _specials(dtype, n, rng):
    """Random raw bits, so NaN payloads, infinities, -0 and subnormals occur."""
    if dtype in ("bf16", "fp16"):
        return rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
    if dtype == "fp32":
        return rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    return rng.integers(-(1 << 31), 1 << 31, n, dtype=np.int64).astype(np.int32)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", [(1, 7), (2, 4096), (3, 100_003), (8, 1 << 18), (16, 12_345)])
@pytest.mark.parametrize("threads", [1, 2, 3, 0])
def test_allreduce_mt_same_bits(oracle_mod, dtype, W, N, threads):
    ins = workloads.rank_buffers(W, N, dtype, "normal" if dtype != "int32" else "int32", seed_base=11 * W + N % 97)
    assert np.array_equal(_u(oracle_mod.allreduce_mt(ins, dtype, threads)), _u(oracle_mod.allreduce(ins, dtype)))
    rng = np.random.default_rng(W * 1000 + N)
    raw = [_specials(dtype, N, rng) for _ in range(W)]
    assert np.array_equal(_u(oracle_mod.allreduce_mt(raw, dtype, threads)), _u(oracle_mod.allreduce(raw, dtype)))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("threads", [1, 4, 0])
def test_gathers_mt_same_bits(oracle_mod, dtype, threads):
    rng = np.random.default_rng(7)
    W, N = 8, (3 << 20) // workloads.ELEM_BYTES[dtype] + 5   # several 1 MiB pieces per rank, ragged
    ins = [_specials(dtype, N, rng) for _ in range(W)]
    assert np.array_equal(_u(oracle_mod.allgather_rank_major_mt(ins, dtype, threads)),
                          _u(oracle_mod.allgather_rank_major(ins, dtype)))
    splits = [N // 3 - 17, 0, 17, N - N // 3]
    assert np.array_equal(_u(oracle_mod.allgather_param_contiguous_mt(ins, splits, dtype, threads)),
                          _u(oracle_mod.allgather_param_contiguous(ins, splits, dtype)))


def test_mt_rejects_what_the_definition_rejects(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.allgather_param_contiguous_mt([np.zeros(4, np.uint16)] * 2, [5, -1], "bf16")
    assert oracle_mod.max_threads() >= 1
