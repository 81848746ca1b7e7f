"""Pins of the CPU oracle to things other than itself.

Each check below fixes the oracle against a fact that does not come from the
oracle: hand-worked IEEE arithmetic (tests/golden), exhaustive or random
comparison of the element conversions with torch / numpy, closed forms, the
FSDP meaning of the param-contiguous layout, and an independent torch CPU
chain for the reduction.  They are chosen so that a plausible slip in
oracle.c (a dropped rank, a wrong start value, a reversed order, a different
accumulator width, a wrong rounding rule, a transposed layout index) fails at
least one of them; tests/test_oracle_mutants.py plants such slips to show it.
"""
import json
import os

import numpy as np
import pytest
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits(hexes, dtype):
    if dtype == "int32":
        return np.array(hexes, dtype=np.int64).astype(np.int32)
    if dtype == "fp32":
        return np.array([int(h, 16) for h in hexes], dtype=np.uint32).view(np.float32)
    return np.array([int(h, 16) for h in hexes], dtype=np.uint16)


def _u(a):
    """raw bits as an unsigned integer array, for exact comparison"""
    a = np.asarray(a)
    return a.view({2: np.uint16, 4: np.uint32}[a.dtype.itemsize])


def _same_bits_nan_as_class(got_bits, want_bits, is_nan_got, is_nan_want):
    assert np.array_equal(is_nan_got, is_nan_want), "NaN positions differ"
    keep = ~is_nan_want
    bad = np.nonzero(got_bits[keep] != want_bits[keep])[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


# ---------------------------------------------------------------- conversions

def _torch_bf16_bits_to_f32(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()


def _torch_f32_to_bf16_bits(x):
    return torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_widen_exhaustive(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.to_f32("bf16", bits)
    want = _torch_bf16_bits_to_f32(bits)
    _same_bits_nan_as_class(_u(got), _u(want), np.isnan(got), np.isnan(want))


def test_fp16_widen_exhaustive(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.to_f32("fp16", bits)
    want = bits.view(np.float16).astype(np.float32)
    _same_bits_nan_as_class(_u(got), _u(want), np.isnan(got), np.isnan(want))


def _narrowing_inputs():
    rng = np.random.default_rng(12345)
    rand = rng.integers(0, 1 << 32, size=1 << 24, dtype=np.uint64).astype(np.uint32)
    # bit patterns at and around every 16-bit rounding boundary of a spread of
    # exponents: ties (low half 0x8000 / 0x1000 ...), one below and one above.
    hi = rng.integers(0, 1 << 16, size=1 << 16, dtype=np.uint64).astype(np.uint32) << 16
    edges = [hi | 0x8000, hi | 0x7FFF, hi | 0x8001, hi | 0x1000, hi | 0x0FFF, hi | 0x1001,
             hi | 0x2000, hi | 0x3000]
    specials = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7F8000, 0x7F7F7FFF,
                         0x00008000, 0x00018000, 0x00000001, 0x807FFFFF, 0x477FE000,
                         0x477FEFFF, 0x477FF000, 0x33000000, 0x33000001, 0x387FC000,
                         0x38800000, 0x337FFFFF, 0x32FFFFFF], dtype=np.uint32)
    return np.concatenate([rand] + edges + [specials]).view(np.float32)


def test_f32_to_bf16_matches_torch(oracle_mod):
    x = _narrowing_inputs()
    got = oracle_mod.f32_to("bf16", x)
    want = _torch_f32_to_bf16_bits(x)
    gn = np.isnan(_torch_bf16_bits_to_f32(got))
    wn = np.isnan(_torch_bf16_bits_to_f32(want))
    _same_bits_nan_as_class(got, want, gn, wn)


def test_f32_to_fp16_matches_numpy(oracle_mod):
    x = _narrowing_inputs()
    got = oracle_mod.f32_to("fp16", x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    _same_bits_nan_as_class(got, want, np.isnan(got.view(np.float16)), np.isnan(want.view(np.float16)))


# ---------------------------------------------------------------- allreduce

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden("allreduce_cases.json"), ids=lambda c: c["name"])
def test_allreduce_golden(oracle_mod, case):
    dt = case["dtype"]
    ins = [_bits(v, dt) for v in case["inputs"]]
    got = oracle_mod.allreduce(ins, dt)
    want = _bits(case["expected"], dt)
    assert np.array_equal(_u(got), _u(want)), (case["name"], _u(got), _u(want))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
def test_allreduce_w1_is_identity(oracle_mod, dtype):
    """One rank: the sum is the rank's own buffer, bit for bit (every finite
    value, both zeros, subnormals and infinities survive the widening to
    binary32 and the narrowing back)."""
    if dtype in ("bf16", "fp16"):
        x = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        keep = ~np.isnan(oracle_mod.to_f32(dtype, x))
        x = x[keep]
    else:
        x = workloads.rank_buffer(1 << 16, dtype, "bits", 7)
        if dtype == "fp32":
            x = x[~np.isnan(x)]
    got = oracle_mod.allreduce([x], dtype)
    assert np.array_equal(_u(got), _u(x))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_allreduce_w2_is_correctly_rounded_sum(oracle_mod, dtype):
    """Two ranks whose values lie in [2^-8, 1] (or are 0): the binary64 sum is
    exact, and the single rounding of that exact sum to the element type is
    the answer (closed form; rounding done by torch, not by the oracle)."""
    rng = np.random.default_rng(99)
    n = 1 << 16
    tdt = workloads.TORCH_DTYPE[dtype]
    vals = []
    for _ in range(2):
        mag = np.exp2(rng.uniform(-8, 0, size=n)).astype(np.float32)
        sign = np.where(rng.integers(0, 2, size=n) == 1, -1.0, 1.0).astype(np.float32)
        v = torch.from_numpy(mag * sign).to(tdt)
        v[::97] = 0
        vals.append(v)
    exact = vals[0].double() + vals[1].double()
    want = exact.to(tdt)
    ins = [v.view(torch.int16).numpy().view(np.uint16) if dtype != "fp32" else v.numpy()
           for v in vals]
    got = oracle_mod.allreduce(ins, dtype)
    want_np = want.view(torch.int16).numpy().view(np.uint16) if dtype != "fp32" else want.numpy()
    assert np.array_equal(_u(got), _u(want_np))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("W", [3, 8])
def test_allreduce_matches_torch_cpu_chain(oracle_mod, dtype, W):
    """An independent restatement through torch CPU element-wise ops:
    acc = x0.float(); acc = acc + xr.float() for r = 1..W-1; acc.to(dtype)."""
    n = 40_000
    ins = workloads.rank_buffers(W, n, dtype, "normal", seed_base=500 + W)
    tdt = workloads.TORCH_DTYPE[dtype]

    def t(a):
        if dtype == "fp32":
            return torch.from_numpy(a.copy())
        return torch.from_numpy(a.view(np.int16).copy()).view(tdt)

    acc = t(ins[0]).float()
    for r in range(1, W):
        acc = acc + t(ins[r]).float()
    want = acc.to(tdt)
    want_np = want.numpy() if dtype == "fp32" else want.view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.allreduce(ins, dtype)
    assert np.array_equal(_u(got), _u(want_np))


def test_allreduce_int32_wraps_like_modular_sum(oracle_mod):
    W, n = 8, 50_000
    ins = workloads.rank_buffers(W, n, "int32", "int", seed_base=77)
    total = np.zeros(n, dtype=np.int64)
    for a in ins:
        total += a.astype(np.int64)
    want = ((total + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32)
    assert np.array_equal(oracle_mod.allreduce(ins, "int32"), want)


def test_allreduce_is_rank_order_sensitive_only_through_rounding(oracle_mod):
    """Reversing the ranks changes some fp32 results (so the order is really
    fixed), but never by more than the rounding of W-1 binary32 additions."""
    W, n = 8, 100_000
    ins = workloads.rank_buffers(W, n, "fp32", "normal", seed_base=31)
    fwd = oracle_mod.allreduce(ins, "fp32")
    rev = oracle_mod.allreduce(ins[::-1], "fp32")
    assert not np.array_equal(fwd, rev)
    exact = np.sum(np.stack(ins).astype(np.float64), axis=0)
    bound = (W - 1) * np.finfo(np.float32).eps * np.sum(np.abs(np.stack(ins)), axis=0, dtype=np.float64)
    assert np.all(np.abs(fwd - exact) <= bound)


def test_allreduce_brute_force_tiny(oracle_mod):
    """All W in 1..4 on 6 elements, by an explicit Python loop over exact
    binary32 additions (numpy float32 scalars)."""
    for W in range(1, 5):
        ins = workloads.rank_buffers(W, 6, "fp32", "normal", seed_base=900 + W)
        want = np.empty(6, dtype=np.float32)
        for i in range(6):
            acc = np.float32(ins[0][i])
            for r in range(1, W):
                acc = np.float32(acc + np.float32(ins[r][i]))
            want[i] = acc
        assert np.array_equal(_u(oracle_mod.allreduce(ins, "fp32")), _u(want))


def test_allreduce_empty(oracle_mod):
    got = oracle_mod.allreduce([np.zeros(0, np.uint16)] * 3, "bf16")
    assert got.size == 0


# ---------------------------------------------------------------- allgathers

@pytest.mark.parametrize("case", _golden("allgather_cases.json"), ids=lambda c: c["name"])
def test_allgather_golden(oracle_mod, case):
    ins = [np.array(v, dtype=np.int32) for v in case["inputs"]]
    if case["kind"] == "rank_major":
        got = oracle_mod.allgather_rank_major(ins, "int32")
    else:
        got = oracle_mod.allgather_param_contiguous(ins, case["splits"], "int32")
    assert got.tolist() == case["expected"]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", [(1, 5), (2, 3), (3, 1001), (8, 4096)])
def test_rank_major_matches_torch_cat(oracle_mod, dtype, W, N):
    ins = workloads.rank_buffers(W, N, dtype, "bits", seed_base=40 + W)
    want = torch.cat([torch.from_numpy(a.view(np.uint8).copy()) for a in ins]).numpy()
    got = oracle_mod.allgather_rank_major(ins, dtype)
    assert np.array_equal(got.view(np.uint8), want)


def test_param_contiguous_is_fsdp_unshard(oracle_mod):
    """FSDP meaning of the layout: when every rank holds the r-th even slice
    of each flattened weight, the param-contiguous output is the weights
    themselves, concatenated in param order."""
    W = 4
    params = (("a", 6, 8), ("b", 4, 4), ("c", 12, 2), ("d", 4, 1))
    full, shards = workloads.fsdp_layer_shards(W, layer=0, params=params)
    got = oracle_mod.allgather_param_contiguous(shards, workloads.shard_sizes(params, W), "bf16")
    assert np.array_equal(got, np.concatenate(full))


def test_param_contiguous_is_a_permutation_of_rank_major(oracle_mod):
    """Same multiset of bytes as the rank-major output, and each output
    element is a distinct input element (tags make every element unique)."""
    W, splits = 3, [5, 1, 0, 7, 2]
    S = sum(splits)
    ins = [np.arange(r * 1000, r * 1000 + S, dtype=np.int32) for r in range(W)]
    pc = oracle_mod.allgather_param_contiguous(ins, splits, "int32")
    rm = oracle_mod.allgather_rank_major(ins, "int32")
    assert sorted(pc.tolist()) == sorted(rm.tolist())
    assert len(set(pc.tolist())) == W * S


def test_param_contiguous_single_split_equals_rank_major(oracle_mod):
    ins = workloads.rank_buffers(5, 333, "fp16", "bits", seed_base=8)
    a = oracle_mod.allgather_param_contiguous(ins, [333], "fp16")
    b = oracle_mod.allgather_rank_major(ins, "fp16")
    assert np.array_equal(a, b)


def test_param_contiguous_unsplit_weights_qwen_layer_shapes(oracle_mod):
    """The full one-layer FSDP split table, at 1/64 scale of the row count
    (same seven weights, same order and ratios)."""
    W = 8
    params = tuple((n, max(1, r // 64), c) for n, r, c in workloads.FSDP_LAYER_PARAMS)
    full, shards = workloads.fsdp_layer_shards(W, layer=1, params=params)
    got = oracle_mod.allgather_param_contiguous(shards, workloads.shard_sizes(params, W), "bf16")
    assert np.array_equal(got, np.concatenate(full))


def node_block_scatter(shards, splits, G):
    """The PR's node-block form of the param-contiguous gather ("ccl:
    hierarchical cross-node AllGather (intra-node SDMA + inter-node RDMA)
    #441", the commit adding enqueue_param_contiguous), written out
    independently of the oracle: ranks come in node blocks of G; for node
    block m and param s the scatter starts at O_s*W + m*G*E_s and the ranks
    of the block follow each other at a stride of E_s."""
    W = len(shards)
    S = sum(splits)
    out = np.full(W * S, -1, dtype=np.int64)
    for m in range(W // G):
        o = 0
        for e in splits:
            block_offset = o * W + m * G * e
            for j in range(G):
                r = m * G + j
                dst = block_offset + j * e
                out[dst:dst + e] = shards[r][o:o + e]
            o += e
    return out


@pytest.mark.parametrize("W", [4, 8, 6])
def test_param_contiguous_independent_of_node_grouping(oracle_mod, W):
    """Every node-block size G that divides W puts every byte where the
    oracle's single formula does: G is not an argument of the layout."""
    splits = [5, 0, 9, 1, 16]
    S = sum(splits)
    shards = [np.arange(r * 10_000, r * 10_000 + S, dtype=np.int32) for r in range(W)]
    want = oracle_mod.allgather_param_contiguous(shards, splits, "int32")
    for G in [g for g in range(1, W + 1) if W % g == 0]:
        got = node_block_scatter(shards, splits, G)
        assert (got >= 0).all(), f"G={G} leaves holes"
        assert np.array_equal(got, want.astype(np.int64)), f"G={G}"
