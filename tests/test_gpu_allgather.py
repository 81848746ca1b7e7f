"""GPU parity: rank-major, list-output and param-contiguous allgather
through the C ABI, bit for bit against the CPU oracle, on every engine
(128-bit loads/stores, TMA bulk copies, the GPU's copy engines).  Random-bit
inputs carry NaN and Inf encodings, which must survive untouched."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GuardedOutputs, RankBuffers, assert_bitwise

pytestmark = pytest.mark.gpu

ENGINES = {"ldst": 1, "tma": 2, "copy_engine": 3}


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


def gather(rr, W, dtype, ins, splits=None, engine="tma", materialise=None, blocks_per_rank=0,
           layout="packed"):
    pad = pad_for(rr, W)
    pad.set_option("gather_engine", ENGINES[engine])
    pad.set_option("blocks_per_rank", blocks_per_rank)
    n = ins[0].size
    bufs = RankBuffers(W, n, dtype, layout=layout)
    bufs.fill(ins)
    outs = GuardedOutputs(W, W * n, dtype, materialise=materialise)
    if splits is None:
        rr.rr_allgather(bufs.ptrs, outs.ptrs, W, n, dtype, pad)
    else:
        rr.rr_allgather_param_contiguous(bufs.ptrs, outs.ptrs, W, splits, dtype, pad)
    pad.status()
    assert pad.get_option("last_engine") == ENGINES[engine]
    pad.set_option("blocks_per_rank", 0)
    return bufs, outs


RM_SHAPES = [(2, 4096), (1, 17), (2, 3), (3, 1001), (8, 8192), (8, 4097), (5, 123_457), (16, 2048),
             (8, 1)]


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", RM_SHAPES, ids=[f"W{w}_N{n}" for w, n in RM_SHAPES])
def test_rank_major_matches_oracle(rr, engine, dtype, W, N):
    ins = workloads.rank_buffers(W, N, dtype, "bits", seed_base=40 * W + N % 89)
    want = oracle.allgather_rank_major(ins, dtype)
    bufs, outs = gather(rr, W, dtype, ins, engine=engine)
    for q in range(W):
        assert_bitwise(outs.host(q), want, f"output {q}")
    outs.check_guards()
    for r in range(W):
        assert_bitwise(bufs.host(r), ins[r], f"shard {r} after the call")


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("materialise", [(0,), (2, 5), (7,)])
def test_rank_major_subset_of_outputs(rr, engine, materialise):
    W, N, dtype = 8, 300_000, "bf16"
    ins = workloads.rank_buffers(W, N, dtype, "bits", seed_base=3)
    want = oracle.allgather_rank_major(ins, dtype)
    _, outs = gather(rr, W, dtype, ins, engine=engine, materialise=materialise)
    for q in materialise:
        assert_bitwise(outs.host(q), want, f"output {q}")
    outs.check_guards()


SPLIT_TABLES = {
    "aligned": [4096, 512, 512, 4096, 8 * 2368, 8 * 2368, 8 * 2368],
    "ragged": [5, 1, 0, 7, 2, 1023, 3],
    "empty_ends": [0, 64, 0, 0, 33, 0],
    "one": [77_777],
    "many_small": [1 + (i * 7) % 13 for i in range(256)],
}


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("dtype", ["bf16", "fp32", "int32", "fp16"])
@pytest.mark.parametrize("table", list(SPLIT_TABLES))
@pytest.mark.parametrize("W", [2, 3, 8])
def test_param_contiguous_matches_oracle(rr, engine, dtype, table, W):
    splits = SPLIT_TABLES[table]
    ins = workloads.rank_buffers(W, sum(splits), dtype, "bits", seed_base=900 + W)
    want = oracle.allgather_param_contiguous(ins, splits, dtype)
    _, outs = gather(rr, W, dtype, ins, splits=splits, engine=engine)
    for q in range(W):
        assert_bitwise(outs.host(q), want, f"{table} output {q}")
    outs.check_guards()


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("blocks", [1, 3, 100])
def test_param_contiguous_fixed_blocks(rr, engine, blocks):
    """One block per rank (the single-block degenerate case) and more blocks
    than params: same bytes."""
    W, splits, dtype = 4, [1000, 24, 4096, 8, 333], "bf16"
    ins = workloads.rank_buffers(W, sum(splits), dtype, "bits", seed_base=5)
    want = oracle.allgather_param_contiguous(ins, splits, dtype)
    _, outs = gather(rr, W, dtype, ins, splits=splits, engine=engine, blocks_per_rank=blocks)
    for q in range(W):
        assert_bitwise(outs.host(q), want)


AUTO_CASES = {
    # (W, splits per rank in bf16 elements (None = rank-major), numel, kept outputs, engine expected);
    # bulk copies from 256 MiB moved per call (shards read + outputs written)
    "W8_16MiB": (8, None, 8 << 20, (0,), 2),
    "W8_16MiB_less_16B": (8, None, (8 << 20) - 8, (0,), 1),
    "W8_param_aligned": (8, [3 << 20, 8, 5 << 20, 4096], None, (0,), 2),
    "W8_param_split_off_16B": (8, [3 << 20, 9, 5 << 20, 4096], None, (0,), 1),
    "W8_1MiB": (8, None, 1 << 19, (0,), 1),
    "W8_11MiB_two_outputs": (8, None, 11 << 19, (0, 6), 2),
    "W2_32MiB": (2, None, 16 << 20, (1,), 1),
    "W2_64MiB": (2, None, 32 << 20, (1,), 2),
    "W8_1MiB_all_outputs": (8, None, 1 << 19, tuple(range(8)), 2),
    "W8_128KiB_two_outputs": (8, None, 1 << 16, (0, 5), 1),
    "W4_param_2MiB_two_outputs": (4, [1 << 19, 24, (1 << 19) - 24], None, (1, 2), 2),
}


@pytest.mark.parametrize("case", list(AUTO_CASES))
def test_automatic_engine_choice(rr, case):
    """The automatic gather engine: bulk copies when a call moves at least
    256 MiB (8 MiB with two or more kept outputs) and every split boundary is
    a multiple of 16 bytes, loads/stores otherwise; the bytes equal the
    oracle's either way."""
    W, splits, numel, keep, expect = AUTO_CASES[case]
    dtype = "bf16"
    pad = pad_for(rr, W)
    pad.set_option("gather_engine", 0)
    n = numel if splits is None else sum(splits)
    ins = workloads.rank_buffers(W, n, dtype, "bits", seed_base=77)
    bufs = RankBuffers(W, n, dtype)
    bufs.fill(ins)
    outs = GuardedOutputs(W, W * n, dtype, materialise=keep)
    if splits is None:
        want = oracle.allgather_rank_major(ins, dtype)
        rr.rr_allgather(bufs.ptrs, outs.ptrs, W, n, dtype, pad)
    else:
        want = oracle.allgather_param_contiguous(ins, splits, dtype)
        rr.rr_allgather_param_contiguous(bufs.ptrs, outs.ptrs, W, splits, dtype, pad)
    pad.status()
    assert pad.get_option("last_engine") == expect
    for q in keep:
        assert_bitwise(outs.host(q), want, f"{case} output {q}")
    outs.check_guards()


@pytest.mark.parametrize("engine", list(ENGINES))
def test_fsdp_layer_full(rr, engine):
    """One transformer layer (hidden 3584 / kv 512 / ffn 18944), W=8, bf16,
    N(0, 0.02): the whole output against the oracle and against the unsharded
    weights themselves."""
    cfg = workloads.FSDP_LAYER
    W = cfg["W"]
    full, shards = workloads.fsdp_layer_shards(W, layer=0, sigma=cfg["sigma"], seed_base=cfg["seed_base"])
    splits = workloads.shard_sizes(workloads.FSDP_LAYER_PARAMS, W)
    want = oracle.allgather_param_contiguous(shards, splits, "bf16")
    assert np.array_equal(want, np.concatenate(full))
    _, outs = gather(rr, W, "bf16", shards, splits=splits, engine=engine, materialise=(0, 5))
    for q in (0, 5):
        assert_bitwise(outs.host(q), want, f"output {q}")
    outs.check_guards()


def test_fsdp_28_layers_unshard_property(rr):
    """28 layers back to back on distinct device buffers, as the benchmark
    runs them.  Weights are drawn on the device; the check is the property
    that holds at any size: the param-contiguous output of layer l equals
    layer l's flattened weights concatenated in param order."""
    cfg = workloads.FSDP_LAYER
    W, L = cfg["W"], cfg["layers"]
    splits = workloads.shard_sizes(workloads.FSDP_LAYER_PARAMS, W)
    S = sum(splits)
    pad = pad_for(rr, W)
    pad.set_option("gather_engine", 0)
    g = torch.Generator(device="cuda").manual_seed(cfg["seed_base"])
    layers = []
    for l in range(L):
        weights = (torch.randn(W * S, generator=g, device="cuda") * cfg["sigma"]).to(torch.bfloat16)
        shards = torch.empty((W, S), dtype=torch.bfloat16, device="cuda")
        o = 0
        for s, e in enumerate(splits):
            shards[:, o:o + e] = weights[o * W:(o + e) * W].view(W, e)
            o += e
        out = torch.empty(W * S, dtype=torch.bfloat16, device="cuda")
        layers.append((weights, shards, out))
    for weights, shards, out in layers:
        rr.rr_allgather_param_contiguous([shards[r] for r in range(W)], [out] + [None] * (W - 1), W,
                                         splits, "bf16", pad)
    pad.status()
    for l, (weights, _, out) in enumerate(layers):
        assert torch.equal(out.view(torch.int16), weights.view(torch.int16)), f"layer {l}"


def _sweep_sizes():
    return [1 << k for k in range(10, 30)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
def test_allgather_size_sweep(rr, dtype):
    """W=8, 1 KiB .. 512 MiB per rank, random bits.  Up to 64 MiB per rank
    the whole output is compared with the oracle on the host; above, on the
    device, with the property every size obeys: output slice r is rank r's
    shard (at 512 MiB per rank the output is exactly 2^32 bytes, so its last
    byte offset is 2^32 - 1; test_gathers_past_4_gib goes beyond)."""
    W = 8
    eb = workloads.ELEM_BYTES[dtype]
    pad = pad_for(rr, W)
    pad.set_option("gather_engine", 0)
    for nbytes in _sweep_sizes():
        n = nbytes // eb
        if nbytes <= 64 << 20:
            ins = workloads.rank_buffers(W, n, dtype, "bits", seed_base=4000 + nbytes % 1000)
            want = oracle.allgather_rank_major(ins, dtype)
            bufs = RankBuffers(W, n, dtype)
            bufs.fill(ins)
            outs = GuardedOutputs(W, W * n, dtype, materialise=(0,))
            rr.rr_allgather(bufs.ptrs, outs.ptrs, W, n, dtype, pad)
            pad.status()
            assert_bitwise(outs.host(0), want, f"{nbytes} B per rank")
            outs.check_guards()
            del bufs, outs
        else:
            it = torch.int16 if eb == 2 else torch.int32
            info = torch.iinfo(it)
            gen = torch.Generator(device="cuda").manual_seed(nbytes)
            shards = torch.randint(info.min, info.max, (W, n), dtype=it, device="cuda", generator=gen)
            out = torch.empty(W * n, dtype=it, device="cuda")
            rr.rr_allgather([shards[r] for r in range(W)], [out] + [None] * (W - 1), W, n, dtype, pad)
            pad.status()
            assert torch.equal(out.view(W, n), shards), f"{nbytes} B per rank"
            del shards, out
            torch.cuda.empty_cache()


# Byte offsets of 2^31 and 2^32 and more: a gather whose output passes 4 GiB
# ("ccl: hierarchical cross-node AllGather (intra-node SDMA + inter-node RDMA)
# #441": its large-profile commit probes u32 byte-offset overflow with a
# gathered int32 output past 2^31 bytes).  576 MiB per rank at W=8: a 4.5 GiB
# output.
BIG_BYTES = 576 << 20
WINDOWS = (1 << 31, 1 << 32)


def _host_windows(t_bytes, centers, half=8192):
    """Bytes [c - half, c + half) of a device uint8 view, for each center c."""
    return [t_bytes[c - half:c + half].cpu().numpy() for c in centers]


@pytest.mark.parametrize("kind", ["rank_major", "param_contiguous"])
def test_gathers_past_4_gib(rr, kind):
    """W=8, 576 MiB of random bits per rank, output 4.5 GiB, on every gather
    engine: the whole output is checked on the device against the layout
    definition, and compared with the oracle on the host (the whole output
    for the default engine, 16 KiB windows around byte offsets 2^31 and 2^32
    and the last 16 KiB for every engine).  The param-contiguous table puts a
    piece across 2^32 bytes and the last two params past it."""
    W, dtype = 8, "int32"
    n = BIG_BYTES // 4
    gen = torch.Generator(device="cuda").manual_seed(4321)
    shards = torch.randint(-(1 << 31), (1 << 31) - 1, (W, n), dtype=torch.int32, device="cuda", generator=gen)
    host_in = [shards[r].cpu().numpy() for r in range(W)]
    if kind == "rank_major":
        splits = [n]
        want = oracle.allgather_rank_major_mt(host_in, dtype)
    else:
        splits = [n - 1_000_003 - 5, 5, 1_000_003]
        want = oracle.allgather_param_contiguous_mt(host_in, splits, dtype)
    want_b = want.view(np.uint8)
    total = W * n * 4
    assert total > (1 << 32) + (1 << 20)
    out = torch.empty(W * n, dtype=torch.int32, device="cuda")
    pad = pad_for(rr, W)
    try:
        for engine in (0, 2, 3):
            pad.set_option("gather_engine", engine)
            out.fill_(-1)
            if kind == "rank_major":
                rr.rr_allgather([shards[r] for r in range(W)], [out] + [None] * (W - 1), W, n, dtype, pad)
            else:
                rr.rr_allgather_param_contiguous([shards[r] for r in range(W)], [out] + [None] * (W - 1), W,
                                                 splits, dtype, pad)
            pad.status()
            # the definition, on the device
            o = 0
            for e in splits:
                got = out[o * W:(o + e) * W].view(W, e)
                assert torch.equal(got, shards[:, o:o + e]), f"engine {engine}: param at element {o}"
                o += e
            # the oracle, on the host
            ob = out.view(torch.uint8)
            centers = list(WINDOWS) + [total - 8192]
            for c, w in zip(centers, _host_windows(ob, centers)):
                assert np.array_equal(w, want_b[c - 8192:c + 8192]), f"engine {engine}: bytes around {c}"
            if engine == 0:
                assert np.array_equal(ob.cpu().numpy(), want_b), "engine 0: whole output against the oracle"
    finally:
        pad.set_option("gather_engine", 0)
    del shards, out
    torch.cuda.empty_cache()


def test_gather_argument_errors(rr):
    W, N = 4, 1024
    pad = pad_for(rr, W)
    bufs = RankBuffers(W, N, "fp32")
    outs = GuardedOutputs(W, W * N, "fp32")
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather(bufs.ptrs, [bufs.ptrs[1] - 16, None, None, None], W, N, "fp32", pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather_param_contiguous(bufs.ptrs, outs.ptrs, W, [10, -1], "fp32", pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather_param_contiguous(bufs.ptrs, outs.ptrs, W, [1] * 257, "fp32", pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather(bufs.ptrs, [outs.ptrs[0] + 4, None, None, None], W, N, "fp32", pad)
    assert e.value.status == rr.RR_ERR_ALIGNMENT
    pad.status()


LIST_SHAPES = [(2, 4096), (3, 1001), (8, 8195), (16, 2048), (8, 1), (5, 77_777)]


class ListOutputs:
    """W lists of W device buffers (row q = rank q's all_gather tensor_list),
    every buffer a separate slice of one arena with canaries on both sides
    and a ragged lead, so that no buffer sits at an allocation's base and
    the rows are not laid out rank-major."""

    def __init__(self, W, n, dtype, materialise=None):
        eb = workloads.ELEM_BYTES[dtype]
        self.W, self.n, self.dtype, self.eb = W, n, dtype, eb
        self.rows = set(range(W)) if materialise is None else set(materialise)
        self.stride = ((n * eb + 15) // 16) * 16 + 2 * 256
        self.arena = torch.full((W * W * self.stride + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
        base = self.arena.data_ptr()
        # buffer (q, r) sits at slot (r * W + q) reversed: column-major and backwards
        self.off = {}
        for q in range(W):
            for r in range(W):
                slot = W * W - 1 - (r * W + q)
                self.off[(q, r)] = 2048 + slot * self.stride + 256
        self.lists = [[base + self.off[(q, r)] for r in range(W)] if q in self.rows else None
                      for q in range(W)]

    def host(self, q, r):
        o = self.off[(q, r)]
        t = self.arena[o:o + self.n * self.eb]
        return t.cpu().numpy().view(workloads.STORAGE[self.dtype])

    def check_guards(self):
        a = self.arena.cpu().numpy()
        used = np.zeros(a.size, dtype=bool)
        for q in self.rows:
            for r in range(self.W):
                o = self.off[(q, r)]
                used[o:o + self.n * self.eb] = True
        assert np.all(a[~used] == 0xA5), "a byte outside the list buffers was written"


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32", "int32"])
@pytest.mark.parametrize("W,N", LIST_SHAPES, ids=[f"W{w}_N{n}" for w, n in LIST_SHAPES])
def test_list_output_matches_oracle(rr, engine, dtype, W, N):
    """torch.distributed.all_gather semantics: buffer r of every list holds
    rank r's shard, i.e. slice r of the oracle's rank-major output."""
    ins = workloads.rank_buffers(W, N, dtype, "bits", seed_base=70 * W + N % 97)
    want = oracle.allgather_rank_major(ins, dtype)
    pad = pad_for(rr, W)
    pad.set_option("gather_engine", ENGINES[engine])
    bufs = RankBuffers(W, N, dtype)
    bufs.fill(ins)
    materialise = (0,) if W == 16 else None
    outs = ListOutputs(W, N, dtype, materialise=materialise)
    rr.rr_allgather_list(bufs.ptrs, outs.lists, W, N, dtype, pad)
    pad.status()
    assert pad.get_option("last_engine") == ENGINES[engine]
    for q in sorted(outs.rows):
        for r in range(W):
            assert_bitwise(outs.host(q, r), want[r * N:(r + 1) * N], f"list {q} buffer {r}")
    outs.check_guards()


def test_list_output_argument_errors(rr):
    W, N = 4, 1024
    pad = pad_for(rr, W)
    pad.set_option("gather_engine", 0)
    bufs = RankBuffers(W, N, "fp32")
    outs = ListOutputs(W, N, "fp32")
    half = [outs.lists[0][:2] + [None, None]] + outs.lists[1:]
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather_list(bufs.ptrs, half, W, N, "fp32", pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather_list(bufs.ptrs, [None] * W, W, N, "fp32", pad)
    assert e.value.status == rr.RR_ERR_INVALID_ARG
    dup = [list(row) for row in outs.lists]
    dup[2][3] = dup[1][0]
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather_list(bufs.ptrs, dup, W, N, "fp32", pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    onto_shard = [list(row) for row in outs.lists]
    onto_shard[0][1] = bufs.ptrs[3]
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather_list(bufs.ptrs, onto_shard, W, N, "fp32", pad)
    assert e.value.status == rr.RR_ERR_ALIAS
    odd = [list(row) for row in outs.lists]
    odd[3][2] = odd[3][2] + 4
    with pytest.raises(rr.RRError) as e:
        rr.rr_allgather_list(bufs.ptrs, odd, W, N, "fp32", pad)
    assert e.value.status == rr.RR_ERR_ALIGNMENT
    # nothing was written by the rejected calls
    a = outs.arena.cpu().numpy()
    assert np.all(a == 0xA5)
    pad.status()


@pytest.mark.parametrize("engine", list(ENGINES))
def test_engines_agree_on_the_fsdp_layer_and_the_list(rr, engine):
    """Every engine, given the same shards, writes the same bytes as the
    oracle into a param-contiguous output and into list outputs, back to
    back on one pad (the copy engines leave the pad's generation as it
    was, the kernels advance it)."""
    W, dtype = 8, "bf16"
    splits = [4096, 512, 512, 4096, 9, 8 * 2368, 8 * 2368]
    ins = workloads.rank_buffers(W, sum(splits), dtype, "bits", seed_base=77)
    want = oracle.allgather_param_contiguous(ins, splits, dtype)
    pad = pad_for(rr, W)
    g0 = pad.get_option("generation")
    _, outs = gather(rr, W, dtype, ins, splits=splits, engine=engine, materialise=(1, 6))
    g1 = pad.get_option("generation")
    assert (g1 == g0) if engine == "copy_engine" else (g1 != g0)
    for q in (1, 6):
        assert_bitwise(outs.host(q), want, f"output {q}")
    outs.check_guards()
