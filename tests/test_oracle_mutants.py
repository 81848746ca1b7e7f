"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a one-line slip applied to a copy of oracle/oracle.c, built in
a temporary directory and swapped in for the real library while a quick set
of pins from test_oracle_pins.py runs.  A mutant that no pin catches would
mean the pins cannot tell that mistake from the right answer.  The real
oracle is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "drop_last_rank": ("for (int r = 1; r < W; ++r) acc = acc + load_as_f32",
                       "for (int r = 1; r < W - 1; ++r) acc = acc + load_as_f32"),
    "start_from_plus_zero": ("float acc = load_as_f32(in[0], dtype, i);",
                             "float acc = 0.0f + load_as_f32(in[0], dtype, i);"),
    "reverse_rank_order": ("float acc = load_as_f32(in[0], dtype, i);\n"
                           "        for (int r = 1; r < W; ++r) acc = acc + load_as_f32(in[r], dtype, i);",
                           "float acc = load_as_f32(in[W - 1], dtype, i);\n"
                           "        for (int r = W - 2; r >= 0; --r) acc = acc + load_as_f32(in[r], dtype, i);"),
    "bf16_accumulator": ("acc = acc + load_as_f32(in[r], dtype, i);",
                         "acc = dtype == ORACLE_BF16 ? oracle_bf16_to_f32(oracle_f32_to_bf16(acc + load_as_f32(in[r], dtype, i))) : acc + load_as_f32(in[r], dtype, i);"),
    "bf16_truncate": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;",
                      "(void)dropped;"),
    "bf16_ties_away": ("(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    "fp16_wrong_subnormal_quantum": ("E = -24;\n", "E = -25;\n"),
    "fp16_ties_away": ("(frac == 0.5f && (q & 1u))", "(frac == 0.5f)"),
    "sign_flip_rank": ("acc = acc + load_as_f32(in[r], dtype, i);",
                       "acc = r == 1 ? acc - load_as_f32(in[r], dtype, i) : acc + load_as_f32(in[r], dtype, i);"),
    "int32_drop_rank0": ("uint32_t acc = (uint32_t)((const int32_t *)in[0])[i];", "uint32_t acc = 0u;"),
    "pc_missing_rank_stride": ("(O * W + (int64_t)r * E)", "(O + (int64_t)r * E)"),
    "pc_transposed": ("(O * W + (int64_t)r * E)", "((int64_t)r * total + O)"),
    "rank_major_reversed": ("(size_t)r * (size_t)numel * (size_t)esize, in[r]",
                            "(size_t)(W - 1 - r) * (size_t)numel * (size_t)esize, in[r]"),
}


def _quick_pins():
    om = oracle
    for c in pins._golden("allreduce_cases.json"):
        yield lambda c=c: pins.test_allreduce_golden(om, c)
    for c in pins._golden("allgather_cases.json"):
        yield lambda c=c: pins.test_allgather_golden(om, c)
    for dt in ("bf16", "fp16", "fp32", "int32"):
        yield lambda dt=dt: pins.test_allreduce_w1_is_identity(om, dt)
    for dt in ("bf16", "fp16", "fp32"):
        yield lambda dt=dt: pins.test_allreduce_matches_torch_cpu_chain(om, dt, 3)
    yield lambda: pins.test_allreduce_int32_wraps_like_modular_sum(om)
    yield lambda: pins.test_param_contiguous_is_fsdp_unshard(om)
    yield lambda: pins.test_rank_major_matches_torch_cat(om, "int32", 3, 1001)


# oracle.c holds the single-threaded definitions first, then the multi-threaded
# copies of the same loops after this marker.
MT_MARK = "/* ------------------------------------------------------------ multi-threaded"


def _build_mutant(tmp_path, name, old, new, part="single"):
    text = open(SRC).read()
    head, mark, tail = text.partition(MT_MARK)
    assert mark, "multi-threaded section marker missing"
    if part == "single":
        assert head.count(old) == 1, f"mutant {name}: anchor not found exactly once"
        head = head.replace(old, new)
    else:
        assert tail.count(old) == 1, f"mutant {name}: anchor not found exactly once in the threaded loops"
        tail = tail.replace(old, new)
    src = tmp_path / f"{name}_{part}.c"
    src.write_text(head + mark + tail)
    so = tmp_path / f"{name}_{part}.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(src), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, name, old, new)
    real = oracle.lib()
    mutant = ctypes.CDLL(so)
    for fn in ("oracle_allreduce", "oracle_allgather_rank_major",
               "oracle_allgather_param_contiguous", "oracle_cast"):
        f = getattr(mutant, fn)
        f.argtypes = getattr(real, fn).argtypes
        f.restype = ctypes.c_int
    oracle._lib = mutant
    caught = 0
    try:
        for pin in _quick_pins():
            try:
                pin()
            except AssertionError:
                caught += 1
    finally:
        oracle._lib = real
    assert caught > 0, f"no pin caught mutant {name}"


def test_real_oracle_passes_quick_pins():
    for pin in _quick_pins():
        pin()


# The same slips planted in the multi-threaded copies of the loops (where
# their anchor occurs there): comparing the threaded entry points with the
# single-threaded definitions, as tests/test_oracle_mt.py does, must catch them.
MT_MUTANTS = sorted(n for n, (old, _) in MUTANTS.items()
                    if open(SRC).read().partition(MT_MARK)[2].count(old) == 1)


def test_threaded_mutants_exist():
    assert len(MT_MUTANTS) >= 5, MT_MUTANTS


@pytest.mark.parametrize("name", MT_MUTANTS)
def test_threaded_mutant_is_caught(tmp_path, name):
    import numpy as np
    import workloads
    old, new = MUTANTS[name]
    mutant = ctypes.CDLL(_build_mutant(tmp_path, name, old, new, part="threaded"))
    real = oracle.lib()
    for fn in ("oracle_allreduce_mt", "oracle_allgather_rank_major_mt", "oracle_allgather_param_contiguous_mt"):
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
        getattr(mutant, fn).restype = ctypes.c_int
    caught = False
    for dtype in ("bf16", "fp32", "int32"):
        ins = workloads.rank_buffers(4, 1001, dtype, "int" if dtype == "int32" else "normal", seed_base=77)
        st = [np.ascontiguousarray(a) for a in ins]
        ptrs = (ctypes.c_void_p * 4)(*[a.ctypes.data for a in st])
        out = np.empty(1001, dtype=st[0].dtype)
        mutant.oracle_allreduce_mt(ptrs, 4, 1001, oracle.DTYPES[dtype], out.ctypes.data, 2)
        caught |= not np.array_equal(out.view(np.uint8), oracle.allreduce(ins, dtype).view(np.uint8))
        out = np.empty(4 * 1001, dtype=st[0].dtype)
        mutant.oracle_allgather_rank_major_mt(ptrs, 4, 1001, oracle.ELEM_SIZE[dtype], out.ctypes.data, 2)
        caught |= not np.array_equal(out.view(np.uint8), oracle.allgather_rank_major(ins, dtype).view(np.uint8))
        splits = [300, 0, 701]
        sp = (ctypes.c_int64 * 3)(*splits)
        mutant.oracle_allgather_param_contiguous_mt(ptrs, 4, sp, 3, oracle.ELEM_SIZE[dtype], out.ctypes.data, 2)
        caught |= not np.array_equal(out.view(np.uint8),
                                     oracle.allgather_param_contiguous(ins, splits, dtype).view(np.uint8))
    # W = 1 over every bf16 pattern: the sum is the input itself, -0 included
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    one = (ctypes.c_void_p * 1)(allbits.ctypes.data)
    out = np.empty(1 << 16, dtype=np.uint16)
    mutant.oracle_allreduce_mt(one, 1, 1 << 16, oracle.DTYPES["bf16"], out.ctypes.data, 2)
    caught |= not np.array_equal(out, oracle.allreduce([allbits], "bf16"))
    assert caught, f"threaded mutant {name} gives the same bits as the definition"
