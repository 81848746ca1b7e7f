"""CPU oracle for the reduce and gather data movement of a custom collective.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The CUDA library and
its Python binding never import it; the oracle imports nothing from them.

The arithmetic lives in ``oracle.c`` (plain scalar C loops, one function per
definition; its header cites the passages each follows).  This module only
marshals numpy arrays into it.  Buffers are numpy arrays holding the raw
element bits: bf16 and fp16 as ``uint16``, fp32 as ``float32`` and int32 as
``int32``.

Parity status (each is pinned by tests/test_oracle_pins.py):
  * allreduce            -- pinned (closed forms, brute force, torch CPU chain,
                            rank-order counterexample, int32 wrap).
  * rank-major allgather -- pinned (torch.cat bytes, hand fixture).
  * param-contiguous AG  -- pinned (hand fixture from the layout formula,
                            permutation of rank-major, torch.cat per param).
  * element conversions  -- pinned (torch / numpy over exhaustive 16-bit
                            inputs and 2^24 random binary32 patterns).
"""
import ctypes
import numpy as np

from . import build as _build

DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2, "int32": 3}
NP_STORAGE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "int32": np.int32}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4, "int32": 4}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        l = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        l.oracle_allreduce.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64, ctypes.c_int, vp]
        l.oracle_allgather_rank_major.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64, ctypes.c_int, vp]
        l.oracle_allgather_param_contiguous.argtypes = [ctypes.POINTER(vp), ctypes.c_int,
                                                        ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                                        ctypes.c_int, vp]
        l.oracle_cast.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int64]
        i32 = ctypes.c_int
        l.oracle_allreduce_mt.argtypes = l.oracle_allreduce.argtypes + [i32]
        l.oracle_allgather_rank_major_mt.argtypes = l.oracle_allgather_rank_major.argtypes + [i32]
        l.oracle_allgather_param_contiguous_mt.argtypes = l.oracle_allgather_param_contiguous.argtypes + [i32]
        l.oracle_max_threads.argtypes = []
        for f in (l.oracle_allreduce, l.oracle_allgather_rank_major,
                  l.oracle_allgather_param_contiguous, l.oracle_cast, l.oracle_allreduce_mt,
                  l.oracle_allgather_rank_major_mt, l.oracle_allgather_param_contiguous_mt,
                  l.oracle_max_threads):
            f.restype = ctypes.c_int
        _lib = l
    return _lib


def _ptrs(arrays):
    arr = (ctypes.c_void_p * len(arrays))()
    for i, a in enumerate(arrays):
        assert a.flags["C_CONTIGUOUS"]
        arr[i] = a.ctypes.data
    return arr


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments")


def _as_storage(inputs, dtype):
    st = NP_STORAGE[dtype]
    out = []
    for a in inputs:
        a = np.ascontiguousarray(a)
        if a.dtype != st:
            if a.dtype.itemsize != np.dtype(st).itemsize:
                raise TypeError(f"{dtype} buffers must hold {np.dtype(st).itemsize}-byte elements")
            a = a.view(st)
        out.append(a.reshape(-1))
    return out


def allreduce(inputs, dtype):
    """Sum of the W rank buffers (fp32 accumulate in rank order 0..W-1, then
    round-to-nearest-even; int32 wraps).  Returns the one output every rank
    holds."""
    ins = _as_storage(inputs, dtype)
    n = ins[0].size
    assert all(a.size == n for a in ins)
    out = np.empty(n, dtype=NP_STORAGE[dtype])
    _check(lib().oracle_allreduce(_ptrs(ins), len(ins), n, DTYPES[dtype],
                                  out.ctypes.data if n else None), "allreduce")
    return out


def allgather_rank_major(inputs, dtype):
    """all_gather_into_tensor output: rank r's buffer at element r*N."""
    ins = _as_storage(inputs, dtype)
    n = ins[0].size
    assert all(a.size == n for a in ins)
    out = np.empty(n * len(ins), dtype=NP_STORAGE[dtype])
    _check(lib().oracle_allgather_rank_major(_ptrs(ins), len(ins), n, ELEM_SIZE[dtype],
                                             out.ctypes.data if out.size else None), "allgather")
    return out


def allgather_param_contiguous(inputs, splits, dtype):
    """FSDP [param][rank] output: rank r's piece of param s at O_s*W + r*E_s."""
    ins = _as_storage(inputs, dtype)
    splits = [int(s) for s in splits]
    total = sum(splits)
    assert all(a.size == total for a in ins)
    sp = (ctypes.c_int64 * max(1, len(splits)))(*splits)
    out = np.empty(total * len(ins), dtype=NP_STORAGE[dtype])
    _check(lib().oracle_allgather_param_contiguous(_ptrs(ins), len(ins), sp, len(splits),
                                                   ELEM_SIZE[dtype],
                                                   out.ctypes.data if out.size else None),
           "param-contiguous allgather")
    return out


def max_threads():
    """Host threads the multi-threaded entry points use by default (1 when
    the library was built without OpenMP)."""
    return int(lib().oracle_max_threads())


def allreduce_mt(inputs, dtype, threads=0):
    """allreduce() with the element range split over host threads: the same
    additions in the same order per element, so the same bits."""
    ins = _as_storage(inputs, dtype)
    n = ins[0].size
    assert all(a.size == n for a in ins)
    out = np.empty(n, dtype=NP_STORAGE[dtype])
    _check(lib().oracle_allreduce_mt(_ptrs(ins), len(ins), n, DTYPES[dtype],
                                     out.ctypes.data if n else None, int(threads)), "allreduce_mt")
    return out


def allgather_rank_major_mt(inputs, dtype, threads=0):
    """allgather_rank_major() with the copies split over host threads."""
    ins = _as_storage(inputs, dtype)
    n = ins[0].size
    assert all(a.size == n for a in ins)
    out = np.empty(n * len(ins), dtype=NP_STORAGE[dtype])
    _check(lib().oracle_allgather_rank_major_mt(_ptrs(ins), len(ins), n, ELEM_SIZE[dtype],
                                                out.ctypes.data if out.size else None, int(threads)),
           "allgather_mt")
    return out


def allgather_param_contiguous_mt(inputs, splits, dtype, threads=0):
    """allgather_param_contiguous() with the copies split over host threads."""
    ins = _as_storage(inputs, dtype)
    splits = [int(s) for s in splits]
    total = sum(splits)
    assert all(a.size == total for a in ins)
    sp = (ctypes.c_int64 * max(1, len(splits)))(*splits)
    out = np.empty(total * len(ins), dtype=NP_STORAGE[dtype])
    _check(lib().oracle_allgather_param_contiguous_mt(_ptrs(ins), len(ins), sp, len(splits),
                                                      ELEM_SIZE[dtype],
                                                      out.ctypes.data if out.size else None, int(threads)),
           "param-contiguous allgather_mt")
    return out


def f32_to(dtype, x):
    """binary32 array -> raw bits of bf16 / fp16 (round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(x.size, dtype=np.uint16)
    _check(lib().oracle_cast(x.ctypes.data, DTYPES["fp32"], out.ctypes.data, DTYPES[dtype], x.size), "cast")
    return out


def to_f32(dtype, bits):
    """raw bits of bf16 / fp16 -> binary32 array (exact)."""
    b = np.ascontiguousarray(bits).view(np.uint16).reshape(-1)
    out = np.empty(b.size, dtype=np.float32)
    _check(lib().oracle_cast(b.ctypes.data, DTYPES[dtype], out.ctypes.data, DTYPES["fp32"], b.size), "cast")
    return out
