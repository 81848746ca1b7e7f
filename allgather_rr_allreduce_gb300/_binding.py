"""ctypes binding of librr.so (include/rr.h).  Argument marshalling only.

Every function has the C name and the C argument order.  Device buffers may
be given as integers (device addresses) or as CUDA tensors (their data
pointer is used); dtypes as rr_dtype codes, "bf16"/"fp16"/"fp32"/"int32" or
torch dtypes; streams as integers, torch.cuda.Stream objects, or None for
torch's current stream.  A non-zero rr_status raises RRError.  Nothing here
computes: if librr.so is missing, every call raises.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librr.so")

RR_BF16, RR_FP16, RR_FP32, RR_INT32 = 0, 1, 2, 3
RR_OK = 0
STATUS_NAMES = {
    0: "RR_OK", 1: "RR_ERR_INVALID_ARG", 2: "RR_ERR_UNSUPPORTED_DTYPE", 3: "RR_ERR_ALIGNMENT",
    4: "RR_ERR_ALIAS", 5: "RR_ERR_TOO_MANY_BLOCKS", 6: "RR_ERR_CUDA", 7: "RR_ERR_TIMEOUT",
    8: "RR_ERR_WRONG_DEVICE",
}
RR_ERR_INVALID_ARG, RR_ERR_UNSUPPORTED_DTYPE, RR_ERR_ALIGNMENT, RR_ERR_ALIAS = 1, 2, 3, 4
RR_ERR_TOO_MANY_BLOCKS, RR_ERR_CUDA, RR_ERR_TIMEOUT, RR_ERR_WRONG_DEVICE = 5, 6, 7, 8
RR_BARRIER_ARRIVE, RR_BARRIER_STAGE, RR_BARRIER_MID, RR_BARRIER_END = 0, 1, 2, 3
RR_MAX_WORLD, RR_MAX_SPLITS = 16, 256

OPTIONS = {
    "timeout_ns": 0, "blocks_per_rank": 1, "gather_engine": 2, "inject_skip": 3, "round_bytes": 4,
    "reduce_engine": 5, "twoshot_mode": 6, "device_generation": 7, "debug_iterations": 8,
    "debug_skew_ns": 9,
    "generation": 16, "last_grid": 17, "last_blocks_per_rank": 18, "last_engine": 19,
    "world_size": 20, "max_blocks_per_rank": 21,
}
_DTYPE_NAMES = {"bf16": RR_BF16, "fp16": RR_FP16, "fp32": RR_FP32, "int32": RR_INT32}


class RRError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


_lib = None
_vp = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)


def lib():
    """Load librr.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with allgather_rr_allreduce_gb300.build.build()")
        l = ctypes.CDLL(LIB_PATH)
        i32, i64, u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
        sig = {
            "rr_signal_pad_create": [i32, i32, u64, ctypes.POINTER(_vp)],
            "rr_signal_pad_destroy": [_vp],
            "rr_signal_pad_status": [_vp, _vp],
            "rr_signal_pad_timeout_info": [_vp, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                           ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_uint32)],
            "rr_signal_pad_set_option": [_vp, i32, i64],
            "rr_signal_pad_get_option": [_vp, i32, ctypes.POINTER(i64)],
            "rr_allreduce_oneshot": [_PP, _PP, _PP, i32, i64, i32, i32, _vp, _vp],
            "rr_allreduce_twoshot": [_PP, _PP, _PP, i32, i64, i32, i32, _vp, _vp],
            "rr_allgather": [_PP, _PP, i32, i64, i32, _vp, _vp],
            "rr_allgather_param_contiguous": [_PP, _PP, i32, ctypes.POINTER(i64), i32, i32, _vp, _vp],
            "rr_allgather_list": [_PP, _PP, i32, i64, i32, _vp, _vp],
            "rr_allreduce_oneshot_noalloc": [_PP, _PP, _PP, i32, i64, i32, i32, _vp],
            "rr_allreduce_oneshot_noalloc_status": [_vp],
        }
        for name, args in sig.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        l.rr_status_string.argtypes = [ctypes.c_int]
        l.rr_status_string.restype = ctypes.c_char_p
        l.rr_last_error.argtypes = []
        l.rr_last_error.restype = ctypes.c_char_p
        _lib = l
    return _lib


def _check(status):
    if status != RR_OK:
        raise RRError(status, lib().rr_last_error().decode(errors="replace"))


def _addr(x):
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if getattr(x, "is_cuda", True) is False:
            raise ValueError("device buffers must be CUDA tensors or device addresses")
        return x.data_ptr()
    raise TypeError(f"cannot take a device address from {type(x)!r}")


def pointer_array(items):
    """Host array of device addresses (NULL for None)."""
    arr = (ctypes.c_void_p * len(items))()
    for i, x in enumerate(items):
        arr[i] = _addr(x) or None
    return arr


def dtype_code(dtype):
    if isinstance(dtype, int):
        return dtype
    if isinstance(dtype, str):
        return _DTYPE_NAMES[dtype]
    import torch
    return {torch.bfloat16: RR_BF16, torch.float16: RR_FP16, torch.float32: RR_FP32,
            torch.int32: RR_INT32}[dtype]


def stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class SignalPad:
    """Owner of an rr_signal_pad*.  close() (or garbage collection) destroys it."""

    def __init__(self, handle, world_size):
        self.handle = handle
        self.world_size = world_size

    @property
    def _as_parameter_(self):
        return ctypes.c_void_p(self.handle)

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check(lib().rr_signal_pad_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def status(self, stream=None):
        """rr_signal_pad_status: synchronise the stream, raise RRError on a recorded timeout."""
        _check(lib().rr_signal_pad_status(self.handle, stream_handle(stream)))

    def timeout_info(self):
        b, r, k = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        g = ctypes.c_uint32()
        _check(lib().rr_signal_pad_timeout_info(self.handle, ctypes.byref(b), ctypes.byref(r),
                                                ctypes.byref(k), ctypes.byref(g)))
        return {"barrier": b.value, "rank": r.value, "block": k.value, "generation": g.value}

    def set_option(self, name, value):
        _check(lib().rr_signal_pad_set_option(self.handle, OPTIONS[name], int(value)))

    def get_option(self, name):
        v = ctypes.c_int64()
        _check(lib().rr_signal_pad_get_option(self.handle, OPTIONS[name], ctypes.byref(v)))
        return v.value


def rr_signal_pad_create(world_size, max_blocks_per_rank=0, timeout_ns=0):
    h = ctypes.c_void_p()
    _check(lib().rr_signal_pad_create(world_size, max_blocks_per_rank, timeout_ns, ctypes.byref(h)))
    return SignalPad(h.value, world_size)


def rr_signal_pad_destroy(pad):
    pad.close()


def rr_signal_pad_status(pad, stream=None):
    pad.status(stream)


def _pad_handle(pad):
    return pad.handle if isinstance(pad, SignalPad) else pad


def rr_allreduce_oneshot(inputs, rank_bufs, outputs, world_size, numel, dtype, copy_mode, pad,
                         stream=None):
    ins = pointer_array(inputs) if inputs is not None else None
    _check(lib().rr_allreduce_oneshot(ins, pointer_array(rank_bufs), pointer_array(outputs),
                                      world_size, numel, dtype_code(dtype), int(bool(copy_mode)),
                                      _pad_handle(pad), stream_handle(stream)))


def rr_allreduce_twoshot(inputs, rank_bufs, outputs, world_size, numel, dtype, copy_mode, pad,
                         stream=None):
    ins = pointer_array(inputs) if inputs is not None else None
    _check(lib().rr_allreduce_twoshot(ins, pointer_array(rank_bufs), pointer_array(outputs),
                                      world_size, numel, dtype_code(dtype), int(bool(copy_mode)),
                                      _pad_handle(pad), stream_handle(stream)))


def rr_allreduce_oneshot_noalloc(inputs, rank_bufs, outputs, world_size, numel, dtype, copy_mode,
                                 stream=None):
    """The one-shot allreduce without a pad (the library's static signal array)."""
    ins = pointer_array(inputs) if inputs is not None else None
    _check(lib().rr_allreduce_oneshot_noalloc(ins, pointer_array(rank_bufs), pointer_array(outputs),
                                              world_size, numel, dtype_code(dtype),
                                              int(bool(copy_mode)), stream_handle(stream)))


def rr_allreduce_oneshot_noalloc_status(stream=None):
    """Synchronise the stream; raise RRError if the last allocation-free call timed out."""
    _check(lib().rr_allreduce_oneshot_noalloc_status(stream_handle(stream)))


def rr_allgather(rank_bufs, outputs, world_size, numel_per_rank, dtype, pad, stream=None):
    _check(lib().rr_allgather(pointer_array(rank_bufs), pointer_array(outputs), world_size,
                              numel_per_rank, dtype_code(dtype), _pad_handle(pad),
                              stream_handle(stream)))


def rr_allgather_param_contiguous(rank_bufs, outputs, world_size, split_sizes, dtype, pad,
                                  stream=None):
    n = len(split_sizes)
    sp = (ctypes.c_int64 * max(1, n))(*[int(s) for s in split_sizes])
    _check(lib().rr_allgather_param_contiguous(pointer_array(rank_bufs), pointer_array(outputs),
                                               world_size, sp, n, dtype_code(dtype),
                                               _pad_handle(pad), stream_handle(stream)))


def rr_allgather_list(rank_bufs, output_lists, world_size, numel_per_rank, dtype, pad, stream=None):
    """output_lists: W entries, each a list of W device buffers (rank q's
    all_gather tensor_list) or None (not materialised)."""
    flat = []
    for row in output_lists:
        flat.extend([None] * world_size if row is None else list(row))
    _check(lib().rr_allgather_list(pointer_array(rank_bufs), pointer_array(flat), world_size,
                                   numel_per_rank, dtype_code(dtype), _pad_handle(pad),
                                   stream_handle(stream)))


def bound_call(name, *args):
    """Marshal the arguments of one C entry point once and return a
    zero-argument callable that re-issues the call (for back-to-back issue
    where per-call Python marshalling would dominate).  Arguments are given
    in the C order, already in C form except for pointer lists, dtypes,
    pads and streams, which are converted here."""
    fn = getattr(lib(), name)
    conv = []
    for a in args:
        if isinstance(a, (list, tuple)):
            conv.append(pointer_array(a))
        elif isinstance(a, SignalPad):
            conv.append(a.handle)
        else:
            conv.append(a)
    l = lib()

    def call():
        st = fn(*conv)
        if st != RR_OK:
            raise RRError(st, l.rr_last_error().decode(errors="replace"))
    return call
