"""Reduce and gather data movement of a custom collective, native to GB300.

W ranks are emulated on one GPU: their registered buffers are plain device
buffers in this GPU's HBM.  The work runs in hand-written sm_103a kernels in
librr.so behind the C ABI of include/rr.h: one-shot and two-shot allreduce,
rank-major allgather_into_tensor, the list-output all_gather, the FSDP
param-contiguous allgather, and the signal pad of generation flags that
orders the ranks' blocks.  This package is the thin Python binding of that library (argument marshalling
only); PyTorch serves for device memory and streams.
"""
from ._binding import (  # noqa: F401
    LIB_PATH, OPTIONS, RR_BARRIER_ARRIVE, RR_BARRIER_END, RR_BARRIER_MID, RR_BARRIER_STAGE, RR_BF16,
    RR_ERR_ALIAS, RR_ERR_ALIGNMENT, RR_ERR_CUDA, RR_ERR_INVALID_ARG, RR_ERR_TIMEOUT,
    RR_ERR_TOO_MANY_BLOCKS, RR_ERR_UNSUPPORTED_DTYPE, RR_ERR_WRONG_DEVICE, RR_FP16, RR_FP32, RR_INT32,
    RR_MAX_SPLITS, RR_MAX_WORLD, RR_OK, RRError, SignalPad, bound_call, dtype_code, lib,
    pointer_array, rr_allgather, rr_allgather_list, rr_allgather_param_contiguous, rr_allreduce_oneshot,
    rr_allreduce_oneshot_noalloc, rr_allreduce_oneshot_noalloc_status, rr_allreduce_twoshot,
    rr_signal_pad_create, rr_signal_pad_destroy, rr_signal_pad_status, stream_handle,
)
