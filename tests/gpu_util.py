"""Helpers for the GPU parity tests: device buffers built from the seeded
host arrays of workloads.py, guard canaries around every output, and bitwise
comparison with the oracle.  Host arrays carry raw element bits; device
tensors are filled by a bit copy, never by a float conversion."""
import numpy as np
import torch

import workloads

GUARD = 256          # canary bytes on each side of every output
CANARY = 0xA5


def _int_view(arr):
    return arr.view(np.int16) if arr.dtype.itemsize == 2 else arr.view(np.int32)


def to_device(arr, dtype, device="cuda"):
    """Host storage array -> CUDA tensor of the element type (bit copy)."""
    t = torch.from_numpy(np.ascontiguousarray(_int_view(np.ascontiguousarray(arr)))).to(device)
    return t.view(workloads.TORCH_DTYPE[dtype])


def to_host(t, dtype):
    """CUDA tensor -> host storage array (bit copy)."""
    it = torch.int16 if workloads.ELEM_BYTES[dtype] == 2 else torch.int32
    a = t.contiguous().view(it).cpu().numpy()
    return a.view(workloads.STORAGE[dtype])


class RankBuffers:
    """W device buffers of n elements each.

    layout "packed": one allocation, rank r at byte offset lead + r*stride,
    stride rounded up to 16 bytes, so that the pointers sit inside a larger
    allocation, not at its base.  layout "separate": one allocation per rank.
    """

    def __init__(self, W, n, dtype, layout="packed", lead=4096, device="cuda"):
        eb = workloads.ELEM_BYTES[dtype]
        self.W, self.n, self.dtype, self.eb = W, n, dtype, eb
        self.stride = ((n * eb + 15) // 16) * 16
        if layout == "packed":
            self.arena = torch.zeros(lead + W * self.stride + 64, dtype=torch.uint8, device=device)
            base = self.arena.data_ptr() + lead
            self.ptrs = [base + r * self.stride for r in range(W)]
            self._views = [self.arena[lead + r * self.stride: lead + r * self.stride + n * eb]
                           for r in range(W)]
        else:
            self._views = [torch.zeros(max(16, n * eb), dtype=torch.uint8, device=device)[: n * eb]
                           for _ in range(W)]
            self.arena = None
            self.ptrs = [v.data_ptr() for v in self._views]

    def fill(self, arrays):
        for v, a in zip(self._views, arrays):
            if a.size:
                v.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8)).to(v.device))

    def host(self, r):
        return self._views[r].cpu().numpy().view(workloads.STORAGE[self.dtype])


class GuardedOutputs:
    """W output buffers of n_out elements (None for ranks not materialised),
    each with GUARD canary bytes before and after."""

    def __init__(self, W, n_out, dtype, materialise=None, device="cuda"):
        eb = workloads.ELEM_BYTES[dtype]
        self.dtype, self.eb, self.n_out = dtype, eb, n_out
        materialise = range(W) if materialise is None else materialise
        self.bufs = []
        for r in range(W):
            if r in materialise:
                t = torch.full((2 * GUARD + n_out * eb,), CANARY, dtype=torch.uint8, device=device)
                self.bufs.append(t)
            else:
                self.bufs.append(None)
        self.ptrs = [None if t is None else t.data_ptr() + GUARD for t in self.bufs]

    def poison(self, byte=0x5A):
        for t in self.bufs:
            if t is not None:
                t[GUARD: GUARD + self.n_out * self.eb].fill_(byte)

    def host(self, r):
        t = self.bufs[r]
        return t[GUARD: GUARD + self.n_out * self.eb].cpu().numpy().view(workloads.STORAGE[self.dtype])

    def check_guards(self):
        for r, t in enumerate(self.bufs):
            if t is None:
                continue
            head = t[:GUARD].cpu().numpy()
            tail = t[GUARD + self.n_out * self.eb:].cpu().numpy()
            assert (head == CANARY).all() and (tail == CANARY).all(), f"output {r}: guard bytes overwritten"


def bits(a):
    a = np.asarray(a)
    return a.view({2: np.uint16, 4: np.uint32}[a.dtype.itemsize])


def assert_bitwise(got, want, what=""):
    g, w = bits(got), bits(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.nonzero(g != w)[0]
    assert bad.size == 0, f"{what}: {bad.size} of {g.size} elements differ; first {bad[:8].tolist()} got {g[bad[:4]].tolist()} want {w[bad[:4]].tolist()}"
