"""Benchmark of the reduce/gather hot path on one GB300 (W ranks emulated in
its HBM), printing one JSON line.

A step is one pass of the whole hot path over the large workload (W=8, bf16,
2^24 elements = 32 MiB per rank, N(0,1)), one launch per op:
  oneshot_copy_off   one-shot allreduce, registered buffers, rank 0's output
  oneshot_copy_on    one-shot allreduce, inputs staged in-kernel, rank 0's output
  twoshot_copy_off   two-shot allreduce, all W outputs
  twoshot_copy_on    two-shot allreduce with in-kernel staging, all W outputs
  allgather          rank-major all_gather_into_tensor, rank 0's output
  allgather_pc       param-contiguous (FSDP) allgather of one transformer layer
                     (hidden 3584 / kv 512 / ffn 18944, W=8), rank 0's output
value = algorithmic bytes of the step / device time of the step (GB/s).
Algorithmic bytes of an op = every byte that exists before the call and must
be read once, plus every byte written (re-reads of data written earlier in
the same call are not counted).  Each op has its own buffers (>= 288 MiB per
op, more than the 129 MB L2), so no op starts with its inputs in L2.

--impl reference times the CPU oracle (the plain definition of every op) on
the host on a sample of the same workload and reports the same metric.
Under torchrun each rank runs an independent replica (the path does not
shard over GPUs); the time is the max over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "achieved HBM GB/s and % of 8 TB/s roofline per op vs bytes/rank; small-msg µs"
NOMINAL_HBM_GBS = 8000.0
W, N = workloads.LARGE["W"], workloads.LARGE["N"]
EB = 2
OP_NAMES = ("oneshot_copy_off", "oneshot_copy_on", "twoshot_copy_off", "twoshot_copy_on",
            "allgather", "allgather_pc")


GATHER_ENGINES = ("auto", "ldst", "tma", "copy_engine")  # pad option gather_engine 0..3


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def code_tokens(text):
    """C/C++/CUDA source with comments removed and whitespace runs collapsed
    (string and character literals kept as written), so that editing a
    comment leaves the hash of the code unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash():
    """Hash of the kernel sources' code (comments and layout ignored)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "allgather_rr_allreduce_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_op):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("csrc_sha256_16") != source_hash():
        return None
    ent = d.get("ops", {}).get(kernel_op)
    return None if ent is None else ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 50 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except (OSError, ValueError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxes, reasons = [], [], set()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "samples": len(sms),
                "reasons": sorted(reasons)}


def max_over_ranks(x, world):
    """Max of a float over all ranks of the default process group (NCCL or
    gloo); x itself when there is one rank."""
    if world <= 1:
        return float(x)
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


# ---------------------------------------------------------------------- GPU arm

class Step:
    """Device buffers and pre-marshalled C calls of one step (all ops, or the
    subset `ops`; `n` elements per rank for the allreduce / allgather ops and
    the FSDP layer's splits divided by `pc_div`)."""

    def __init__(self, rr, stream, seed, ops=OP_NAMES, n=N, pc_div=1):
        import ctypes
        self.rr = rr
        self.stream = stream
        self.ops = tuple(ops)
        self.n = n
        dev = "cuda"
        g = torch.Generator(device=dev).manual_seed(seed)

        def ranks():
            return torch.randn((W, n), generator=g, device=dev).to(torch.bfloat16)

        def empty(*shape):
            return torch.empty(shape, dtype=torch.bfloat16, device=dev)

        def rows(t):
            return [t[r].data_ptr() for r in range(W)]

        def only0(t):
            return [t.data_ptr()] + [None] * (W - 1)

        self.pad = rr.rr_signal_pad_create(W)
        sh = stream.cuda_stream
        bf16 = rr.RR_BF16
        bc = rr.bound_call
        self.splits = [e // pc_div for e in workloads.shard_sizes(workloads.FSDP_LAYER_PARAMS, W)]
        S = sum(self.splits)
        self.pc_shard_bytes = S * EB
        self._sp = (ctypes.c_int64 * len(self.splits))(*self.splits)
        self.calls, ins, outs = {}, [], []
        for op in self.ops:
            if op == "oneshot_copy_off":
                x, y = ranks(), empty(n)
                self.calls[op] = bc("rr_allreduce_oneshot", None, rows(x), only0(y), W, n, bf16, 0, self.pad, sh)
            elif op == "oneshot_copy_on":
                x, reg, y = ranks(), empty(W, n), empty(n)
                self.calls[op] = bc("rr_allreduce_oneshot", rows(x), rows(reg), only0(y), W, n, bf16, 1,
                                    self.pad, sh)
            elif op == "twoshot_copy_off":
                x, y = ranks(), empty(W, n)
                self.calls[op] = bc("rr_allreduce_twoshot", None, rows(x), rows(y), W, n, bf16, 0, self.pad, sh)
            elif op == "twoshot_copy_on":
                x, reg, y = ranks(), empty(W, n), empty(W, n)
                self.calls[op] = bc("rr_allreduce_twoshot", rows(x), rows(reg), rows(y), W, n, bf16, 1,
                                    self.pad, sh)
            elif op == "allgather":
                x, y = ranks(), empty(W * n)
                self.calls[op] = bc("rr_allgather", rows(x), only0(y), W, n, bf16, self.pad, sh)
            elif op == "allgather_pc":
                x = (torch.randn((W, S), generator=g, device=dev) * 0.02).to(torch.bfloat16)
                y = empty(W * S)
                self.calls[op] = bc("rr_allgather_param_contiguous", rows(x), only0(y), W, self._sp,
                                    len(self.splits), bf16, self.pad, sh)
            else:
                raise ValueError(f"unknown op {op}")
            ins.append(x)
            outs.append(y)
        self._bufs = (ins, outs)
        # host-side copies for the end-to-end measurement
        self.e2e_pairs_in = [(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for t in ins]
        for d, h in self.e2e_pairs_in:
            h.copy_(d)
        self.e2e_pairs_out = [(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for t in outs]

    def bytes_by_op(self):
        nb = self.n * EB
        full = {
            "oneshot_copy_off": W * nb + nb,            # read W buffers, write rank 0's output
            "oneshot_copy_on": W * nb + W * nb + nb,    # + stage W inputs into the registered buffers
            "twoshot_copy_off": W * nb + W * nb,        # read W buffers, write W outputs
            "twoshot_copy_on": W * nb + W * nb + W * nb,
            "allgather": W * nb + W * nb,               # read W shards, write one W*N output
            "allgather_pc": 2 * W * self.pc_shard_bytes,
        }
        return {op: full[op] for op in self.ops}

    def run(self, events=None, only=None):
        """One step.  events[i] = (start, end) pair recorded around op i
        (every op, or only op index `only`)."""
        for i, name in enumerate(self.ops):
            timed = events is not None and (only is None or i == only)
            if timed:
                events[i][0].record(self.stream)
            self.calls[name]()
            if timed:
                events[i][1].record(self.stream)

    def run_e2e(self):
        """One step end to end on one stream: every op's inputs host->device,
        the step, every output device->host."""
        for d, h in self.e2e_pairs_in:
            d.copy_(h, non_blocking=True)
        self.run()
        for d, h in self.e2e_pairs_out:
            h.copy_(d, non_blocking=True)

    def e2e_bytes(self):
        bi = sum(h.numel() * h.element_size() for _, h in self.e2e_pairs_in)
        bo = sum(h.numel() * h.element_size() for _, h in self.e2e_pairs_out)
        return bi, bo


def run_e2e_pipelined(sets, steps, start):
    """`steps` end-to-end steps, alternating between the Step objects in
    `sets` (two identical sets of device and pinned host buffers, calls on
    the same compute stream), with the host<->device copies on their own
    streams: while step k computes and its outputs travel device->host, the
    inputs of step k+1 travel host->device into the other set (the link is
    full duplex).  Events keep each set's buffers safe: its inputs are
    overwritten only after its previous step has read them, and its outputs
    only after they have been copied out.  Every step copies all its inputs
    in and all its outputs out.  Returns the event recorded on the compute
    stream after the last copy out."""
    compute = sets[0].stream
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    cin.wait_event(start)
    done_compute = [None] * len(sets)
    done_out = [None] * len(sets)
    last = None
    for k in range(steps):
        i = k % len(sets)
        st = sets[i]
        if done_compute[i] is not None:
            cin.wait_event(done_compute[i])
        with torch.cuda.stream(cin):
            for d, h in st.e2e_pairs_in:
                d.copy_(h, non_blocking=True)
        arrived = torch.cuda.Event()
        arrived.record(cin)
        compute.wait_event(arrived)
        if done_out[i] is not None:
            compute.wait_event(done_out[i])
        st.run()
        done_compute[i] = torch.cuda.Event()
        done_compute[i].record(compute)
        cout.wait_event(done_compute[i])
        with torch.cuda.stream(cout):
            for d, h in st.e2e_pairs_out:
                h.copy_(d, non_blocking=True)
        done_out[i] = last = torch.cuda.Event()
        last.record(cout)
    compute.wait_event(last)
    end = torch.cuda.Event(enable_timing=True)
    end.record(compute)
    return end


def latency_sweep(rr, stream, reps=1000, batch=250):
    """Small messages, W=8, bf16, one-shot and two-shot, all W outputs, `reps`
    back-to-back calls on one pad.  Calls are queued behind a sleep kernel so
    the events time the GPU executing them back to back (not host issue)."""
    pad = rr.rr_signal_pad_create(W)
    sh = stream.cuda_stream
    out = {"oneshot": {}, "twoshot": {}, "issue_bound_oneshot": {}}
    g = torch.Generator(device="cuda").manual_seed(workloads.LATENCY["seed_base"])
    for nbytes in workloads.LATENCY["bytes_per_rank"]:
        n = nbytes // EB
        x = (torch.rand((W, n), generator=g, device="cuda") * 2 - 1).to(torch.bfloat16)
        y = torch.empty((W, n), dtype=torch.bfloat16, device="cuda")
        rows_x = [x[r].data_ptr() for r in range(W)]
        rows_y = [y[r].data_ptr() for r in range(W)]
        for algo in ("oneshot", "twoshot"):
            call = rr.bound_call(f"rr_allreduce_{algo}", None, rows_x, rows_y, W, n, rr.RR_BF16, 0, pad, sh)
            for _ in range(20):
                call()
            total_ms = 0.0
            with torch.cuda.stream(stream):
                for _ in range(reps // batch):
                    torch.cuda._sleep(20_000_000)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(batch):
                        call()
                    e1.record(stream)
                    e1.synchronize()
                    total_ms += e0.elapsed_time(e1)
            out[algo][str(nbytes)] = round(1000.0 * total_ms / reps, 3)
            if algo == "oneshot":
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                stream.synchronize()
                e0.record(stream)
                for _ in range(reps):
                    call()
                e1.record(stream)
                e1.synchronize()
                out["issue_bound_oneshot"][str(nbytes)] = round(1000.0 * e0.elapsed_time(e1) / reps, 3)
    pad.status(stream)
    pad.close()
    out.update(graph_latency(rr, stream, batch=batch))
    return out


def small_config_latency(rr, stream, reps=1000):
    """The small workload (W=2, bf16, 4096 elements per rank, U[-1,1]):
    one-shot allreduce and rank-major allgather into rank 0's output, GPU
    time per call over `reps` back-to-back calls queued behind a sleep."""
    cfg = workloads.SMALL
    W2, n = cfg["W"], cfg["N"]
    g = torch.Generator(device="cuda").manual_seed(cfg["seed_base"])
    x = (torch.rand((W2, n), generator=g, device="cuda") * 2 - 1).to(torch.bfloat16)
    y = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    z = torch.empty(W2 * n, dtype=torch.bfloat16, device="cuda")
    pad = rr.rr_signal_pad_create(W2)
    sh = stream.cuda_stream
    rows = [x[r].data_ptr() for r in range(W2)]
    calls = {"oneshot_allreduce": rr.bound_call("rr_allreduce_oneshot", None, rows, [y.data_ptr(), None], W2, n,
                                                rr.RR_BF16, 0, pad, sh),
             "allgather": rr.bound_call("rr_allgather", rows, [z.data_ptr(), None], W2, n, rr.RR_BF16, pad, sh)}
    out = {"workload": cfg["name"]}
    for name, call in calls.items():
        for _ in range(20):
            call()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(20_000_000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                call()
            e1.record(stream)
        e1.synchronize()
        out[f"{name}_us"] = round(1000.0 * e0.elapsed_time(e1) / reps, 3)
    pad.status(stream)
    pad.close()
    return out


def graph_latency(rr, stream, batch=250, reps=3):
    """The same calls captured in a CUDA graph (pad with the device-resident
    generation counter), replayed back to back: GPU time per call."""
    res = {"graph_oneshot": {}, "graph_twoshot": {}}
    pad = rr.rr_signal_pad_create(W)
    pad.set_option("device_generation", 1)
    g = torch.Generator(device="cuda").manual_seed(workloads.LATENCY["seed_base"] + 1)
    for nbytes in workloads.LATENCY["bytes_per_rank"]:
        n = nbytes // EB
        x = (torch.rand((W, n), generator=g, device="cuda") * 2 - 1).to(torch.bfloat16)
        y = torch.empty((W, n), dtype=torch.bfloat16, device="cuda")
        rows_x = [x[r].data_ptr() for r in range(W)]
        rows_y = [y[r].data_ptr() for r in range(W)]
        for algo in ("oneshot", "twoshot"):
            fn = getattr(rr, f"rr_allreduce_{algo}")
            with torch.cuda.stream(stream):
                fn(None, rows_x, rows_y, W, n, "bf16", 0, pad, stream)
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                cs = torch.cuda.current_stream()
                for _ in range(batch):
                    fn(None, rows_x, rows_y, W, n, "bf16", 0, pad, cs)
            graph.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    graph.replay()
                e1.record(stream)
            e1.synchronize()
            res[f"graph_{algo}"][str(nbytes)] = round(1000.0 * e0.elapsed_time(e1) / (reps * batch), 3)
            del graph
    pad.status(stream)
    pad.close()
    return res


def ops_alone(step, reps=50):
    """Each op of the step on its own: `reps` back-to-back calls on the op's
    buffers (inputs larger than L2) between one pair of events, so each call
    also absorbs only its own predecessor's L2 write-back."""
    out = {}
    bytes_by_op = step.bytes_by_op()
    for name in step.ops:
        call = step.calls[name]
        for _ in range(5):
            call()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(step.stream)
        for _ in range(reps):
            call()
        e1.record(step.stream)
        e1.synchronize()
        us = 1000.0 * e0.elapsed_time(e1) / reps
        gbs = bytes_by_op[name] / us / 1e3
        out[name] = {"us": round(us, 2), "GBps": round(gbs, 1), "pct_of_8TBps": round(100 * gbs / NOMINAL_HBM_GBS, 2)}
    step.pad.status(step.stream)
    return out


def ag_sweep_dtypes(rr, stream, sizes=(1 << 20, 1 << 25, 1 << 29)):
    """The rank-major allgather at a few sizes per rank for every dtype
    (W=8, rank 0's output, 10 back-to-back calls each): the copy moves raw
    bytes, so the dtype should not matter."""
    pad = rr.rr_signal_pad_create(W)
    sh = stream.cuda_stream
    out = {}
    for dtype in ("bf16", "fp16", "fp32", "int32"):
        eb = workloads.ELEM_BYTES[dtype]
        tdt = workloads.TORCH_DTYPE[dtype]
        for nbytes in sizes:
            n = nbytes // eb
            x = torch.empty((W, n), dtype=tdt, device="cuda")
            y = torch.empty(W * n, dtype=tdt, device="cuda")
            call = rr.bound_call("rr_allgather", [x[r].data_ptr() for r in range(W)],
                                 [y.data_ptr()] + [None] * (W - 1), W, n, rr.dtype_code(dtype), pad, sh)
            call()
            count = 40 if nbytes < (1 << 24) else 10
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(count):
                call()
            e1.record(stream)
            e1.synchronize()
            us = 1000.0 * e0.elapsed_time(e1) / count
            out[f"{dtype}_{nbytes}"] = {"us": round(us, 2), "GBps": round(2 * W * nbytes / us / 1e3, 1)}
            del x, y
    pad.status(stream)
    pad.close()
    torch.cuda.empty_cache()
    return out


def ag_sweep(rr, stream):
    """Rank-major allgather, W=8, bf16, 1 KiB .. 512 MiB per rank (powers of
    two), rank 0's output: GPU time per call, back to back.  Small sizes
    rotate through several buffer sets (up to 64) so that consecutive calls
    touch different memory; a size whose rotated sets span less than twice
    the L2 is marked l2_resident (its GB/s is not an HBM figure)."""
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    pad = rr.rr_signal_pad_create(W)
    sh = stream.cuda_stream
    out = {}
    for nbytes in workloads.AG_SWEEP["bytes_per_rank"]:
        n = nbytes // EB
        foot = 2 * W * nbytes
        sets = max(1, min(64, -(-4 * l2 // foot)))
        bufs = [(torch.empty((W, n), dtype=torch.bfloat16, device="cuda"),
                 torch.empty(W * n, dtype=torch.bfloat16, device="cuda")) for _ in range(sets)]
        calls = [rr.bound_call("rr_allgather", [x[r].data_ptr() for r in range(W)],
                               [y.data_ptr()] + [None] * (W - 1), W, n, rr.RR_BF16, pad, sh)
                 for x, y in bufs]
        count = 400 if nbytes <= (1 << 20) else (60 if nbytes <= (64 << 20) else 10)
        count = max(count, sets)
        for _ in range(1 if nbytes <= (64 << 20) else 3):  # fresh buffers: warm them first
            for c in calls:
                c()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(20_000_000)
            e0.record(stream)
            for i in range(count):
                calls[i % sets]()
            e1.record(stream)
        e1.synchronize()
        us = 1000.0 * e0.elapsed_time(e1) / count
        gbs = 2 * W * nbytes / us / 1e3
        out[str(nbytes)] = {"us": round(us, 2), "GBps": round(gbs, 1),
                            "pct_of_8TBps": round(100 * gbs / NOMINAL_HBM_GBS, 2),
                            "l2_resident": sets * foot < 2 * l2}
        del calls, bufs
    pad.status(stream)
    pad.close()
    torch.cuda.empty_cache()
    return out


class FsdpLayers:
    """28 param-contiguous allgathers back to back, one per layer, rank 0's
    output.  All layers' shards sit in one tensor and all outputs in another
    (about 13 GB each)."""

    def __init__(self, rr, stream):
        import ctypes
        cfg = workloads.FSDP_LAYER
        self.L = cfg["layers"]
        self.stream = stream
        self.splits = workloads.shard_sizes(workloads.FSDP_LAYER_PARAMS, W)
        self.S = sum(self.splits)
        self.pad = rr.rr_signal_pad_create(W)
        g = torch.Generator(device="cuda").manual_seed(cfg["seed_base"])
        self._sp = (ctypes.c_int64 * len(self.splits))(*self.splits)
        self.X = torch.empty((self.L, W, self.S), dtype=torch.bfloat16, device="cuda")
        for l in range(self.L):
            self.X[l].copy_((torch.randn((W, self.S), generator=g, device="cuda") * cfg["sigma"]).to(torch.bfloat16))
        self.Y = torch.empty((self.L, W * self.S), dtype=torch.bfloat16, device="cuda")
        self.calls = [rr.bound_call("rr_allgather_param_contiguous", [self.X[l, r].data_ptr() for r in range(W)],
                                    [self.Y[l].data_ptr()] + [None] * (W - 1), W, self._sp, len(self.splits),
                                    rr.RR_BF16, self.pad, stream.cuda_stream) for l in range(self.L)]
        # the shards are drawn on the default stream; the gathers run on `stream`
        torch.cuda.synchronize()

    def one_pass(self, per_layer=False):
        L, stream = self.L, self.stream
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(L + 1)]
        evs[0].record(stream)
        for i, c in enumerate(self.calls):
            c()
            if per_layer or i == L - 1:
                evs[i + 1].record(stream)
        evs[-1].synchronize()
        per = [1000 * evs[i].elapsed_time(evs[i + 1]) for i in range(L)] if per_layer else None
        return evs[0].elapsed_time(evs[-1]), per

    def measure(self):
        # A training step gathers the same persistent buffers every step: the
        # figure is the steady state after 8 untimed passes; the first pass
        # over the fresh layers is reported beside it.
        L = self.L
        first, first_per = self.one_pass(True)
        for _ in range(8):
            self.one_pass()
        ms = min(self.one_pass()[0] for _ in range(4))
        _, steady_per = self.one_pass(True)
        self.pad.status(self.stream)
        total = L * 2 * W * self.S * EB
        return {"ms": round(ms, 4), "GBps": round(total / ms / 1e6, 1), "bytes": total,
                "pct_of_8TBps": round(100 * total / ms / 1e6 / NOMINAL_HBM_GBS, 2),
                "us_per_layer": round(1000 * ms / L, 2),
                "first_pass_us_per_layer": round(1000 * first / L, 2),
                "first_pass_first_layer_us": round(first_per[0], 1),
                "first_pass_other_layers_us_median": round(statistics.median(first_per[1:]), 1),
                "steady_layer_us_min_median_max": [round(min(steady_per), 1), round(statistics.median(steady_per), 1),
                                                   round(max(steady_per), 1)],
                "how": "steady state: best of 4 passes after 8 untimed passes over the 28 layers; per-layer "
                       "figures from one more pass with an event pair around every layer"}

    def close(self):
        self.pad.close()
        del self.X, self.Y, self.calls
        torch.cuda.empty_cache()


def overlap_gemm(rr, stream, n_ag=40, mkn=8192):
    """Rank-major allgather (W=8, 32 MiB bf16 per rank, rank 0's output) on
    every gather engine, alone and while cuBLAS bf16 GEMMs (mkn^3) run on a
    second stream: does the gather slow down when it shares the GPU with
    compute, and by how much does it slow the GEMMs?  The copy engines take
    no SM.  Per engine: n_ag gathers; the GEMM count is chosen so that both
    streams are busy for about the same time."""
    n = N
    g = torch.Generator(device="cuda").manual_seed(workloads.LARGE["seed_base"] + 5)
    x = torch.randn((W, n), generator=g, device="cuda").to(torch.bfloat16)
    y = torch.empty(W * n, dtype=torch.bfloat16, device="cuda")
    a = torch.randn((mkn, mkn), generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn((mkn, mkn), generator=g, device="cuda").to(torch.bfloat16)
    c = torch.empty((mkn, mkn), dtype=torch.bfloat16, device="cuda")
    gs = torch.cuda.Stream()
    pad = rr.rr_signal_pad_create(W)
    call = rr.bound_call("rr_allgather", [x[r].data_ptr() for r in range(W)],
                         [y.data_ptr()] + [None] * (W - 1), W, n, rr.RR_BF16, pad, stream.cuda_stream)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def gemm():
        with torch.cuda.stream(gs):
            torch.matmul(a, b, out=c)

    def span(st, fn, k):
        e0, e1 = ev(), ev()
        e0.record(st)
        for _ in range(k):
            fn()
        e1.record(st)
        e1.synchronize()
        return e0.elapsed_time(e1)

    for _ in range(3):
        gemm()
    gemm_ms = span(gs, gemm, 10) / 10
    out = {"bytes_per_call": 2 * W * n * EB, "gemm": f"bf16 {mkn}x{mkn}x{mkn} (cuBLAS via torch.matmul)",
           "gemm_alone_us": round(1000 * gemm_ms, 1), "engines": {}}
    for name, code in (("ldst", 1), ("tma", 2), ("copy_engine", 3)):
        pad.set_option("gather_engine", code)
        for _ in range(5):
            call()
        stream.synchronize()
        ag_ms = span(stream, call, n_ag) / n_ag
        n_gemm = max(1, round(n_ag * ag_ms / gemm_ms))
        # both streams start together behind one event, issue interleaved
        torch.cuda.synchronize()
        go = ev()
        go.record(stream)
        gs.wait_event(go)
        a0, a1, g0, g1 = ev(), ev(), ev(), ev()
        a0.record(stream)
        g0.record(gs)
        ratio = n_ag / n_gemm
        issued = 0
        for i in range(n_gemm):
            gemm()
            while issued < round((i + 1) * ratio):
                call()
                issued += 1
        while issued < n_ag:
            call()
            issued += 1
        a1.record(stream)
        g1.record(gs)
        torch.cuda.synchronize()
        ag_with = a0.elapsed_time(a1) / n_ag
        gemm_with = g0.elapsed_time(g1) / n_gemm
        makespan = max(go.elapsed_time(a1), go.elapsed_time(g1))
        serial = n_ag * ag_ms + n_gemm * gemm_ms
        out["engines"][name] = {
            "ag_alone_us": round(1000 * ag_ms, 1), "ag_with_gemm_us": round(1000 * ag_with, 1),
            "ag_slowdown": round(ag_with / ag_ms, 3), "gemms": n_gemm,
            "gemm_with_ag_us": round(1000 * gemm_with, 1), "gemm_slowdown": round(gemm_with / gemm_ms, 3),
            "makespan_ms": round(makespan, 3), "serial_ms": round(serial, 3),
            "overlap_gain": round(serial / makespan, 3)}
    pad.status(stream)
    pad.close()
    return out


def run_gpu(args, rank, world, local_rank):
    import allgather_rr_allreduce_gb300 as rr
    from allgather_rr_allreduce_gb300 import build as rr_build
    rr_build.build()
    torch.cuda.set_device(local_rank)
    stream = torch.cuda.Stream()
    # The 28 FSDP layers are the first large allocation of the process, as a
    # training job allocates its weights before its scratch buffers; a second
    # set allocated at the end (`fsdp_28_layers_allocated_late`) shows that
    # the order does not matter.
    fsdp_layers = FsdpLayers(rr, stream) if (rank == 0 and not args.no_extras) else None
    ops = tuple(args.only.split(",")) if args.only else OP_NAMES
    step = Step(rr, stream, seed=workloads.LARGE["seed_base"] + 97 * rank, ops=ops,
                n=args.numel or N, pc_div=args.pc_div)
    step.pad.set_option("reduce_engine", ("auto", "ldst", "tma").index(args.reduce_engine))
    step.pad.set_option("twoshot_mode", ("auto", "pull", "push").index(args.twoshot_mode))
    step.pad.set_option("gather_engine", GATHER_ENGINES.index(args.gather_engine))
    bytes_by_op = step.bytes_by_op()
    step_bytes = sum(bytes_by_op.values())
    torch.cuda.synchronize()

    def new_events():
        return [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in ops]

    def op_ms(evs, i):
        return [e[i][0].elapsed_time(e[i][1]) for e in evs]

    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()
    # Warm-up, with an event pair around every op: picks the op with the
    # largest share of the step (the roofline kernel).
    warm = [new_events() for _ in range(args.warmup)]
    for k in range(args.warmup):
        step.run(warm[k])
    stream.synchronize()
    tail = warm[max(1, args.warmup // 2):] or warm
    dom_i = max(range(len(ops)), key=lambda i: statistics.mean(op_ms(tail, i)))

    # Timed region: exactly K steps; events only around the roofline op (an
    # event pair between two launches costs a few microseconds, so none are
    # put around the other ops here).
    events = [new_events() for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        step.run(events[k], only=dom_i)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if rank == 0 else None
    step.pad.status(stream)
    elapsed_ms = t_start.elapsed_time(t_end)
    dom_ms = op_ms(events, dom_i)

    # Per-op breakdown, after the timed region: event pairs around every op.
    n_prof = min(args.steps, 100)
    prof = [new_events() for _ in range(n_prof)]
    for k in range(n_prof):
        step.run(prof[k])
    stream.synchronize()
    per_op_ms = {name: op_ms(prof, i) for i, name in enumerate(ops)}

    max_ms = max_over_ranks(elapsed_ms, world)

    # Extras that need only device memory run before the end-to-end leg (which
    # adds a second set of step buffers and pinned host copies of both).  A
    # second set of 28 layers, allocated after everything else, is timed at
    # the end.
    early = {}
    if rank == 0 and not args.no_extras:
        early["ops_alone"] = ops_alone(step)
        early["fsdp_28_layers"] = fsdp_layers.measure()
        fsdp_layers.close()

    # end to end through the public API: host inputs in, host outputs out
    e2e_steps = max(2, min(args.steps, 6))
    with torch.cuda.stream(stream):
        step.run_e2e()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            step.run_e2e()
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    # the same steps with the copies pipelined across steps over two buffer
    # sets (the headline e2e)
    step_b = Step(rr, stream, seed=workloads.LARGE["seed_base"] + 97 * rank + 1, ops=ops,
                  n=args.numel or N, pc_div=args.pc_div)
    for opt in ("reduce_engine", "twoshot_mode", "gather_engine"):
        step_b.pad.set_option(opt, step.pad.get_option(opt))
    e2e_steps_p = 2 * e2e_steps
    with torch.cuda.stream(stream):
        run_e2e_pipelined([step, step_b], 2, torch.cuda.Event())
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e1 = run_e2e_pipelined([step, step_b], e2e_steps_p, e0)
    torch.cuda.synchronize()
    step_b.pad.status(stream)
    e2e_pipe_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps_p, world)
    # Whether overlapping the two copy directions pays depends on the host
    # (on some boxes concurrent copies in and out are slower than serial
    # ones): both schedules are timed, the faster one is the figure.
    e2e_ms = min(e2e_pipe_ms, e2e_serial_ms)
    bi, bo = step.e2e_bytes()

    if rank != 0:
        return None

    peak, peak_kind = measured_peaks()
    op_stats = {}
    for name in ops:
        ms = statistics.mean(per_op_ms[name])
        gbs = bytes_by_op[name] / ms / 1e6
        qs = statistics.quantiles(per_op_ms[name], n=10) if len(per_op_ms[name]) >= 10 else [ms] * 9
        op_stats[name] = {"bytes": bytes_by_op[name], "us": round(1000 * ms, 2),
                     "us_median": round(1000 * statistics.median(per_op_ms[name]), 2),
                     "us_p10": round(1000 * qs[0], 2), "us_p90": round(1000 * qs[-1], 2),
                     "GBps": round(gbs, 1), "pct_of_8TBps": round(100 * gbs / NOMINAL_HBM_GBS, 2),
                     f"frac_of_{peak_kind}": round(gbs / peak, 4)}
    dominant = ops[dom_i]
    dom_gbs = bytes_by_op[dominant] / statistics.mean(dom_ms) / 1e6
    ms_per_step = max_ms / args.steps
    value = world * step_bytes / ms_per_step / 1e6

    extras = dict(early)
    if not args.no_extras:
        late = FsdpLayers(rr, stream)
        extras["fsdp_28_layers_allocated_late"] = late.measure()
        late.close()
        extras["latency_us"] = latency_sweep(rr, stream)
        extras["small_config"] = small_config_latency(rr, stream)
        extras["allgather_sweep"] = ag_sweep(rr, stream)
        extras["allgather_dtypes"] = ag_sweep_dtypes(rr, stream)
        extras["overlap_gemm"] = overlap_gemm(rr, stream)

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded torch RNG on the device; N(0,1) ranks, N(0,0.02) layer shards)",
        "config": {"workload": workload_name(ops, step.n, args.pc_div),
                   "reduce_engine": args.reduce_engine, "twoshot_mode": args.twoshot_mode,
                   "gather_engine": args.gather_engine, "W": W, "numel_per_rank": step.n, "bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2 (every op >= 288 MiB of its own buffers; L2 129 MB)",
                   "parallelism": f"replicas x{world} (no inter-GPU collective; W ranks emulated per GPU)"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(dom_gbs, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (STREAM-style copy, burst)", "unit": "GB/s",
                     "frac": round(dom_gbs / peak, 4), "traffic": recorded_traffic(dominant),
                     "us_per_launch": round(1000 * statistics.mean(dom_ms), 2),
                     "algorithmic_bytes_per_launch": bytes_by_op[dominant]},
        "ops": op_stats,
        "ops_note": f"per-op breakdown from {n_prof} extra steps with an event pair around every op "
                    "(each pair adds a few us to its op); value uses the timed steps",
        "e2e": {"value": round(world * step_bytes / e2e_ms / 1e6, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "schedule": "pipelined" if e2e_pipe_ms <= e2e_serial_ms else "serial",
                "how": "public API calls on device buffers; every step copies all inputs host->device "
                       "from pinned memory and all outputs device->host.  Two schedules are timed and "
                       "the faster is the figure: serial (copies in, the step, copies out, on one "
                       "stream) and pipelined (steps alternate between two buffer sets so that one "
                       "step's copies in overlap the previous step's copies out, two copy streams)",
                "serial_ms_per_step": round(e2e_serial_ms, 3),
                "serial_value": round(world * step_bytes / e2e_serial_ms / 1e6, 1),
                "pipelined_ms_per_step": round(e2e_pipe_ms, 3),
                "pipelined_value": round(world * step_bytes / e2e_pipe_ms / 1e6, 1),
                "steps": {"serial": e2e_steps, "pipelined": e2e_steps_p}},
        "gpu_launches": len(ops) * args.steps,
        "clocks": clocks,
        "cpu_baseline": None,
    }
    line.update(extras)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    return line


def workload_name(ops, n, pc_div):
    if tuple(ops) == OP_NAMES and n == N and pc_div == 1:
        return ("W8_bf16_2^24 (32 MiB/rank): oneshot+twoshot x copy_mode off/on, rank-major allgather; "
                "one FSDP layer (hidden 3584/kv 512/ffn 18944) param-contiguous allgather")
    return f"subset {','.join(ops)} at W=8, {n} bf16 per rank, layer splits / {pc_div} (not the full step)"


# ---------------------------------------------------------------------- CPU arm

def _cpu_workload(sample_div, seed):
    n = N // sample_div
    splits = [e // sample_div for e in workloads.shard_sizes(workloads.FSDP_LAYER_PARAMS, W)]
    ins = {k: workloads.rank_buffers(W, n, "bf16", "normal", seed_base=seed + 10 * i)
           for i, k in enumerate(("os_off", "os_on", "ts_off", "ts_on", "ag"))}
    ins["pc"] = workloads.rank_buffers(W, sum(splits), "bf16", "normal", seed_base=seed + 99, sigma=0.02)
    return n, splits, ins


def _cpu_step(oracle, n, splits, ins, threads=1):
    # The oracle's definition of each op.  Staging (copy_mode) is a copy of
    # each input into its registered buffer, then the same sum.  threads > 1
    # runs the oracle's multi-threaded entry points (the same loops with the
    # element range split over host threads; same bits).
    if threads == 1:
        ar, ag, pc = oracle.allreduce, oracle.allgather_rank_major, oracle.allgather_param_contiguous
        args = ()
    else:
        ar, ag, pc = oracle.allreduce_mt, oracle.allgather_rank_major_mt, oracle.allgather_param_contiguous_mt
        args = (threads,)
    ar(ins["os_off"], "bf16", *args)
    staged = [np.array(a, copy=True) for a in ins["os_on"]]
    ar(staged, "bf16", *args)
    ar(ins["ts_off"], "bf16", *args)
    staged = [np.array(a, copy=True) for a in ins["ts_on"]]
    ar(staged, "bf16", *args)
    ag(ins["ag"], "bf16", *args)
    pc(ins["pc"], splits, "bf16", *args)


def host_cores():
    """Cores this process may run on, and the CPU model name."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.startswith("Model name:"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return cores, model


def _time_cpu_steps(oracle, n, splits, ins, threads, warmup, steps):
    for _ in range(warmup):
        _cpu_step(oracle, n, splits, ins, threads)
    t0 = time.perf_counter()
    for _ in range(steps):
        _cpu_step(oracle, n, splits, ins, threads)
    return (time.perf_counter() - t0) / steps


def _cpu_bytes(n, splits):
    nb = n * EB
    pc = sum(splits) * EB
    # same accounting as the GPU arm; two-shot outputs counted for all W ranks
    # (the oracle writes one vector; the other W-1 are identical copies).
    return (W * nb + nb) + (2 * W * nb + nb) + 2 * W * nb + 3 * W * nb + 2 * W * nb + 2 * W * pc


def cpu_baseline(sample_div=4, reps=3):
    """The oracle on the host: every core (the multi-threaded entry points,
    one thread per core), and one core beside it, on a sample of the step."""
    import oracle
    oracle.lib()
    cores, model = host_cores()
    n, splits, ins = _cpu_workload(sample_div, seed=7000)
    b = _cpu_bytes(n, splits)
    dt_all = _time_cpu_steps(oracle, n, splits, ins, cores, 1, reps)
    dt_one = _time_cpu_steps(oracle, n, splits, ins, 1, 1, reps)
    return {"value": round(b / dt_all / 1e9, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": model,
            "sample": f"one step at 1/{sample_div} of every op's elements per rank ({n} elements per rank, "
                      f"layer splits / {sample_div}), {reps} timed rep(s) after one warm-up: {dt_all:.3f} s per "
                      f"step on {cores} threads (the oracle's loops with the element range split over "
                      f"threads, same bits), {dt_one:.3f} s on one",
            "single_core": {"value": round(b / dt_one / 1e9, 3), "unit": "GB/s", "cores": 1,
                            "s_per_step": round(dt_one, 4)},
            "s_per_step": round(dt_all, 4)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.lib()
    cores, model = host_cores()
    sample_div = 16
    n, splits, ins = _cpu_workload(sample_div, seed=8000)
    dt = _time_cpu_steps(oracle, n, splits, ins, cores, args.warmup, args.steps)
    dt_one = _time_cpu_steps(oracle, n, splits, ins, 1, 1, 3)
    b = _cpu_bytes(n, splits)
    v = b / dt / 1e9
    sample = (f"each step: the whole hot path at 1/{sample_div} of every op's elements per rank "
              f"({n} bf16 per rank, layer splits / {sample_div}); C oracle on {cores} threads (its loops "
              f"with the element range split over threads, same bits)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * dt, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; N(0,1) ranks, N(0,0.02) layer shards)",
        "config": {"workload": f"W8_bf16_2^24 hot path, sampled at 1/{sample_div}", "W": W,
                   "numel_per_rank": n, "parallelism": f"CPU oracle on {cores} host threads, rank 0 only"},
        "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "cpu_model": model, "sample": sample,
                         "single_core": {"value": round(b / dt_one / 1e9, 3), "unit": "GB/s", "cores": 1}},
        "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("rr", "reference"), default="rr")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-op standalone timing, the latency sweep, the 28-layer run, the "
                         "allgather size sweep and the GEMM-overlap run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="", help="comma-separated subset of ops (profiling runs)")
    ap.add_argument("--numel", type=int, default=0, help="elements per rank for the allreduce/allgather ops")
    ap.add_argument("--pc-div", type=int, default=1, help="divide the FSDP layer's splits by this")
    ap.add_argument("--reduce-engine", choices=("auto", "ldst", "tma"), default="auto",
                    help="allreduce engine (pad option reduce_engine)")
    ap.add_argument("--twoshot-mode", choices=("auto", "pull", "push"), default="auto",
                    help="two-shot allgather phase (pad option twoshot_mode)")
    ap.add_argument("--gather-engine", choices=GATHER_ENGINES, default="auto",
                    help="gather engine (pad option gather_engine)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        line = run_gpu(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
