// C-ABI host layer (include/rr.h): argument checks, signal pads, the choice
// of blocks per rank, and one cooperative launch per call.
//
// No call here allocates, synchronises or copies to the device except
// rr_signal_pad_create / _destroy / _status.  Pointer arrays are copied by
// value into the kernel's parameter block.  Argument checks come before any
// CUDA call, so they also run on a machine without a GPU.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "rr_internal.h"

struct rr_signal_pad {
    int device;
    int W;
    int Bmax;
    uint64_t timeout_ns;
    uint32_t *flags;   // device
    uint64_t *rflags;  // device, round flags
    uint32_t *status;  // device, rr::kStatusWords words
    uint64_t *dev_gen; // device generation counter (device-generation mode)
    uint32_t *done;    // device tally of finished blocks (device-generation mode)
    uint64_t *lflags;  // device, rank-local boundary flags (in-launch iteration mode)
    int device_gen;    // 0: host counter passed per call; 1: device counter (graph-capturable)
    uint32_t gen;      // generation of the last call (0 = none yet): low 32 bits of gen64
    uint64_t gen64;    // 64-bit call counter; round flags grow with it
    int64_t round_bytes;  // 0 = automatic
    int inject;        // -1 or rank*4 + barrier
    int blocks_override;
    int engine;        // gathers: 0 auto (= 1), 1 ldst, 2 tma, 3 copy engines
    int reduce_engine; // one-shot with copy_mode off: 0 auto, 1 ldst, 2 tma
    int twoshot_mode;  // 0 auto, 1 pull (middle barrier), 2 push (owner broadcasts)
    int iters;         // in-launch iterations per call (test mode; 1 = off)
    uint32_t skew_ns;  // per-rank delay step before each iteration (test mode)
    int last_grid;
    int last_B;
    int last_engine;
    uint32_t timeout_info[4];  // barrier, rank, block, generation of the last cleared timeout
};

namespace {

thread_local char g_err[512];

rr_status fail(rr_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

rr_status ok()
{
    g_err[0] = 0;
    return RR_OK;
}

rr_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(RR_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int elem_bytes(rr_dtype d)
{
    switch (d) {
    case RR_BF16:
    case RR_FP16: return 2;
    case RR_FP32:
    case RR_INT32: return 4;
    default: return 0;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
    uintptr_t lo, hi;
};
Span span_of(const void *p, int64_t bytes)
{
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + (uintptr_t)bytes};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo < a.hi && b.lo < b.hi; }

// ---------------------------------------------------------------- device info
std::mutex g_mu;
std::map<int, int> g_sms;                               // device -> SM count
std::map<std::pair<int, const void *>, int> g_occ;      // (device, kernel) -> blocks per SM

rr_status resident_blocks(int dev, const rr::KernelChoice &k, int *out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    auto sit = g_sms.find(dev);
    if (sit == g_sms.end()) {
        int sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiProcessorCount)");
        sit = g_sms.emplace(dev, sms).first;
    }
    auto key = std::make_pair(dev, k.fn);
    auto oit = g_occ.find(key);
    if (oit == g_occ.end()) {
        // The default limit covers 48 KiB of static + dynamic shared memory,
        // so any dynamic amount is declared (a 48 KiB ring beside a few
        // static words would otherwise fit no block at all).
        if (k.smem > 0) {
            cudaError_t e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(maxDynamicSharedMemorySize)");
        }
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, k.threads, k.smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        oit = g_occ.emplace(key, per_sm).first;
    }
    *out = oit->second * sit->second;
    return RR_OK;
}

int sm_count(int dev)
{
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_sms.find(dev);
    return it == g_sms.end() ? 0 : it->second;
}

// Blocks per rank: enough that each block moves about `per_block` bytes, no
// more than the pad allows, and few enough that all W*B blocks are resident
// at once (the ranks' blocks wait on each other, so every one of them must
// be running).  A fixed count set on the pad overrides the first rule.
// Gathers: 32 KiB per block.  Reductions: 96 KiB per block (their
// small-message latency, W=8, graph-replayed, was lowest with about one block
// per 16 KiB per rank for the one-shot with every output kept and one per
// 32 KiB for the two-shot: each block added to a barrier costs more than the
// bytes it takes over).  Large messages reach the residency cap either way.
constexpr int64_t kBytesPerBlock = 32 * 1024;
constexpr int64_t kReduceBytesPerBlock = 96 * 1024;

rr_status plan_blocks(rr_signal_pad *pad, const rr::KernelChoice &k, int W, int64_t total_bytes,
                      int *B, int64_t per_block = kBytesPerBlock)
{
    int resident = 0;
    rr_status st = resident_blocks(pad->device, k, &resident);
    if (st != RR_OK) return st;
    int cap = resident / W;
    if (cap < 1) return fail(RR_ERR_TOO_MANY_BLOCKS, "%d ranks do not fit on the device at once", W);
    if (cap > pad->Bmax) cap = pad->Bmax;
    if (pad->blocks_override > 0) {
        if (pad->blocks_override > cap)
            return fail(RR_ERR_TOO_MANY_BLOCKS,
                        "blocks_per_rank=%d exceeds the %d blocks per rank that can run at once here",
                        pad->blocks_override, cap);
        *B = pad->blocks_override;
        return RR_OK;
    }
    if (k.per_sm > 0) {
        const int pref = k.per_sm * sm_count(pad->device) / W;
        if (pref >= 1 && pref < cap) cap = pref;
    }
    int64_t want = (total_bytes + (int64_t)W * per_block - 1) / ((int64_t)W * per_block);
    if (want < 1) want = 1;
    *B = (int)(want < cap ? want : cap);
    return RR_OK;
}

// Vectors per round of a pipelined chunk: `pref` by default (or the pad's
// option), rounded to whole granules, and large enough that the longest
// chunk needs fewer than 2^kRoundBits rounds.
int64_t round_vectors(int64_t option_bytes, int64_t pref, int64_t longest_chunk)
{
    int64_t p = option_bytes > 0 ? option_bytes / 16 : pref;
    const int64_t min_p = (longest_chunk + (1 << rr::kRoundBits) - 2) / ((1 << rr::kRoundBits) - 1);
    if (p < min_p) p = min_p;
    p = ((p + rr::kGranuleVec - 1) / rr::kGranuleVec) * rr::kGranuleVec;
    return p < rr::kGranuleVec ? rr::kGranuleVec : p;
}

// Signal arguments of the next call.  A call of `iters` in-launch
// iterations takes generations gen64 .. gen64 + iters - 1, none of whose low
// 32-bit words may be 0 (the pad starts zeroed); consecutive generations
// alternate in parity, across calls too.
rr::SignalArgs signal_args(rr_signal_pad *pad, int iters = 1)
{
    rr::SignalArgs s;
    s.flags = pad->flags;
    s.lflags = pad->lflags;
    s.status = pad->status;
    s.timeout_ns = pad->timeout_ns;
    const uint64_t spins = pad->timeout_ns / 64 + 4096;
    s.max_spins = spins > 0xffffffffull ? 0xffffffffu : (uint32_t)spins;
    if (pad->device_gen) {
        // the kernel takes its generation from the device counter
        rr::SignalArgs d;
        std::memset(&d, 0, sizeof d);
        d.flags = pad->flags;
        d.lflags = pad->lflags;
        d.rflags = pad->rflags;
        d.status = pad->status;
        d.timeout_ns = pad->timeout_ns;
        d.max_spins = s.max_spins;
        d.W = pad->W;
        d.Bmax = pad->Bmax;
        d.inject = pad->inject;
        d.dev_gen = pad->dev_gen;
        d.done = pad->done;
        return d;
    }
    pad->gen64 += 1;
    // g is never 0 (the pad starts zeroed); skipping by 2 keeps the parity
    auto bad = [&](uint64_t g) {
        const uint32_t lo = (uint32_t)g;
        return lo == 0u || (uint64_t)lo + (uint64_t)(iters - 1) > 0xffffffffull;
    };
    while (bad(pad->gen64)) pad->gen64 += 2;
    s.g = (uint32_t)pad->gen64;
    s.rflags = pad->rflags;
    s.rbase = pad->gen64 << rr::kRoundBits;
    pad->gen64 += (uint64_t)(iters - 1);
    pad->gen = (uint32_t)pad->gen64;
    s.dev_gen = nullptr;
    s.done = nullptr;
    s.W = pad->W;
    s.Bmax = pad->Bmax;
    s.inject = pad->inject;
    return s;
}

template <class Args>
rr_status launch(rr_signal_pad *pad, const rr::KernelChoice &k, int grid, const Args &args,
                 cudaStream_t stream)
{
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)k.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)k.smem;
    cfg.stream = stream;
    // Cooperative (every block resident at once) and programmatic (the grid
    // may be launched while the previous one in the stream drains; every
    // kernel waits for it in begin_call before touching memory): graph-replayed
    // calls at W=8 take 0.2-0.65 us less from 16 to 256 KiB per rank.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *params[1] = {const_cast<Args *>(&args)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, k.fn, params);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC");
    pad->last_grid = grid;
    return ok();
}

rr_status check_pad(rr_signal_pad *pad, int W)
{
    if (!pad) return fail(RR_ERR_INVALID_ARG, "pad is NULL");
    if (W < 1 || W > RR_MAX_WORLD) return fail(RR_ERR_INVALID_ARG, "world_size %d outside 1..%d", W, RR_MAX_WORLD);
    if (W != pad->W) return fail(RR_ERR_INVALID_ARG, "world_size %d but the pad was made for %d", W, pad->W);
    return RR_OK;
}

rr_status check_device(rr_signal_pad *pad)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != pad->device)
        return fail(RR_ERR_WRONG_DEVICE, "current device %d, pad lives on device %d", dev, pad->device);
    return RR_OK;
}

// In-launch iterations (test mode): iteration k's slices start k * stride
// bytes after the given pointers, stride = the per-iteration size rounded up
// to 16 bytes (every slice stays 16-byte aligned).
int64_t iter_stride(int64_t bytes) { return (bytes + 15) & ~(int64_t)15; }
bool iterating(const rr_signal_pad *pad) { return pad->iters > 1 || pad->skew_ns > 0; }
rr_status check_iterating(const rr_signal_pad *pad)
{
    if (pad->device_gen)
        return fail(RR_ERR_INVALID_ARG, "in-launch iterations need the host generation counter (device_generation 0)");
    return RR_OK;
}

rr_status allreduce_common(bool twoshot, const void *const *inputs, void *const *rank_bufs,
                           void *const *outputs, int W, int64_t numel, rr_dtype dtype, int copy_mode,
                           rr_signal_pad *pad, cudaStream_t stream)
{
    rr_status st = check_pad(pad, W);
    if (st != RR_OK) return st;
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(RR_ERR_UNSUPPORTED_DTYPE, "dtype %d", (int)dtype);
    if (numel < 0 || numel > ((int64_t)1 << 40)) return fail(RR_ERR_INVALID_ARG, "numel %lld", (long long)numel);
    if (!rank_bufs || !outputs) return fail(RR_ERR_INVALID_ARG, "rank_bufs / outputs array is NULL");
    if (copy_mode && !inputs) return fail(RR_ERR_INVALID_ARG, "copy_mode needs the inputs array");
    const int64_t bytes = numel * eb;
    const bool iterate = iterating(pad);
    if (iterate) {
        st = check_iterating(pad);
        if (st != RR_OK) return st;
        if (dtype != RR_BF16) return fail(RR_ERR_INVALID_ARG, "in-launch iterations run bf16 reductions only");
        if (twoshot && pad->twoshot_mode == 1)
            return fail(RR_ERR_INVALID_ARG, "in-launch iterations run the push two-shot only");
        if (pad->reduce_engine != 0)
            return fail(RR_ERR_INVALID_ARG, "in-launch iterations run the automatic reduce engine only");
    }
    // bytes each pointer covers: every iteration's slice (rank buffers too
    // with copy_mode off; with copy_mode on every iteration stages into the
    // same rank buffers)
    const int64_t span_io = iterate ? iter_stride(bytes) * (pad->iters - 1) + bytes : bytes;
    const int64_t span_buf = copy_mode ? bytes : span_io;
    int nout = 0;
    for (int r = 0; r < W; ++r) {
        if (!rank_bufs[r]) return fail(RR_ERR_INVALID_ARG, "rank_bufs[%d] is NULL", r);
        if (!aligned16(rank_bufs[r])) return fail(RR_ERR_ALIGNMENT, "rank_bufs[%d] not 16-byte aligned", r);
        if (copy_mode) {
            if (!inputs[r]) return fail(RR_ERR_INVALID_ARG, "inputs[%d] is NULL", r);
            if (!aligned16(inputs[r])) return fail(RR_ERR_ALIGNMENT, "inputs[%d] not 16-byte aligned", r);
        }
        if (outputs[r]) {
            if (!aligned16(outputs[r])) return fail(RR_ERR_ALIGNMENT, "outputs[%d] not 16-byte aligned", r);
            ++nout;
        } else if (twoshot) {
            return fail(RR_ERR_INVALID_ARG, "two-shot needs every output; outputs[%d] is NULL", r);
        }
    }
    if (nout == 0) return fail(RR_ERR_INVALID_ARG, "no output is materialised");
    // In place: the two-shot with copy_mode off accepts outputs[r] ==
    // rank_bufs[r] (the sum replaces every rank's buffer).
    const bool in_place_ok = twoshot && !copy_mode;
    for (int i = 0; i < W; ++i) {
        const Span bi = span_of(rank_bufs[i], span_buf);
        for (int j = 0; j < W; ++j) {
            if (j > i && overlaps(bi, span_of(rank_bufs[j], span_buf)))
                return fail(RR_ERR_ALIAS, "rank_bufs[%d] and rank_bufs[%d] overlap", i, j);
            if (copy_mode && overlaps(bi, span_of(inputs[j], span_io)))
                return fail(RR_ERR_ALIAS, "rank_bufs[%d] and inputs[%d] overlap", i, j);
            if (in_place_ok && i == j && outputs[j] == rank_bufs[i]) continue;
            if (outputs[j] && overlaps(bi, span_of(outputs[j], span_io)))
                return fail(RR_ERR_ALIAS, "rank_bufs[%d] and outputs[%d] overlap%s", i, j,
                            i == j && !in_place_ok ? " (only the two-shot with copy_mode off runs in place)" : "");
        }
        if (!outputs[i]) continue;
        const Span oi = span_of(outputs[i], span_io);
        for (int j = 0; j < W; ++j) {
            if (j > i && outputs[j] && overlaps(oi, span_of(outputs[j], span_io)))
                return fail(RR_ERR_ALIAS, "outputs[%d] and outputs[%d] overlap", i, j);
            if (copy_mode && overlaps(oi, span_of(inputs[j], span_io)))
                return fail(RR_ERR_ALIAS, "outputs[%d] and inputs[%d] overlap", i, j);
        }
    }
    if (numel == 0) return ok();
    st = check_device(pad);
    if (st != RR_OK) return st;

    const bool push = pad->twoshot_mode != 1;
    // bulk-copy engine: one-shot loads (copy_mode off), or staging by a
    // producer warp (copy_mode on; for the two-shot only with the push
    // allgather).  Automatic: auto_staged with copy_mode, auto_bulk_oneshot
    // without.  In-launch iterations always stage by bulk copies (copy_mode)
    // and reduce with loads/stores (copy_mode off).
    const bool tma = copy_mode ? ((!twoshot || push) &&
                                  (iterate || pad->reduce_engine == 2 ||
                                   (pad->reduce_engine == 0 && rr::auto_staged(twoshot, W, bytes, nout))))
                               : (!twoshot && (pad->reduce_engine == 2 ||
                                               (pad->reduce_engine == 0 && !iterate && rr::auto_bulk_oneshot(W, bytes, nout))));
    const rr::KernelChoice k = iterate ? rr::iter_reduce_kernel_for(twoshot, W, copy_mode != 0)
                               : tma ? (copy_mode ? rr::staged_kernel_for(dtype, W, twoshot)
                                                  : rr::oneshot_tma_kernel_for(dtype, W))
                               : twoshot ? rr::twoshot_kernel_for(dtype, W, copy_mode != 0, push)
                                         : rr::oneshot_kernel_for(dtype, W, copy_mode != 0);
    int64_t moved = twoshot ? bytes * (W + 1) + (int64_t)(W - 1) * bytes * 2
                            : (int64_t)nout * bytes * (W + 1);
    if (copy_mode) moved += 2 * (int64_t)W * bytes;
    int B = 0;
    st = plan_blocks(pad, k, W, moved, &B, kReduceBytesPerBlock);
    if (st != RR_OK) return st;

    rr::ReduceArgs a;
    std::memset(&a, 0, sizeof a);
    for (int r = 0; r < W; ++r) {
        a.in[r] = copy_mode ? inputs[r] : nullptr;
        a.buf[r] = rank_bufs[r];
        a.out[r] = outputs[r];
        if (outputs[r]) a.qlist[a.nout++] = r;
    }
    a.numel = numel;
    a.nvec = bytes / 16;
    a.W = W;
    a.B = B;
    a.copy_mode = copy_mode ? 1 : 0;
    {
        // longest chunk of any block: one-shot chunks split the message, two-shot
        // chunks split an owned segment
        const int64_t ng = (a.nvec + rr::kGranuleVec - 1) / rr::kGranuleVec;
        const int64_t seg = twoshot ? (ng + W - 1) / W : ng;
        if (tma && copy_mode) {
            // staged kernel: pieces of the message (one-shot) or of every
            // owner's segment (two-shot), dealt to the rank's blocks in turn
            const int64_t seglen = seg * rr::kGranuleVec < a.nvec ? seg * rr::kGranuleVec : a.nvec;
            a.round_vec = rr::staged_piece_vectors(pad->round_bytes, seglen, twoshot ? W : 1, B);
        } else {
            const int64_t longest = ((seg + B - 1) / B) * rr::kGranuleVec;
            // Default round sizes keep one round of every block's bytes well
            // inside L2: the two-shot moves W ranges per round.
            a.round_vec = round_vectors(pad->round_bytes, twoshot ? 512 : 4096, longest);
        }
    }
    a.iters = iterate ? pad->iters : 1;
    a.skew_ns = iterate ? pad->skew_ns : 0u;
    a.stride = iter_stride(bytes);
    a.sig = signal_args(pad, a.iters);
    pad->last_B = B;
    pad->last_engine = tma ? 2 : 1;
    return launch(pad, k, W * B, a, stream);
}

// Bytes a gather pointer covers: `bytes` per call, or every iteration's
// slice in the in-launch iteration mode.
int64_t gather_span(const rr_signal_pad *pad, int64_t bytes)
{
    return iterating(pad) ? iter_stride(bytes) * (pad->iters - 1) + bytes : bytes;
}

// Checks shared by every gather: pad, dtype, split table (-> a.off, in
// bytes), rank buffers.  *shard = bytes per rank.
rr_status gather_prepare(const void *const *rank_bufs, int W, const int64_t *splits, int nsplit,
                         rr_dtype dtype, rr_signal_pad *pad, rr::GatherArgs &a, int64_t *shard)
{
    rr_status st = check_pad(pad, W);
    if (st != RR_OK) return st;
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(RR_ERR_UNSUPPORTED_DTYPE, "dtype %d", (int)dtype);
    if (nsplit < 0 || nsplit > RR_MAX_SPLITS)
        return fail(RR_ERR_INVALID_ARG, "num_splits %d outside 0..%d", nsplit, RR_MAX_SPLITS);
    if (nsplit > 0 && !splits) return fail(RR_ERR_INVALID_ARG, "split_sizes is NULL");
    if (!rank_bufs) return fail(RR_ERR_INVALID_ARG, "rank_bufs array is NULL");
    int64_t total = 0;
    a.off[0] = 0;
    for (int s = 0; s < nsplit; ++s) {
        if (splits[s] < 0) return fail(RR_ERR_INVALID_ARG, "split_sizes[%d] = %lld", s, (long long)splits[s]);
        total += splits[s];
        if (total > ((int64_t)1 << 40)) return fail(RR_ERR_INVALID_ARG, "shard too large");
        a.off[s + 1] = total * eb;
    }
    for (int r = 0; r < W; ++r) {
        if (!rank_bufs[r]) return fail(RR_ERR_INVALID_ARG, "rank_bufs[%d] is NULL", r);
        if (!aligned16(rank_bufs[r])) return fail(RR_ERR_ALIGNMENT, "rank_bufs[%d] not 16-byte aligned", r);
        a.src[r] = rank_bufs[r];
    }
    a.W = W;
    a.nsplit = nsplit;
    *shard = total * eb;
    return RR_OK;
}

// Enqueue a gather whose arguments are complete but for B and the signal
// arguments.  Engine 3 (copy engines) issues one cudaMemcpyAsync per
// (materialised output, rank, param) slot instead of a kernel: stream order
// stands in for the barriers, since on one GPU the copies start after
// whatever wrote the shards and end before whatever reads the outputs.
template <class Args>
rr_status run_gather(rr_signal_pad *pad, Args &a, int64_t shard, bool list, cudaStream_t stream)
{
    rr_status st = check_device(pad);
    if (st != RR_OK) return st;
    const int engine = pad->engine != 0 ? pad->engine : rr::auto_gather_engine(a, shard);
    const bool iterate = iterating(pad);
    if (iterate) {
        st = check_iterating(pad);
        if (st != RR_OK) return st;
        if (engine == 3) return fail(RR_ERR_INVALID_ARG, "in-launch iterations run the gather kernels, not the copy engines");
    }
    if (engine == 3) {
        for (int q = 0; q < a.nout; ++q)
            for (int r = 0; r < a.W; ++r)
                for (int s = 0; s < a.nsplit; ++s) {
                    const int64_t o = a.off[s], len = a.off[s + 1] - o;
                    if (len == 0) continue;
                    cudaError_t e = cudaMemcpyAsync(rr::slot_dst(a, q, r, s, o),
                                                    static_cast<const char *>(a.src[r]) + o, (size_t)len,
                                                    cudaMemcpyDeviceToDevice, stream);
                    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
                }
        pad->last_grid = 0;
        pad->last_B = 0;
        pad->last_engine = 3;
        return ok();
    }
    const rr::KernelChoice k = iterate ? rr::iter_gather_kernel_for(engine, list) : rr::gather_kernel_for(engine, list);
    int B = 0;
    st = plan_blocks(pad, k, a.W, shard * a.W + shard * a.W * a.nout, &B);
    if (st != RR_OK) return st;
    a.B = B;
    a.iters = iterate ? pad->iters : 1;
    a.skew_ns = iterate ? pad->skew_ns : 0u;
    a.src_stride = iter_stride(shard);
    a.out_stride = iter_stride(shard * a.W);
    a.sig = signal_args(pad, a.iters);
    pad->last_B = B;
    pad->last_engine = engine;
    return launch(pad, k, a.W * B, a, stream);
}

rr_status gather_common(const void *const *rank_bufs, void *const *outputs, int W,
                        const int64_t *splits, int nsplit, rr_dtype dtype, rr_signal_pad *pad,
                        cudaStream_t stream)
{
    rr::GatherArgs a;
    std::memset(&a, 0, sizeof a);
    int64_t shard = 0;
    rr_status st = gather_prepare(rank_bufs, W, splits, nsplit, dtype, pad, a, &shard);
    if (st != RR_OK) return st;
    if (!outputs) return fail(RR_ERR_INVALID_ARG, "outputs array is NULL");
    const int64_t outb = shard * W;
    for (int r = 0; r < W; ++r) {
        if (outputs[r]) {
            if (!aligned16(outputs[r])) return fail(RR_ERR_ALIGNMENT, "outputs[%d] not 16-byte aligned", r);
            a.out[r] = outputs[r];
            a.qlist[a.nout++] = r;
        }
    }
    if (a.nout == 0) return fail(RR_ERR_INVALID_ARG, "no output is materialised");
    const int64_t ospan = gather_span(pad, outb), sspan = gather_span(pad, shard);
    for (int i = 0; i < W; ++i) {
        if (!outputs[i]) continue;
        const Span oi = span_of(outputs[i], ospan);
        for (int j = 0; j < W; ++j) {
            if (j > i && outputs[j] && overlaps(oi, span_of(outputs[j], ospan)))
                return fail(RR_ERR_ALIAS, "outputs[%d] and outputs[%d] overlap", i, j);
            if (overlaps(oi, span_of(rank_bufs[j], sspan)))
                return fail(RR_ERR_ALIAS, "outputs[%d] and rank_bufs[%d] overlap", i, j);
        }
    }
    if (shard == 0) return ok();
    return run_gather(pad, a, shard, false, stream);
}

rr_status gather_list_impl(const void *const *rank_bufs, void *const *out_lists, int W, int64_t numel,
                           rr_dtype dtype, rr_signal_pad *pad, cudaStream_t stream)
{
    if (numel < 0) return fail(RR_ERR_INVALID_ARG, "numel_per_rank %lld", (long long)numel);
    rr::GatherListArgs a;
    std::memset(&a, 0, sizeof a);
    int64_t shard = 0;
    rr_status st = gather_prepare(rank_bufs, W, &numel, 1, dtype, pad, a, &shard);
    if (st != RR_OK) return st;
    if (!out_lists) return fail(RR_ERR_INVALID_ARG, "output list array is NULL");
    for (int q = 0; q < W; ++q) {
        int set = 0;
        for (int r = 0; r < W; ++r) {
            void *p = out_lists[q * W + r];
            if (!p) continue;
            if (!aligned16(p)) return fail(RR_ERR_ALIGNMENT, "output list %d entry %d not 16-byte aligned", q, r);
            a.lst[q * W + r] = p;
            ++set;
        }
        if (set != 0 && set != W)
            return fail(RR_ERR_INVALID_ARG, "output list %d has %d of %d buffers (all or none)", q, set, W);
        if (set) a.qlist[a.nout++] = q;
    }
    if (a.nout == 0) return fail(RR_ERR_INVALID_ARG, "no output is materialised");
    // Every list buffer against every other one and every rank buffer.
    const int64_t sspan = gather_span(pad, shard);
    for (int i = 0; i < W * W; ++i) {
        if (!a.lst[i]) continue;
        const Span si = span_of(a.lst[i], sspan);
        for (int j = i + 1; j < W * W; ++j)
            if (a.lst[j] && overlaps(si, span_of(a.lst[j], sspan)))
                return fail(RR_ERR_ALIAS, "output list %d entry %d and list %d entry %d overlap", i / W, i % W,
                            j / W, j % W);
        for (int r = 0; r < W; ++r)
            if (overlaps(si, span_of(rank_bufs[r], sspan)))
                return fail(RR_ERR_ALIAS, "output list %d entry %d and rank_bufs[%d] overlap", i / W, i % W, r);
    }
    if (shard == 0) return ok();
    return run_gather(pad, a, shard, true, stream);
}

}  // namespace

extern "C" {

rr_status rr_signal_pad_create(int world_size, int max_blocks_per_rank, uint64_t timeout_ns,
                               rr_signal_pad **out)
{
    if (!out) return fail(RR_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (world_size < 1 || world_size > RR_MAX_WORLD)
        return fail(RR_ERR_INVALID_ARG, "world_size %d outside 1..%d", world_size, RR_MAX_WORLD);
    if (max_blocks_per_rank < 0 || max_blocks_per_rank > 65536)
        return fail(RR_ERR_INVALID_ARG, "max_blocks_per_rank %d", max_blocks_per_rank);
    const int Bmax = max_blocks_per_rank ? max_blocks_per_rank : rr::kDefaultMaxBlocks;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const size_t nflags = (size_t)world_size * rr::kNumBarriers * 2 * (size_t)Bmax * (size_t)world_size;
    const size_t nrflags = (size_t)world_size * rr::kRoundKinds * (size_t)Bmax * (size_t)world_size;
    const size_t flag_bytes = ((nflags * sizeof(uint32_t) + 255) / 256) * 256;
    const size_t rflag_bytes = nrflags * sizeof(uint64_t);
    const size_t status_bytes = rr::kStatusWords * sizeof(uint32_t);  // 32: keeps 8-byte alignment
    // after the generation counter and the block tally: the rank-local
    // boundary flags of the in-launch iteration mode, [W][Bmax] uint64
    const size_t lflag_off = ((flag_bytes + rflag_bytes + status_bytes + sizeof(uint64_t) + sizeof(uint32_t) + 7) / 8) * 8;
    const size_t bytes = lflag_off + (size_t)world_size * Bmax * sizeof(uint64_t);
    void *mem = nullptr;
    e = cudaMalloc(&mem, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(signal pad)");
    e = cudaMemset(mem, 0, bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(mem);
        return cuda_fail(e, "zeroing the signal pad");
    }
    rr_signal_pad *p = new rr_signal_pad;
    std::memset(p, 0, sizeof *p);
    p->device = dev;
    p->W = world_size;
    p->Bmax = Bmax;
    p->timeout_ns = timeout_ns ? timeout_ns : rr::kDefaultTimeoutNs;
    p->flags = static_cast<uint32_t *>(mem);
    p->rflags = reinterpret_cast<uint64_t *>(static_cast<char *>(mem) + flag_bytes);
    p->status = reinterpret_cast<uint32_t *>(static_cast<char *>(mem) + flag_bytes + rflag_bytes);
    p->dev_gen = reinterpret_cast<uint64_t *>(static_cast<char *>(mem) + flag_bytes + rflag_bytes + status_bytes);
    p->done = reinterpret_cast<uint32_t *>(p->dev_gen + 1);
    p->lflags = reinterpret_cast<uint64_t *>(static_cast<char *>(mem) + lflag_off);
    p->inject = -1;
    p->iters = 1;
    *out = p;
    return ok();
}

rr_status rr_signal_pad_destroy(rr_signal_pad *pad)
{
    if (!pad) return ok();
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(pad->device);
    cudaError_t e = cudaDeviceSynchronize();
    cudaError_t f = cudaFree(pad->flags);
    if (prev >= 0) cudaSetDevice(prev);
    delete pad;
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (f != cudaSuccess) return cuda_fail(f, "cudaFree(signal pad)");
    return ok();
}

rr_status rr_signal_pad_status(rr_signal_pad *pad, cudaStream_t stream)
{
    if (!pad) return fail(RR_ERR_INVALID_ARG, "pad is NULL");
    rr_status st = check_device(pad);
    if (st != RR_OK) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t words[rr::kStatusWords];
    e = cudaMemcpy(words, pad->status, sizeof words, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    if (words[rr::kStErr] == 0 && words[rr::kStAbort] == 0) return ok();
    pad->timeout_info[0] = words[rr::kStBarrier];
    pad->timeout_info[1] = words[rr::kStRank];
    pad->timeout_info[2] = words[rr::kStBlock];
    pad->timeout_info[3] = words[rr::kStGen];
    e = cudaMemsetAsync(pad->status, 0, sizeof words, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status");
    const rr_status dev_status = words[rr::kStErr] ? (rr_status)words[rr::kStErr] : RR_ERR_TIMEOUT;
    return fail(dev_status, "barrier %u timed out: waiting rank %u, block %u, generation %u",
                words[rr::kStBarrier], words[rr::kStRank], words[rr::kStBlock], words[rr::kStGen]);
}

rr_status rr_signal_pad_timeout_info(rr_signal_pad *pad, int *barrier, int *rank, int *block,
                                     uint32_t *generation)
{
    if (!pad) return fail(RR_ERR_INVALID_ARG, "pad is NULL");
    if (barrier) *barrier = (int)pad->timeout_info[0];
    if (rank) *rank = (int)pad->timeout_info[1];
    if (block) *block = (int)pad->timeout_info[2];
    if (generation) *generation = pad->timeout_info[3];
    return ok();
}

rr_status rr_signal_pad_set_option(rr_signal_pad *pad, rr_option opt, int64_t value)
{
    if (!pad) return fail(RR_ERR_INVALID_ARG, "pad is NULL");
    switch (opt) {
    case RR_OPT_TIMEOUT_NS:
        if (value <= 0) return fail(RR_ERR_INVALID_ARG, "timeout must be positive");
        pad->timeout_ns = (uint64_t)value;
        return ok();
    case RR_OPT_BLOCKS_PER_RANK:
        if (value < 0 || value > pad->Bmax)
            return fail(RR_ERR_INVALID_ARG, "blocks_per_rank %lld outside 0..%d", (long long)value, pad->Bmax);
        pad->blocks_override = (int)value;
        return ok();
    case RR_OPT_GATHER_ENGINE:
        if (value < 0 || value > 3) return fail(RR_ERR_INVALID_ARG, "gather engine %lld", (long long)value);
        pad->engine = (int)value;
        return ok();
    case RR_OPT_INJECT_SKIP:
        if (value < -1 || value >= (int64_t)pad->W * rr::kNumBarriers)
            return fail(RR_ERR_INVALID_ARG, "inject %lld", (long long)value);
        pad->inject = (int)value;
        return ok();
    case RR_OPT_ROUND_BYTES:
        if (value < 0) return fail(RR_ERR_INVALID_ARG, "round_bytes %lld", (long long)value);
        pad->round_bytes = value;
        return ok();
    case RR_OPT_REDUCE_ENGINE:
        if (value < 0 || value > 2) return fail(RR_ERR_INVALID_ARG, "reduce engine %lld", (long long)value);
        pad->reduce_engine = (int)value;
        return ok();
    case RR_OPT_TWOSHOT_MODE:
        if (value < 0 || value > 2) return fail(RR_ERR_INVALID_ARG, "two-shot mode %lld", (long long)value);
        pad->twoshot_mode = (int)value;
        return ok();
    case RR_OPT_DEBUG_ITERATIONS:
        if (value < 1 || value > 4096) return fail(RR_ERR_INVALID_ARG, "iterations %lld outside 1..4096", (long long)value);
        pad->iters = (int)value;
        return ok();
    case RR_OPT_DEBUG_SKEW_NS:
        if (value < 0 || value > 1000000) return fail(RR_ERR_INVALID_ARG, "skew %lld ns outside 0..1e6", (long long)value);
        pad->skew_ns = (uint32_t)value;
        return ok();
    case RR_OPT_DEVICE_GENERATION: {
        if (value < 0 || value > 1) return fail(RR_ERR_INVALID_ARG, "device generation %lld", (long long)value);
        if ((int)value == pad->device_gen) return ok();
        rr_status st = check_device(pad);
        if (st != RR_OK) return st;
        // The pad must be idle; the counter carries over so generations keep growing.
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        if (value) {
            const uint32_t zero = 0;
            e = cudaMemcpy(pad->dev_gen, &pad->gen64, sizeof(uint64_t), cudaMemcpyHostToDevice);
            if (e == cudaSuccess) e = cudaMemcpy(pad->done, &zero, sizeof zero, cudaMemcpyHostToDevice);
        } else {
            e = cudaMemcpy(&pad->gen64, pad->dev_gen, sizeof(uint64_t), cudaMemcpyDeviceToHost);
            pad->gen = (uint32_t)pad->gen64;
        }
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(generation counter)");
        pad->device_gen = (int)value;
        return ok();
    }
    default: return fail(RR_ERR_INVALID_ARG, "option %d cannot be set", (int)opt);
    }
}

rr_status rr_signal_pad_get_option(rr_signal_pad *pad, rr_option opt, int64_t *value)
{
    if (!pad || !value) return fail(RR_ERR_INVALID_ARG, "pad or value is NULL");
    switch (opt) {
    case RR_OPT_TIMEOUT_NS: *value = (int64_t)pad->timeout_ns; break;
    case RR_OPT_BLOCKS_PER_RANK: *value = pad->blocks_override; break;
    case RR_OPT_GATHER_ENGINE: *value = pad->engine; break;
    case RR_OPT_INJECT_SKIP: *value = pad->inject; break;
    case RR_OPT_ROUND_BYTES: *value = pad->round_bytes; break;
    case RR_OPT_REDUCE_ENGINE: *value = pad->reduce_engine; break;
    case RR_OPT_TWOSHOT_MODE: *value = pad->twoshot_mode; break;
    case RR_OPT_GENERATION:
        if (pad->device_gen) {
            // read the device counter (synchronises the device)
            uint64_t g = 0;
            cudaError_t e = cudaDeviceSynchronize();
            if (e == cudaSuccess) e = cudaMemcpy(&g, pad->dev_gen, sizeof g, cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return cuda_fail(e, "reading the generation counter");
            *value = (uint32_t)g;
        } else {
            *value = pad->gen;
        }
        break;
    case RR_OPT_DEVICE_GENERATION: *value = pad->device_gen; break;
    case RR_OPT_DEBUG_ITERATIONS: *value = pad->iters; break;
    case RR_OPT_DEBUG_SKEW_NS: *value = pad->skew_ns; break;
    case RR_OPT_LAST_GRID: *value = pad->last_grid; break;
    case RR_OPT_LAST_BLOCKS_PER_RANK: *value = pad->last_B; break;
    case RR_OPT_LAST_ENGINE: *value = pad->last_engine; break;
    case RR_OPT_WORLD_SIZE: *value = pad->W; break;
    case RR_OPT_MAX_BLOCKS_PER_RANK: *value = pad->Bmax; break;
    default: return fail(RR_ERR_INVALID_ARG, "unknown option %d", (int)opt);
    }
    return ok();
}

rr_status rr_allreduce_oneshot(const void *const *inputs, void *const *rank_bufs, void *const *outputs,
                               int world_size, int64_t numel, rr_dtype dtype, int copy_mode,
                               rr_signal_pad *pad, cudaStream_t stream)
{
    return allreduce_common(false, inputs, rank_bufs, outputs, world_size, numel, dtype, copy_mode, pad,
                            stream);
}

rr_status rr_allreduce_twoshot(const void *const *inputs, void *const *rank_bufs, void *const *outputs,
                               int world_size, int64_t numel, rr_dtype dtype, int copy_mode,
                               rr_signal_pad *pad, cudaStream_t stream)
{
    return allreduce_common(true, inputs, rank_bufs, outputs, world_size, numel, dtype, copy_mode, pad,
                            stream);
}

rr_status rr_allgather(const void *const *rank_bufs, void *const *outputs, int world_size,
                       int64_t numel_per_rank, rr_dtype dtype, rr_signal_pad *pad, cudaStream_t stream)
{
    if (numel_per_rank < 0) return fail(RR_ERR_INVALID_ARG, "numel_per_rank %lld", (long long)numel_per_rank);
    const int64_t split = numel_per_rank;
    return gather_common(rank_bufs, outputs, world_size, &split, 1, dtype, pad, stream);
}

rr_status rr_allgather_param_contiguous(const void *const *rank_bufs, void *const *outputs,
                                        int world_size, const int64_t *split_sizes, int num_splits,
                                        rr_dtype dtype, rr_signal_pad *pad, cudaStream_t stream)
{
    return gather_common(rank_bufs, outputs, world_size, split_sizes, num_splits, dtype, pad, stream);
}

rr_status rr_allgather_list(const void *const *rank_bufs, void *const *output_lists, int world_size,
                            int64_t numel_per_rank, rr_dtype dtype, rr_signal_pad *pad, cudaStream_t stream)
{
    return gather_list_impl(rank_bufs, output_lists, world_size, numel_per_rank, dtype, pad, stream);
}

const char *rr_status_string(rr_status s)
{
    switch (s) {
    case RR_OK: return "RR_OK";
    case RR_ERR_INVALID_ARG: return "RR_ERR_INVALID_ARG";
    case RR_ERR_UNSUPPORTED_DTYPE: return "RR_ERR_UNSUPPORTED_DTYPE";
    case RR_ERR_ALIGNMENT: return "RR_ERR_ALIGNMENT";
    case RR_ERR_ALIAS: return "RR_ERR_ALIAS";
    case RR_ERR_TOO_MANY_BLOCKS: return "RR_ERR_TOO_MANY_BLOCKS";
    case RR_ERR_CUDA: return "RR_ERR_CUDA";
    case RR_ERR_TIMEOUT: return "RR_ERR_TIMEOUT";
    case RR_ERR_WRONG_DEVICE: return "RR_ERR_WRONG_DEVICE";
    default: return "RR_ERR_UNKNOWN";
    }
}

const char *rr_last_error(void) { return g_err; }

}  // extern "C"

// ---------------------------------------------------------------- no-alloc one-shot
// rr_allreduce_oneshot_noalloc: the one-shot allreduce for callers that may
// not allocate device memory.  Its signal pad lives in the fixed array below
// instead of memory from rr_signal_pad_create; everything else is the one-shot
// kernel above, unchanged.
namespace {

constexpr int kNoAllocMaxWorld = 8;    // largest W the fixed pad can serve
constexpr int kNoAllocMaxBlocks = 32;  // largest blocks per rank it can serve
constexpr size_t kNoAllocFlagWords =
    (size_t)kNoAllocMaxWorld * kNoAllocMaxWorld * rr::kNumBarriers * 2 * kNoAllocMaxBlocks;
constexpr size_t kNoAllocRoundWords =  // 32-bit words holding the 64-bit round flags
    2 * (size_t)kNoAllocMaxWorld * kNoAllocMaxWorld * rr::kRoundKinds * kNoAllocMaxBlocks;

struct NoAllocDevice {
    uint32_t *scratch;  // device address of noalloc_scratch on this device
    uint64_t gen;       // generation of the last call on this device
};
std::mutex g_noalloc_mu;
std::map<int, NoAllocDevice> g_noalloc;

}  // namespace

// Flags ([W][4 barriers][2 parities][32 blocks][W] for the call's W), then the
// 64-bit round flags ([W][2][32 blocks][W]), then the status words: 96 KiB +
// 32 B, zero at module load, on every device that loads this library, held
// until the process exits.
static __device__ __align__(256) uint32_t
    noalloc_scratch[kNoAllocFlagWords + kNoAllocRoundWords + rr::kStatusWords];

namespace {

// The record of device `dev` (caller holds g_noalloc_mu).  First use on a
// device: look up the array's device address with this device current (the
// host-side name is not a device address).  A cudaDeviceReset of the device
// voids the address kept here; this library does not support calls on a
// device after it was reset.
rr_status noalloc_device(int dev, NoAllocDevice **out)
{
    auto it = g_noalloc.find(dev);
    if (it == g_noalloc.end()) {
        void *addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc_scratch)");
        it = g_noalloc.emplace(dev, NoAllocDevice{static_cast<uint32_t *>(addr), 0u}).first;
    }
    *out = &it->second;
    return RR_OK;
}

}  // namespace

extern "C" rr_status rr_allreduce_oneshot_noalloc(const void *const *inputs, void *const *rank_bufs,
                                                  void *const *outputs, int world_size, int64_t numel,
                                                  rr_dtype dtype, int copy_mode, cudaStream_t stream)
{
    const int W = world_size;
    if (W < 1 || W > kNoAllocMaxWorld)
        return fail(RR_ERR_INVALID_ARG,
                    "world_size %d: the allocation-free one-shot serves 1..%d ranks (its fixed signal pad "
                    "holds %d x %d ranks x %d blocks per rank); use rr_allreduce_oneshot with a pad",
                    W, kNoAllocMaxWorld, kNoAllocMaxWorld, kNoAllocMaxWorld, kNoAllocMaxBlocks);
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(RR_ERR_UNSUPPORTED_DTYPE, "dtype %d", (int)dtype);
    if (numel < 0 || numel > ((int64_t)1 << 40)) return fail(RR_ERR_INVALID_ARG, "numel %lld", (long long)numel);
    if (!rank_bufs || !outputs) return fail(RR_ERR_INVALID_ARG, "rank_bufs / outputs array is NULL");
    if (copy_mode && !inputs) return fail(RR_ERR_INVALID_ARG, "copy_mode needs the inputs array");
    const int64_t bytes = numel * eb;
    int nout = 0;
    for (int r = 0; r < W; ++r) {
        if (!rank_bufs[r]) return fail(RR_ERR_INVALID_ARG, "rank_bufs[%d] is NULL", r);
        if (!aligned16(rank_bufs[r])) return fail(RR_ERR_ALIGNMENT, "rank_bufs[%d] not 16-byte aligned", r);
        if (copy_mode && !inputs[r]) return fail(RR_ERR_INVALID_ARG, "inputs[%d] is NULL", r);
        if (copy_mode && !aligned16(inputs[r])) return fail(RR_ERR_ALIGNMENT, "inputs[%d] not 16-byte aligned", r);
        if (outputs[r]) {
            if (!aligned16(outputs[r])) return fail(RR_ERR_ALIGNMENT, "outputs[%d] not 16-byte aligned", r);
            ++nout;
        }
    }
    if (nout == 0) return fail(RR_ERR_INVALID_ARG, "no output is materialised");
    for (int i = 0; i < W; ++i) {
        for (int j = 0; j < W; ++j) {
            const Span bi = span_of(rank_bufs[i], bytes);
            if (j > i && overlaps(bi, span_of(rank_bufs[j], bytes)))
                return fail(RR_ERR_ALIAS, "rank_bufs[%d] and rank_bufs[%d] overlap", i, j);
            if (copy_mode && overlaps(bi, span_of(inputs[j], bytes)))
                return fail(RR_ERR_ALIAS, "rank_bufs[%d] and inputs[%d] overlap", i, j);
            if (outputs[j] && overlaps(bi, span_of(outputs[j], bytes)))
                return fail(RR_ERR_ALIAS, "rank_bufs[%d] and outputs[%d] overlap", i, j);
            if (!outputs[i]) continue;
            const Span oi = span_of(outputs[i], bytes);
            if (j > i && outputs[j] && overlaps(oi, span_of(outputs[j], bytes)))
                return fail(RR_ERR_ALIAS, "outputs[%d] and outputs[%d] overlap", i, j);
            if (copy_mode && overlaps(oi, span_of(inputs[j], bytes)))
                return fail(RR_ERR_ALIAS, "outputs[%d] and inputs[%d] overlap", i, j);
        }
    }
    if (numel == 0) return ok();

    // Each call takes its generation from a host counter and passes it as a
    // kernel argument; a launch captured into a CUDA graph would replay with
    // the same generation, so flags from the previous replay would already
    // satisfy its waits.  Refuse the call while the stream is capturing.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &capture);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (capture != cudaStreamCaptureStatusNone)
        return fail(RR_ERR_INVALID_ARG,
                    "the stream is being captured: the allocation-free one-shot takes a new generation from a "
                    "host counter per call, which a graph replay would repeat; use rr_allreduce_oneshot with a "
                    "pad in device-generation mode inside graphs");

    int dev = -1;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    uint32_t *scratch = nullptr;
    uint64_t gen = 0;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        NoAllocDevice *d = nullptr;
        rr_status st = noalloc_device(dev, &d);
        if (st != RR_OK) return st;
        d->gen += 1;
        if ((uint32_t)d->gen == 0) d->gen += 2;
        scratch = d->scratch;
        gen = d->gen;
    }

    const rr::KernelChoice k = rr::oneshot_kernel_for(dtype, W, copy_mode != 0);
    int resident = 0;
    rr_status st = resident_blocks(dev, k, &resident);
    if (st != RR_OK) return st;
    int cap = resident / W;
    if (cap > kNoAllocMaxBlocks) cap = kNoAllocMaxBlocks;
    if (cap < 1) return fail(RR_ERR_TOO_MANY_BLOCKS, "%d ranks do not fit on the device at once", W);
    int64_t moved = (int64_t)nout * bytes * (W + 1) + (copy_mode ? 2 * (int64_t)W * bytes : 0);
    int64_t want = (moved + (int64_t)W * kReduceBytesPerBlock - 1) / ((int64_t)W * kReduceBytesPerBlock);
    const int B = (int)(want < 1 ? 1 : (want < cap ? want : cap));

    // The array keeps the last call's words: the status words must start at
    // zero (a timeout left by an earlier call would stop this one); the flags
    // need no clearing, because a slot only passes for this call's generation.
    uint32_t *status_words = scratch + kNoAllocFlagWords + kNoAllocRoundWords;
    e = cudaMemsetAsync(status_words, 0, rr::kStatusWords * sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status words)");

    rr::ReduceArgs a;
    std::memset(&a, 0, sizeof a);
    for (int r = 0; r < W; ++r) {
        a.in[r] = copy_mode ? inputs[r] : nullptr;
        a.buf[r] = rank_bufs[r];
        a.out[r] = outputs[r];
        if (outputs[r]) a.qlist[a.nout++] = r;
    }
    a.numel = numel;
    a.nvec = bytes / 16;
    a.W = W;
    a.B = B;
    a.copy_mode = copy_mode ? 1 : 0;
    {
        const int64_t ng = (a.nvec + rr::kGranuleVec - 1) / rr::kGranuleVec;
        a.round_vec = round_vectors(0, 4096, ((ng + B - 1) / B) * rr::kGranuleVec);
    }
    a.sig.flags = scratch;
    a.sig.rflags = reinterpret_cast<uint64_t *>(scratch + kNoAllocFlagWords);
    a.sig.rbase = gen << rr::kRoundBits;
    a.sig.status = status_words;
    a.sig.timeout_ns = rr::kDefaultTimeoutNs;
    a.sig.max_spins = (uint32_t)(rr::kDefaultTimeoutNs / 64 + 4096);
    a.sig.g = (uint32_t)gen;
    a.sig.W = W;
    a.sig.Bmax = kNoAllocMaxBlocks;
    a.sig.inject = -1;

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(W * B), 1, 1);
    cfg.blockDim = dim3((unsigned)k.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)k.smem;
    cfg.stream = stream;
    // Cooperative (every block resident at once) and programmatic (the grid
    // may be launched while the previous one in the stream drains; every
    // kernel waits for it in begin_call before touching memory): graph-replayed
    // calls at W=8 take 0.2-0.65 us less from 16 to 256 KiB per rank.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *params[1] = {&a};
    e = cudaLaunchKernelExC(&cfg, k.fn, params);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC");
    return ok();
}

extern "C" rr_status rr_allreduce_oneshot_noalloc_status(cudaStream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int dev = -1;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    uint32_t *status_words = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        auto it = g_noalloc.find(dev);
        if (it == g_noalloc.end()) return ok();  // no call on this device yet
        status_words = it->second.scratch + kNoAllocFlagWords + kNoAllocRoundWords;
    }
    uint32_t words[rr::kStatusWords];
    e = cudaMemcpy(words, status_words, sizeof words, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status words)");
    if (words[rr::kStErr] == 0 && words[rr::kStAbort] == 0) return ok();
    e = cudaMemsetAsync(status_words, 0, sizeof words, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status words");
    const rr_status dev_status = words[rr::kStErr] ? (rr_status)words[rr::kStErr] : RR_ERR_TIMEOUT;
    return fail(dev_status, "barrier %u timed out: waiting rank %u, block %u, generation %u", words[rr::kStBarrier],
                words[rr::kStRank], words[rr::kStBlock], words[rr::kStGen]);
}
