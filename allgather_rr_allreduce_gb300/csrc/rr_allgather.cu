// Rank-major and param-contiguous allgather over W ranks emulated on one GPU.
//
// Rank-major all_gather_into_tensor is the param-contiguous gather with a
// single split, so one kernel serves both.  Rank r's shard is a run of params:
// bytes [off[s], off[s+1]) of the shard hold its piece of param s, and that
// piece lands at byte off[s]*W + r*(off[s+1]-off[s]) of every materialised
// output ("ccl: hierarchical cross-node AllGather (intra-node SDMA +
// inter-node RDMA) #441": rank r lands at O_s*W + r*E_s; one fused launch over
// every (rank, param) slot).
//
// Each rank pushes its own shard into the outputs, as that PR's direct
// scatter does: block (r, b) reads its tiles of shard r once and writes them
// to every output, so a byte is read from HBM once however many outputs
// exist.  Barriers: ARRIVE (every rank has entered, so its output may be
// written), END on block b (every push of block b of every rank has landed
// before anyone leaves; all block indices together cover every tile).
//
// The list-output gather (torch.distributed.all_gather: output q is W
// separate buffers) runs the same kernels with a one-split shard whose
// destination is buffer (q, r) at the shard's own byte offset: only the
// address of a slot differs (slot_dst in rr_internal.h).
//
// Work per block: tiles b, b + B, b + 2B, ... of the rank's shard
// (kGatherTile bytes), so that a rank's blocks move through its shard
// together (see BlockRanges).
//
// Two engines:
//   ldst: 256 threads move 16-byte vectors (8-byte / 4-byte / 2-byte words
//         when a piece is not 16-byte aligned).  The default.
//   tma:  one thread of the block drives a ring of shared-memory stages with
//         cp.async.bulk (global -> shared, completion on an mbarrier) and
//         cp.async.bulk (shared -> global, bulk groups), one load feeding one
//         store per output; the other warps copy the pieces the bulk engine
//         cannot take (not 16-byte aligned, or the last < 16 bytes).
#include "rr_device.cuh"

namespace rr {

constexpr int kLdstThreads = 256;
constexpr int kTmaThreads = 128;
// Two blocks per SM, each with a ring of three 16 KiB stages (two loads in
// flight ahead of the stores being issued): 64 KiB of loads in flight per SM.
// At W=8 (us, rank-major 32 MiB per rank / one FSDP layer): three blocks of
// four stages 92.9 / 152.9, two of three 87.3 / 144.2, four of two 89.2 /
// 146.2, three of two 95.0 / 159.5, one of six or eight 86.1 / 159.7.
constexpr int kTmaStages = 3;
constexpr int kTmaChunk = 16384;  // bytes per stage
constexpr int kTmaSmem = kTmaStages * kTmaChunk;

// First split s whose byte range ends after x (off[] is non-decreasing).
__device__ __forceinline__ int first_split_after(const GatherArgs &a, int64_t x)
{
    int lo = 0, hi = a.nsplit;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a.off[mid + 1] <= x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Piece of split s inside region [x0, x1) of a shard: shard bytes [p0, p1).
__device__ __forceinline__ bool piece_of(const GatherArgs &a, int s, int64_t x0, int64_t x1,
                                         int64_t &p0, int64_t &p1)
{
    const int64_t o = a.off[s], e = a.off[s + 1];
    p0 = o > x0 ? o : x0;
    p1 = e < x1 ? e : x1;
    return p0 < p1;
}

template <class T>
__device__ __forceinline__ T ld_stream(const T *p) { return __ldcs(p); }
template <class T>
__device__ __forceinline__ void st_stream(T *p, T v) { __stcs(p, v); }

// Copy n words of type T, rank r's shard bytes from p0 on (split s), to
// every materialised output, using threads [tid, tid + nthr) of the block.
template <class T, int U, class Args>
__device__ __forceinline__ void push_words(const Args &a, int r, int s, const char *src, int64_t p0,
                                           int64_t n, int tid, int nthr)
{
    const T *sp = reinterpret_cast<const T *>(src + p0);
    for (int64_t base = tid; base < n; base += (int64_t)nthr * U) {
        T x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + (int64_t)u * nthr;
            if (i < n) x[u] = ld_stream(sp + i);
        }
        for (int q = 0; q < a.nout; ++q) {
            T *d = reinterpret_cast<T *>(slot_dst(a, q, r, s, p0));
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = base + (int64_t)u * nthr;
                if (i < n) st_stream(d + i, x[u]);
            }
        }
    }
}

// Copy shard bytes [p0, p0 + len) (a whole number of elements) with the
// widest word both sides' alignment allows.  Output bases are 16-byte aligned
// (checked on the host), so only the offsets and the length decide.
template <class Args>
__device__ __forceinline__ void push_bytes(const Args &a, int r, int s, const char *src, int64_t p0,
                                           int64_t len, int tid, int nthr)
{
    const uint64_t mis = (uint64_t)(uintptr_t)(src + p0) | (uint64_t)slot_offset(a, r, s, p0) |
                         (uint64_t)len;
    if ((mis & 15) == 0) push_words<uint4, 4>(a, r, s, src, p0, len >> 4, tid, nthr);
    else if ((mis & 7) == 0) push_words<uint2, 4>(a, r, s, src, p0, len >> 3, tid, nthr);
    else if ((mis & 3) == 0) push_words<unsigned int, 4>(a, r, s, src, p0, len >> 2, tid, nthr);
    else push_words<unsigned short, 4>(a, r, s, src, p0, len >> 1, tid, nthr);
}

// The shard bytes block b of a rank moves.  With kGatherTile > 0: tiles
// b, b + B, b + 2B, ... of kGatherTile bytes, so that the B blocks of a rank
// stream through one window of its shard together (one moving window per
// rank, as a plain copy has one, instead of one per block); with 0, the
// block's contiguous region of the shard.  Measured at W=8: 16 KiB tiles
// take one FSDP layer from 155.6 to 149.7 us (loads/stores) and 154.7 to
// 152.1 us (bulk copies); 64 and 256 KiB tiles gain less.
constexpr int64_t kGatherTile = 16384;
struct BlockRanges {
    int64_t shard;
    int B, b;
    int64_t t;
    __device__ BlockRanges(int64_t shard_, int B_, int b_) : shard(shard_), B(B_), b(b_), t(kGatherTile > 0 ? b_ : 0) {}
    __device__ bool next(int64_t &x0, int64_t &x1)
    {
        if (kGatherTile == 0) {
            if (t > 0) return false;
            t = 1;
            byte_region(shard, B, b, x0, x1);
            return x0 < x1;
        }
        const int64_t start = t * kGatherTile;
        if (start >= shard) return false;
        x0 = start;
        x1 = start + kGatherTile < shard ? start + kGatherTile : shard;
        t += B;
        return true;
    }
};

// ------------------------------------------------------------------ ldst engine
template <class Args>
__device__ __forceinline__ void gather_kernel_ldst_body(const Args &a, const SignalArgs &sig)
{
    __shared__ int s_ok;
    const int r = blockIdx.x / a.B;
    const int b = blockIdx.x - r * a.B;
    if (b == 0) emit(sig, RR_BARRIER_ARRIVE, r, 0);
    if (!wait(sig, RR_BARRIER_ARRIVE, r, 0, &s_ok)) return;

    const char *src = static_cast<const char *>(a.src[r]);
    BlockRanges ranges(a.off[a.nsplit], a.B, b);
    int64_t x0, x1;
    while (ranges.next(x0, x1)) {
        for (int s = first_split_after(a, x0); s < a.nsplit && a.off[s] < x1; ++s) {
            int64_t p0, p1;
            if (piece_of(a, s, x0, x1, p0, p1))
                push_bytes(a, r, s, src, p0, p1 - p0, threadIdx.x, kLdstThreads);
        }
    }
    emit(sig, RR_BARRIER_END, r, b);
    wait(sig, RR_BARRIER_END, r, b, &s_ok);
}

template <class Args>
__global__ void __launch_bounds__(kLdstThreads) gather_kernel_ldst(const __grid_constant__ Args a)
{
    const SignalArgs sig = begin_call(a.sig);
    gather_kernel_ldst_body(a, sig);
    end_call(sig);
}

// ------------------------------------------------------------------ tma engine
// The part of piece s the bulk engine takes: shard bytes [p0, pend), both
// ends 16-byte aligned on both sides.
template <class Args>
__device__ __forceinline__ bool bulk_part(const Args &a, int r, int s, int64_t x0, int64_t x1,
                                          int64_t &p0, int64_t &pend)
{
    int64_t p1;
    if (!piece_of(a, s, x0, x1, p0, p1)) return false;
    if ((((uint64_t)(uintptr_t)a.src[r] + (uint64_t)p0) & 15) || (slot_offset(a, r, s, p0) & 15))
        return false;
    pend = p0 + ((p1 - p0) & ~(int64_t)15);
    return pend > p0;
}

template <class Args>
__device__ __forceinline__ void gather_kernel_tma_body(const Args &a, const SignalArgs &sig)
{
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ __align__(8) uint64_t full[kTmaStages];
    __shared__ int s_ok;
    const int r = blockIdx.x / a.B;
    const int b = blockIdx.x - r * a.B;
    const char *src = static_cast<const char *>(a.src[r]);

    // Chunk iterator over the bulk parts of the pieces of the block's byte
    // ranges (thread 0): shard byte position, split and length of the next
    // chunk.  s_next is the next piece to look at in the current range.
    BlockRanges ranges(a.off[a.nsplit], a.B, b);
    int64_t tx0 = 0, tx1 = 0;
    int s_next = a.nsplit, cur_s = 0;
    int64_t pos = 0, pend = 0;
    auto next = [&](int64_t &cs, int &csplit, uint32_t &cl) -> bool {
        while (pos >= pend) {
            if (s_next >= a.nsplit || a.off[s_next] >= tx1) {
                if (!ranges.next(tx0, tx1)) return false;
                s_next = first_split_after(a, tx0);
                continue;
            }
            const int s = s_next++;
            int64_t p0, pe;
            if (bulk_part(a, r, s, tx0, tx1, p0, pe)) {
                pos = p0;
                pend = pe;
                cur_s = s;
            }
        }
        const int64_t left = pend - pos;
        cl = (uint32_t)(left < kTmaChunk ? left : kTmaChunk);
        cs = pos;
        csplit = cur_s;
        pos += cl;
        return true;
    };
    int64_t pos_of[kTmaStages];
    int split_of[kTmaStages];
    uint32_t len_of[kTmaStages];
    auto issue = [&](int k, int64_t cs, int csplit, uint32_t cl) {
        const int st = k % kTmaStages;
        pos_of[st] = cs;
        split_of[st] = csplit;
        len_of[st] = cl;
        mbar_expect_tx(&full[st], cl);
        bulk_load(stage_mem + (size_t)st * kTmaChunk, src + cs, cl, &full[st]);
    };
    auto drain = [&](int from, int to) {
        // Let loads already in flight land before this block's shared
        // memory can be handed to anyone else.
        for (int j = from; j < to; ++j)
            (void)mbar_wait_bounded(sig, &full[j % kTmaStages], (uint32_t)(j / kTmaStages) & 1u);
    };

    // The shard is this rank's own data, ready before any barrier: the first
    // loads go out before the ARRIVE wait, whose latency they overlap.  Only
    // the stores into the outputs (peers' buffers) wait for it.
    int nissued = 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTmaStages; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
        int64_t cs;
        int csplit;
        uint32_t cl;
        while (nissued < kTmaStages && next(cs, csplit, cl)) issue(nissued++, cs, csplit, cl);
    }
    if (b == 0) emit(sig, RR_BARRIER_ARRIVE, r, 0);
    else __syncthreads();
    if (!wait(sig, RR_BARRIER_ARRIVE, r, 0, &s_ok)) {
        if (threadIdx.x == 0) drain(0, nissued);
        return;
    }

    if (threadIdx.x >= 32) {
        // Everything the bulk engine does not take.
        const int tid = threadIdx.x - 32, nthr = kTmaThreads - 32;
        BlockRanges rest(a.off[a.nsplit], a.B, b);
        int64_t x0, x1;
        while (rest.next(x0, x1)) {
            for (int sp = first_split_after(a, x0); sp < a.nsplit && a.off[sp] < x1; ++sp) {
                int64_t p0, p1, q0, qend;
                if (!piece_of(a, sp, x0, x1, p0, p1)) continue;
                if (bulk_part(a, r, sp, x0, x1, q0, qend))
                    push_bytes(a, r, sp, src, qend, p1 - qend, tid, nthr);
                else
                    push_bytes(a, r, sp, src, p0, p1 - p0, tid, nthr);
            }
        }
    } else if (threadIdx.x == 0) {
        bool ok = true;
        for (int k = 0; k < nissued; ++k) {
            const int st = k % kTmaStages;
            if (!mbar_wait_bounded(sig, &full[st], (uint32_t)(k / kTmaStages) & 1u)) {
                ok = false;
                drain(k, nissued);
                break;
            }
            fence_async_shared();
            for (int q = 0; q < a.nout; ++q)
                bulk_store(slot_dst(a, q, r, split_of[st], pos_of[st]), stage_mem + (size_t)st * kTmaChunk,
                           len_of[st]);
            bulk_commit();
            if (k >= 1) {
                int64_t cs;
                int csplit;
                uint32_t cl;
                if (next(cs, csplit, cl)) {
                    bulk_wait_read_1();  // chunk k-1's stores have read their stage
                    issue(nissued++, cs, csplit, cl);
                }
            }
        }
        bulk_wait_all();
        fence_async_global();
        if (!ok) record_timeout(sig, RR_BARRIER_END, r, b);
    }
    emit(sig, RR_BARRIER_END, r, b);
    wait(sig, RR_BARRIER_END, r, b, &s_ok);
}

template <class Args>
__global__ void __launch_bounds__(kTmaThreads) gather_kernel_tma(const __grid_constant__ Args a)
{
    const SignalArgs sig = begin_call(a.sig);
    gather_kernel_tma_body(a, sig);
    end_call(sig);
}

// In-launch iterations (test mode): the bodies above run a.iters times in one
// launch (run_iterations).
template <class Args>
__global__ void __launch_bounds__(kLdstThreads) gather_iter_kernel_ldst(const __grid_constant__ Args a)
{
    run_iterations(a, begin_call(a.sig),
                   [](const Args &ai, const SignalArgs &si) { gather_kernel_ldst_body(ai, si); });
}
template <class Args>
__global__ void __launch_bounds__(kTmaThreads) gather_iter_kernel_tma(const __grid_constant__ Args a)
{
    run_iterations(a, begin_call(a.sig),
                   [](const Args &ai, const SignalArgs &si) { gather_kernel_tma_body(ai, si); });
}

KernelChoice iter_gather_kernel_for(int engine, bool list)
{
    if (engine == 2)
        return KernelChoice{list ? (const void *)gather_iter_kernel_tma<GatherListArgs>
                                 : (const void *)gather_iter_kernel_tma<GatherArgs>,
                            kTmaThreads, kTmaSmem};
    return KernelChoice{list ? (const void *)gather_iter_kernel_ldst<GatherListArgs>
                             : (const void *)gather_iter_kernel_ldst<GatherArgs>,
                        kLdstThreads, 0};
}

KernelChoice gather_kernel_for(int engine, bool list)
{
    if (engine == 2)
        return KernelChoice{list ? (const void *)gather_kernel_tma<GatherListArgs>
                                 : (const void *)gather_kernel_tma<GatherArgs>,
                            kTmaThreads, kTmaSmem, 2};
    // As many blocks as fit (four per SM at 62 registers).  Three per SM
    // gathered one FSDP layer 2-3% faster, but layers now run on the bulk-copy
    // kernel, and where this kernel runs now the two plans are within 0.7 us.
    return KernelChoice{list ? (const void *)gather_kernel_ldst<GatherListArgs>
                             : (const void *)gather_kernel_ldst<GatherArgs>,
                        kLdstThreads, 0};
}

}  // namespace rr
