// Internal declarations shared by the C-ABI host layer (rr_api.cu) and the
// kernels (rr_allreduce.cu, rr_allgather.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "rr.h"

#if defined(__CUDACC__)
#define RR_HD __host__ __device__ __forceinline__
#else
#define RR_HD inline
#endif

namespace rr {

constexpr int kNumBarriers = 4;       // rr_barrier values
constexpr int kRoundKinds = 2;        // barriers passed once per round: STAGE, MID
constexpr int kRoundBits = 16;        // rounds per call < 2^16
constexpr int kDefaultMaxBlocks = 1024;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

// Words of the device status block of a pad.
enum StatusWord : int {
    kStErr = 0,      // first rr_status recorded by the device (sticky)
    kStAbort = 1,    // non-zero: every barrier wait gives up at once
    kStBarrier = 2,  // where the first timeout happened ...
    kStRank = 3,
    kStBlock = 4,
    kStGen = 5,
    kStatusWords = 8
};

// Everything a kernel needs to take part in the pad's barriers.
struct SignalArgs {
    uint32_t *flags;     // [W listener][kNumBarriers][2][Bmax][W emitter]
    uint64_t *rflags;    // [W listener][kRoundKinds][Bmax][W emitter], round flags
    uint64_t rbase;      // this call's 64-bit generation << kRoundBits
    uint32_t *status;    // kStatusWords words
    uint64_t timeout_ns; // per wait
    uint32_t max_spins;  // iteration backstop of a wait, in case the timer misbehaves
    uint32_t g;          // generation value of this call (never 0)
    int W;
    int Bmax;
    int inject;          // -1, or rank*4 + barrier whose flags are never emitted
    // Device-resident generation (graph-capturable calls): when non-null, g
    // and rbase are not taken from this struct but from *dev_gen, the 64-bit
    // counter the previous call left; the last block of the call to finish
    // (counted in *done) advances it.
    uint64_t *dev_gen;
    uint32_t *done;
    // In-launch iteration mode: [W][Bmax] flags through which the blocks of
    // one rank meet between iterations (null when the pad has none).
    uint64_t *lflags;
};

// One-shot and two-shot allreduce.
struct ReduceArgs {
    const void *in[RR_MAX_WORLD];  // copy_mode sources
    void *buf[RR_MAX_WORLD];       // registered rank buffers
    void *out[RR_MAX_WORLD];       // outputs (may be null for one-shot)
    int64_t numel;                 // elements per rank
    int64_t nvec;                  // whole 16-byte vectors per rank
    int64_t round_vec;             // vectors per round of a pipelined chunk (multiple of 16)
    int W;
    int B;                         // blocks per rank
    int copy_mode;
    int nout;                      // number of materialised outputs
    int qlist[RR_MAX_WORLD];       // their ranks, ascending
    SignalArgs sig;
    // In-launch iterations (test mode): iteration k works on inputs and
    // outputs (and, with copy_mode off, rank buffers) advanced by k * stride
    // bytes; with copy_mode on every iteration stages into the same rank
    // buffers.  Rank r's blocks sleep ((r + k) mod W) * skew_ns first.
    int iters;
    uint32_t skew_ns;
    int64_t stride;
};

// Rank-major and param-contiguous allgather (rank-major = one split).
struct GatherArgs {
    const void *src[RR_MAX_WORLD];     // rank shards
    void *out[RR_MAX_WORLD];           // outputs (null = not materialised)
    int64_t off[RR_MAX_SPLITS + 1];    // byte offset of param s in a shard; off[nsplit] = shard bytes
    int W;
    int B;
    int nsplit;
    int nout;
    int qlist[RR_MAX_WORLD];
    SignalArgs sig;
    // In-launch iterations (test mode): iteration k reads the shards advanced
    // by k * src_stride bytes and writes the outputs advanced by k * out_stride.
    int iters;
    uint32_t skew_ns;
    int64_t src_stride;
    int64_t out_stride;
};

// List-output allgather (torch.distributed.all_gather): output q is W
// separate buffers, lst[q*W + r] receiving rank r's shard.  Always one split;
// out[] is unused.
struct GatherListArgs : GatherArgs {
    void *lst[RR_MAX_WORLD * RR_MAX_WORLD];
};

// Byte offset, inside its destination buffer, of byte p0 (in split s) of
// rank r's shard.  Param-contiguous: O_s*W + r*E_s + (p0 - O_s), in bytes.
// List output: each rank has a buffer of its own, so the shard's own offset.
RR_HD int64_t slot_offset(const GatherArgs &a, int r, int s, int64_t p0)
{
    const int64_t o = a.off[s], e = a.off[s + 1];
    return o * a.W + (int64_t)r * (e - o) + (p0 - o);
}
RR_HD int64_t slot_offset(const GatherListArgs &, int, int, int64_t p0) { return p0; }

// Address of that byte in the q-th materialised output (qlist order).
RR_HD char *slot_dst(const GatherArgs &a, int q, int r, int s, int64_t p0)
{
    return static_cast<char *>(a.out[a.qlist[q]]) + slot_offset(a, r, s, p0);
}
RR_HD char *slot_dst(const GatherListArgs &a, int q, int r, int, int64_t p0)
{
    return static_cast<char *>(a.lst[a.qlist[q] * a.W + r]) + p0;
}

// ---------------------------------------------------------------- partition
// Work is cut into 256-byte granules (16 vectors of 16 bytes) so that block
// boundaries never split a 128-byte line between two blocks.
constexpr int64_t kGranuleVec = 16;
constexpr int64_t kGranuleBytes = kGranuleVec * 16;

RR_HD int64_t split_point(int64_t n, int64_t parts, int64_t i) { return (n * i) / parts; }

// Vectors [v0, v1) of part i when n vectors are split into `parts` runs of
// whole granules (the last granule may be short).
RR_HD void part_range(int64_t n, int64_t parts, int64_t i, int64_t &v0, int64_t &v1)
{
    const int64_t ng = (n + kGranuleVec - 1) / kGranuleVec;
    int64_t a = split_point(ng, parts, i) * kGranuleVec;
    int64_t b = split_point(ng, parts, i + 1) * kGranuleVec;
    v0 = a < n ? a : n;
    v1 = b < n ? b : n;
}

// Two-shot ownership: rank c owns vectors [c*C, min((c+1)*C, n)) where C is
// ceil(granules / W) granules.
RR_HD void owned_segment(int64_t n, int W, int c, int64_t &s0, int64_t &s1)
{
    const int64_t ng = (n + kGranuleVec - 1) / kGranuleVec;
    const int64_t C = ((ng + W - 1) / W) * kGranuleVec;
    int64_t a = C * c, b = C * (c + 1);
    s0 = a < n ? a : n;
    s1 = b < n ? b : n;
}

// Block b's chunk of rank c's owned segment.
RR_HD void owned_chunk(int64_t n, int W, int B, int c, int b, int64_t &v0, int64_t &v1)
{
    int64_t s0, s1;
    owned_segment(n, W, c, s0, s1);
    int64_t a, e;
    part_range(s1 - s0, B, b, a, e);
    v0 = s0 + a;
    v1 = s0 + e;
}

// Region b (in bytes) of a shard of `bytes` bytes, in whole granules.
RR_HD void byte_region(int64_t bytes, int B, int b, int64_t &x0, int64_t &x1)
{
    const int64_t ng = (bytes + kGranuleBytes - 1) / kGranuleBytes;
    int64_t a = split_point(ng, B, b) * kGranuleBytes;
    int64_t e = split_point(ng, B, b + 1) * kGranuleBytes;
    x0 = a < bytes ? a : bytes;
    x1 = e < bytes ? e : bytes;
}

// ------------------------------------------------- staged copy_mode pieces
// The staged copy_mode kernel cuts each range (one-shot: the message; two-shot:
// every owner's segment) into pieces of P vectors and deals them to a rank's B
// blocks in turn: round k of block b is piece b + kB of every range, and unit
// k * nranges + j is round k of range j.

// Rounds of block b for a range of `len` vectors.
RR_HD int staged_rounds(int64_t len, int64_t P, int B, int b)
{
    const int64_t T = (len + P - 1) / P;
    return T > b ? (int)((T - b + B - 1) / B) : 0;
}

// Piece size P (vectors): 16 KiB by default (or option_bytes), in whole
// granules, doubled until no block has 2^kRoundBits units or more (pieces of
// `nranges` ranges of up to `seglen` vectors over B blocks).  The default
// size is then cut to the smallest that keeps block 0's K rounds, so that
// the B blocks get K rounds each as far as granules allow: 16 KiB pieces of
// a 4 MiB two-shot segment over 19 blocks give 14 rounds to 9 blocks and 13
// to the rest, 15.5 KiB pieces 14 to all (142 against 144 us at W=8 x 32 MiB).
RR_HD int64_t staged_piece_vectors(int64_t option_bytes, int64_t seglen, int nranges, int B)
{
    int64_t p = option_bytes > 0 ? option_bytes / 16 : 1024;
    p = ((p + kGranuleVec - 1) / kGranuleVec) * kGranuleVec;
    if (p < kGranuleVec) p = kGranuleVec;
    for (;;) {
        const int K = staged_rounds(seglen, p, B, 0);
        if ((int64_t)K * nranges < ((int64_t)1 << kRoundBits)) {
            if (option_bytes <= 0 && K > 0) {
                int64_t q = (seglen + (int64_t)B * K - 1) / ((int64_t)B * K);
                q = ((q + kGranuleVec - 1) / kGranuleVec) * kGranuleVec;
                if (q < p) p = q;
            }
            return p;
        }
        p *= 2;
    }
}

// Vectors [ps, pe) of round k of block b in range [s0, s1) (pe <= ps: none).
RR_HD void staged_piece(int64_t s0, int64_t s1, int64_t P, int B, int b, int k, int64_t &ps, int64_t &pe)
{
    ps = s0 + ((int64_t)b + (int64_t)k * B) * P;
    pe = ps + P < s1 ? ps + P : s1;
}

// The reduction items of block (r, b), in unit order.  One-shot: round k's
// piece of the message holds nout * L (output, vector) pairs, split evenly
// over the W blocks of index b (reduce_share's split); this block takes its
// share.  Two-shot: the vectors of round k's piece of rank r's own segment,
// each reduced once and stored into every output.  Every round but the last
// has c_full items, the last c_last.
struct StagedItems {
    int64_t own0, own1, P, c_full, c_last, L_last, n_first, total;
    int K, B, b, r, W, nout, nranges;
    bool twoshot;
    RR_HD void init(bool twoshot_, int64_t own0_, int64_t own1_, int64_t P_, int B_, int b_, int r_, int W_,
                    int nout_)
    {
        twoshot = twoshot_;
        own0 = own0_;
        own1 = own1_;
        P = P_;
        B = B_;
        b = b_;
        r = r_;
        W = W_;
        nout = nout_;
        nranges = twoshot ? W : 1;
        K = staged_rounds(own1 - own0, P, B, b);
        c_full = c_last = L_last = 0;
        if (K > 0) {
            int64_t ps, pe;
            staged_piece(own0, own1, P, B, b, K - 1, ps, pe);
            L_last = pe - ps;
            c_full = twoshot ? P : split_point((int64_t)nout * P, W, r + 1) - split_point((int64_t)nout * P, W, r);
            c_last = twoshot ? L_last
                             : split_point((int64_t)nout * L_last, W, r + 1) - split_point((int64_t)nout * L_last, W, r);
        }
        n_first = (int64_t)(K > 0 ? K - 1 : 0) * c_full;
        total = K > 0 ? n_first + c_last : 0;
    }
    // Item i < total: the unit it needs staged by every rank, the kept output
    // it is stored into (qlist index; -1 = every output) and its vector.
    RR_HD void item(int64_t i, int &unit, int &m, int64_t &v) const
    {
        int k;
        int64_t j;
        if (i < n_first) {
            k = (int)(i / c_full);
            j = i - (int64_t)k * c_full;
        } else {
            k = K - 1;
            j = i - n_first;
        }
        const int64_t ps = own0 + ((int64_t)b + (int64_t)k * B) * P;
        if (twoshot) {
            unit = k * nranges + r;
            m = -1;
            v = ps + j;
        } else {
            const int64_t L = k == K - 1 ? L_last : P;
            const int64_t pos = split_point((int64_t)nout * L, W, r) + j;
            m = (int)(pos / L);
            unit = k;
            v = ps + pos - (int64_t)m * L;
        }
    }
};

// ---------------------------------------------------------------- launchers
// Implemented in rr_allreduce.cu / rr_allgather.cu.  Each returns the kernel
// to launch for the given element type and world size, with its block size
// and dynamic shared memory.
struct KernelChoice {
    const void *fn;
    int threads;
    int smem;
    int per_sm = 0;  // preferred resident blocks per SM for large messages (0 = as many as fit)
};
KernelChoice oneshot_kernel_for(rr_dtype dtype, int W, bool copy_mode);
KernelChoice twoshot_kernel_for(rr_dtype dtype, int W, bool copy_mode, bool push);
KernelChoice oneshot_tma_kernel_for(rr_dtype dtype, int W);  // copy_mode off, bulk-copy loads
// copy_mode on, staging by a bulk-copy producer warp (two-shot: push allgather)
KernelChoice staged_kernel_for(rr_dtype dtype, int W, bool twoshot);
KernelChoice gather_kernel_for(int engine, bool list);  // 1 = loads/stores, 2 = TMA bulk
// In-launch iteration kernels (test mode): bf16 reductions on the default
// engines (one-shot: loads/stores, or bulk-copy staging for copy_mode; two-shot:
// push, or bulk-copy staging for copy_mode) and both gather kernel engines.
KernelChoice iter_reduce_kernel_for(bool twoshot, int W, bool copy_mode);
KernelChoice iter_gather_kernel_for(int engine, bool list);

// ------------------------------------------------------- automatic engines
// Automatic engine of copy_mode: the bulk-copy staging kernel or the
// load/store kernels, by W and bytes per rank.  Measured, bf16, us per call
// (staged / loads-stores): one-shot, rank 0's output, W=2 1..64 MiB per rank
// always slower staged (64 MiB 92.5 / 71.2); W=4 8 MiB 22.8 / 18.6, 16 MiB
// 35.0 / 35.4, 64 MiB 113.1 / 127.1; W=8 2 MiB 14.9 / 13.5, 8 MiB 31.1 /
// 35.9, 32 MiB 103 / 135; W=16 2 MiB 20.6 / 19.8, 4 MiB 31.0 / 38.9.
// The staged one-shot loses once many outputs are kept, each summed from all
// W buffers by the consumer warps: 2 outputs, W=4 32 MiB 86.8 / 78.2, W=8 32
// MiB 123.5 / 162.3, W=16 8 MiB 73.0 / 85.4; all outputs, W=4 32 MiB 139.4 /
// 107.9, W=8 32 MiB 355.7 / 363.5, W=16 8 MiB 337.9 / 295.8, 32 MiB 1588.8 /
// 1214.7; so it runs with one kept output or at most W/4.
// Two-shot, all outputs: W=2 always faster staged (1 MiB 11.6 / 12.5, 64 MiB
// 83.4 / 141.6); W=4 4 MiB 18.4 / 16.9, 8 MiB 25.1 / 29.1; W=8 2 MiB 18.6 /
// 15.7, 8 MiB 42.3 / 46.9; W=16 2 MiB 28.7 / 24.6, 8 MiB 80.6 / 83.7.
inline bool auto_staged(bool twoshot, int W, int64_t bytes_per_rank, int nout)
{
    if (twoshot) return W <= 2 || bytes_per_rank >= ((int64_t)8 << 20);
    return W >= 4 && (int64_t)W * bytes_per_rank >= ((int64_t)64 << 20) && (nout <= 1 || 4 * nout <= W);
}

// Automatic engine of the one-shot with copy_mode off: bulk-copy loads into a
// shared-memory ring when W > 8 and each output reads at least 128 MiB (512
// MiB with more than half the outputs kept), loads/stores otherwise.  Measured, bf16, rank 0's output, us per call
// (loads-stores / bulk): W <= 8 always faster with loads/stores (W=8 32 MiB
// per rank 50.4 / 53.9, 64 MiB 92.3 / 98.5); W=10 8 MiB 16.5 / 22.7, 32 MiB
// 69.9 / 67.6; W=12 8 MiB 23.0 / 26.3, 32 MiB 77.0 / 74.8; W=14 8 MiB 30.8 /
// 28.7; W=16 4 MiB 12.4 / 18.5, 8 MiB 32.9 / 30.1, 64 MiB 183.4 / 168.6.
// Two kept outputs: the same (W=12 8 MiB 37.0 / 41.1, 32 MiB 143.5 / 139.3;
// W=16 8 MiB 49.4 / 46.9).  All outputs: the bulk kernel wins later (W=12 32
// MiB 799.0 / 798.6, W=16 8 MiB 265.1 / 310.9, 32 MiB 1361.7 / 1219.5), so
// with more than half the outputs kept each output must read 512 MiB.
inline bool auto_bulk_oneshot(int W, int64_t bytes_per_rank, int nout)
{
    const int64_t need = (int64_t)(2 * nout > W ? 512 : 128) << 20;
    return W > 8 && (int64_t)W * bytes_per_rank >= need;
}

// Automatic gather engine.  Bulk copies when a call moves at least 256 MiB
// (shards read plus outputs written; 8 MiB with two or more kept outputs)
// and every split boundary sits on a
// multiple of 16 bytes (the bases are checked aligned, so the bulk engine
// then takes every byte); loads/stores otherwise.  Measured, rank-major,
// rank 0's output, us per call (loads/stores, bulk copies): at W=8, 8 MiB per
// rank 28.8 / 29.9, 16 MiB 49.5 / 48.5, 32 MiB 90.1 / 86.5, 512 MiB 1318 /
// 1251; 28 FSDP layers 153-154 / 146 per layer.  Around 128 MiB moved the
// bulk engine loses at every W (W=2 32 MiB per rank 24.7 / 29.6, W=4 16 MiB
// 25.2 / 29.4, W=16 4 MiB 22.7 / 29.0); from 256 MiB up it ties or wins
// (W=4 32 MiB 51.1 / 49.0, W=16 8 MiB 49.4 / 49.2, 16 MiB 90.0 / 86.8).
// With two or more kept outputs the bulk engine also wins below that, from
// 8 MiB moved (W=8, 8 outputs: 256 KiB per rank 16.2 / 11.9, 1 MiB 18.6 /
// 17.1, 32 MiB 409.1 / 399.7; W=4, 4 outputs: 1 MiB 14.2 / 10.6; W=8, 2
// outputs: 1 MiB 12.2 / 11.1, 16 MiB 72.0 / 73.6; below 8 MiB moved the two
// tie or loads/stores lead).
constexpr int64_t kBulkGatherMinBytes = (int64_t)256 << 20;
constexpr int64_t kBulkGatherMinBytesMulti = (int64_t)8 << 20;
inline int auto_gather_engine(const GatherArgs &a, int64_t shard)
{
    const int64_t moved = shard * a.W * (1 + a.nout);
    if (moved < (a.nout >= 2 ? kBulkGatherMinBytesMulti : kBulkGatherMinBytes)) return 1;
    for (int s = 0; s <= a.nsplit; ++s)
        if (a.off[s] & 15) return 1;
    return 2;
}


}  // namespace rr
