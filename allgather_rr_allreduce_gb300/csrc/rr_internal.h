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

}  // namespace rr
