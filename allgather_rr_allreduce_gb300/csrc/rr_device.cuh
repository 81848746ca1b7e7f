// Device primitives: 128-bit memory ops, the signal-pad barrier, element
// arithmetic of the reduction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rr_internal.h"

namespace rr {

// ---------------------------------------------------------------- memory ops
// Data loads go through L2 only (.cg): the same kernel may have written the
// line on another SM (staged buffers, reduced segments), and L1 is not
// coherent across SMs.
__device__ __forceinline__ uint4 ld_vec(const void *p) { return __ldcg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void st_vec(void *p, uint4 v) { __stcg(reinterpret_cast<uint4 *>(p), v); }
// Streaming accesses (evict first): outputs nothing in the call reads back,
// and staged bytes read for the last time.
__device__ __forceinline__ void st_vec_stream(void *p, uint4 v) { __stcs(reinterpret_cast<uint4 *>(p), v); }
__device__ __forceinline__ uint4 ld_vec_stream(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }

// ---------------------------------------------------------------- flags
// Generation flags follow multi_gpu_barrier / block_barrier in "Question and
// suggestions about custom allreduce" (sglang discussion 2918): a release
// store of the flag into the listener's slot, acquire loads on the own slots.
// All ranks live on this GPU, so the scope is .gpu (the single-device form of
// the system-scope acquire that "ccl: hierarchical cross-node AllGather #441"
// found necessary between agents).
__device__ __forceinline__ void st_flag_release(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_flag_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t *flag_slot(const SignalArgs &s, int listener, int bar, int b,
                                               int emitter)
{
    const size_t idx =
        ((((size_t)listener * kNumBarriers + bar) * 2 + (s.g & 1u)) * (size_t)s.Bmax + b) *
            (size_t)s.W +
        emitter;
    return s.flags + idx;
}

// Publish "block b of rank r reached barrier `bar`" to every listener by
// storing `value` into its slot.  All threads of the block call it; the CTA
// barrier orders every thread's earlier writes before the release stores of
// lanes 0..W-1 of warp 0.
__device__ __forceinline__ void emit(const SignalArgs &s, int bar, int r, int b, uint32_t value)
{
    __syncthreads();
    if ((int)threadIdx.x < s.W && s.inject != r * kNumBarriers + bar)
        st_flag_release(flag_slot(s, threadIdx.x, bar, b, r), value);
}
__device__ __forceinline__ void emit(const SignalArgs &s, int bar, int r, int b) { emit(s, bar, r, b, s.g); }

static __device__ __noinline__ void record_timeout(const SignalArgs &s, int bar, int r, int b)
{
    if (atomicCAS(s.status + kStErr, 0u, (uint32_t)RR_ERR_TIMEOUT) == 0u) {
        s.status[kStBarrier] = (uint32_t)bar;
        s.status[kStRank] = (uint32_t)r;
        s.status[kStBlock] = (uint32_t)b;
        s.status[kStGen] = s.g;
    }
    atomicExch(s.status + kStAbort, 1u);
}

// Warp 0 waits until every emitter's slot passes `seen_ok` (lane p polls
// emitter p's slot).  Bounded: gives up after timeout_ns of %globaltimer,
// after max_spins polls, or as soon as the pad's abort word is set (checked on
// the first poll and every 32nd after), and then records the timeout against
// barrier `bar`.  Returns the same verdict to every thread of the block.
struct CtaSync {
    __device__ void operator()() const { __syncthreads(); }
};

template <class Poll, class Sync = CtaSync>
__device__ __forceinline__ bool wait_on(const SignalArgs &s, int bar, int r, int b, Poll poll, int *s_ok,
                                        Sync sync = Sync())
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const bool active = lane < s.W;
        const uint64_t t0 = global_ns();
        bool seen = !active;
        bool ok = true;
        uint32_t ns = 0;
        for (uint32_t spins = 0;; ++spins) {
            uint32_t aborted = 0;
            const bool check = (spins & 31u) == 0u;
            if (check && lane == 0) aborted = ld_relaxed(s.status + kStAbort);
            if (!seen) seen = poll(lane);
            const bool done = __all_sync(0xffffffffu, seen);
            if (check) {
                const bool bad = aborted != 0u || spins > s.max_spins ||
                                 (global_ns() - t0) > s.timeout_ns;
                if (__any_sync(0xffffffffu, bad)) {
                    ok = false;
                    break;
                }
            }
            if (done) break;
            if (spins >= 8) {
                __nanosleep(ns);
                ns = ns < 224 ? ns + 32 : 256;
            }
        }
        if (!ok && lane == 0) record_timeout(s, bar, r, b);
        if (lane == 0) *s_ok = ok ? 1 : 0;
    }
    sync();
    return *s_ok != 0;
}

// Call-level barrier: every emitter's slot of (listener r, bar, block b, this
// call's parity) holds exactly this call's generation g.
__device__ __forceinline__ bool wait(const SignalArgs &s, int bar, int r, int b, int *s_ok)
{
    const uint32_t *slots = flag_slot(s, r, bar, b, 0);
    return wait_on(s, bar, r, b, [&](int p) { return ld_flag_acquire(slots + p) == s.g; }, s_ok);
}

// ------------------------------------------------------------ round flags
// A barrier passed once per round of a pipelined chunk (staging, the two-shot
// middle) stores increasing 64-bit values, rbase + k + 1 for round k, where
// rbase = (64-bit call generation) << kRoundBits; a wait accepts any value at
// or past its target.  Values only grow, so no parity halves are needed, an
// emitter may run ahead by several rounds, and a stale value from an earlier
// call is always below the target (no wrap-around in 2^48 calls).
__device__ __forceinline__ void st_flag64_release(uint64_t *p, uint64_t v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_flag64_acquire(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t ld_flag64_relaxed(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// With a preceding relaxed load that read a release store: acquire.
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ uint64_t *round_slot(const SignalArgs &s, int listener, int kind, int b, int emitter)
{
    return s.rflags + ((((size_t)listener * kRoundKinds + kind) * (size_t)s.Bmax + b) * (size_t)s.W + emitter);
}
// kind 0 = staging (reported as RR_BARRIER_STAGE), 1 = two-shot middle (RR_BARRIER_MID)
__device__ __forceinline__ int round_barrier(int kind) { return kind == 0 ? RR_BARRIER_STAGE : RR_BARRIER_MID; }

__device__ __forceinline__ void emit_round(const SignalArgs &s, int kind, int r, int b, int k)
{
    __syncthreads();
    if ((int)threadIdx.x < s.W && s.inject != r * kNumBarriers + round_barrier(kind))
        st_flag64_release(round_slot(s, threadIdx.x, kind, b, r), s.rbase + (uint64_t)k + 1u);
}
template <class Sync = CtaSync>
__device__ __forceinline__ bool wait_round(const SignalArgs &s, int kind, int r, int b, int k, int *s_ok,
                                           Sync sync = Sync())
{
    const uint64_t *slots = round_slot(s, r, kind, b, 0);
    const uint64_t target = s.rbase + (uint64_t)k + 1u;
    return wait_on(s, round_barrier(kind), r, b,
                   [&](int p) { return (int64_t)(ld_flag64_acquire(slots + p) - target) >= 0; }, s_ok, sync);
}
// Round flags up to round k from a single thread (the producer lane of a
// warp-specialised block): one release fence, then relaxed stores of the
// newest value to all W listeners.  Waits accept any value at or past their
// target, so publishing round k also publishes every earlier round.  The
// caller has made the rounds' data visible (bulk-store completion and an
// async-proxy fence).
__device__ __forceinline__ void st_flag64_relaxed(uint64_t *p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void emit_round_single(const SignalArgs &s, int kind, int r, int b, int k)
{
    if (s.inject == r * kNumBarriers + round_barrier(kind)) return;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    for (int p = 0; p < s.W; ++p) st_flag64_relaxed(round_slot(s, p, kind, b, r), s.rbase + (uint64_t)k + 1u);
}

// ------------------------------------------------------------ bulk copies
// cp.async.bulk (TMA without a tensor map) between global and shared memory,
// completion of loads counted on an mbarrier, stores tracked in bulk groups.
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// A count handed from one thread of a block to another through shared memory
// (release / acquire at block scope): what the writer observed before the
// store is visible to the reader after it reads the value.
__device__ __forceinline__ void st_shared_release(int *p, int v)
{
    asm volatile("st.release.cta.shared::cta.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_shared_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_load(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
                 "r"(bytes)
                 : "memory");
}
// L2 eviction policies for bulk copies: data read once (evict first) and
// data written to be read back soon by other blocks (evict last).
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_load_hint(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void bulk_store_hint(void *gdst, const void *ssrc, uint32_t bytes, uint64_t policy)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// At most N bulk groups still incomplete (the older ones' writes have landed).
template <int N>
__device__ __forceinline__ void bulk_wait_pending() { asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory"); }
// At most N bulk groups still reading their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read_pending()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bounded wait for an mbarrier phase: false after the pad's timeout or
// iteration limit (the caller records the failure and stops).
__device__ __forceinline__ bool mbar_wait_bounded(const SignalArgs &s, uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    for (uint32_t spins = 0; !mbar_try_wait(bar, parity); ++spins) {
        if ((spins & 255u) == 255u && ((global_ns() - t0) > s.timeout_ns || spins > s.max_spins))
            return false;
    }
    return true;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------ call entry / exit
// Generation of this call.  Host counter: as passed.  Device counter: every
// block reads the value the previous call on the pad left (the kernel
// boundary orders that write before this launch) and uses the next one.
__device__ __forceinline__ uint64_t next_generation(uint64_t g64)
{
    g64 += 1;
    if ((uint32_t)g64 == 0) g64 += 2;  // g is never 0; the parity is kept
    return g64;
}

__device__ __forceinline__ SignalArgs begin_call(const SignalArgs &in)
{
    // Launches are programmatic (the next kernel in the stream may start
    // before this one ends): wait until the previous grid has completed and
    // its writes are visible before touching memory, then let the next one
    // launch.  Without a programmatic launch both are no-ops.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    SignalArgs s = in;
    if (s.dev_gen) {
        const uint64_t g64 = next_generation(*(volatile uint64_t *)s.dev_gen);
        s.g = (uint32_t)g64;
        s.rbase = g64 << kRoundBits;
    }
    return s;
}

// Every block passes here once, whatever path it took.  With the device
// counter, the last block to arrive (all others have counted themselves, so
// all have read the counter: every thread read it at the start and used the
// value in the barriers since) resets the tally and stores this call's
// generation for the next call.  No fence: the tally only has to follow the
// reads, and the kernel boundary orders both stores before the next call.
__device__ __forceinline__ void end_call(const SignalArgs &s)
{
    if (!s.dev_gen) return;
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t total = gridDim.x * gridDim.y * gridDim.z;
        if (atomicAdd(s.done, 1u) == total - 1u) {
            *(volatile uint32_t *)s.done = 0u;
            *(volatile uint64_t *)s.dev_gen = s.rbase >> kRoundBits;
        }
    }
}

// ------------------------------------------- in-launch iterations (test mode)
// Several calls in one launch, so that the barriers between one call's end and
// the next call's start are crossed without a kernel boundary in between (on
// several GPUs there is none): iteration k runs with generation g + k and the
// round base of call gen64 + k (the host reserves that range), on its own
// slices of the inputs and outputs.

// Rank r's blocks sleep ((r + k) mod W) * skew_ns before iteration k, so that
// the ranks reach each barrier out of step.
__device__ __forceinline__ void skew_delay(const SignalArgs &s, int r, int k, uint32_t skew_ns)
{
    if (skew_ns == 0u) return;
    const uint64_t d = (uint64_t)((r + k) % s.W) * skew_ns;
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < d) __nanosleep(1000);
}
__device__ __forceinline__ SignalArgs iteration_signal(const SignalArgs &s, int k)
{
    SignalArgs t = s;
    t.g = s.g + (uint32_t)k;
    t.rbase = s.rbase + ((uint64_t)k << kRoundBits);
    return t;
}
__device__ __forceinline__ void advance_args(ReduceArgs &ai, const ReduceArgs &a, int k)
{
    const int64_t off = (int64_t)k * a.stride;
    for (int r = 0; r < a.W; ++r) {
        if (a.in[r]) ai.in[r] = static_cast<const char *>(a.in[r]) + off;
        if (!a.copy_mode) ai.buf[r] = static_cast<char *>(a.buf[r]) + off;
        if (a.out[r]) ai.out[r] = static_cast<char *>(a.out[r]) + off;
    }
}
__device__ __forceinline__ void advance_args(GatherArgs &ai, const GatherArgs &a, int k)
{
    for (int r = 0; r < a.W; ++r) {
        ai.src[r] = static_cast<const char *>(a.src[r]) + (int64_t)k * a.src_stride;
        if (a.out[r]) ai.out[r] = static_cast<char *>(a.out[r]) + (int64_t)k * a.out_stride;
    }
}
__device__ __forceinline__ void advance_args(GatherListArgs &ai, const GatherListArgs &a, int k)
{
    for (int r = 0; r < a.W; ++r) ai.src[r] = static_cast<const char *>(a.src[r]) + (int64_t)k * a.src_stride;
    for (int i = 0; i < a.W * a.W; ++i)
        if (a.lst[i]) ai.lst[i] = static_cast<char *>(a.lst[i]) + (int64_t)k * a.src_stride;
}

// The boundary between two iterations of one rank: every block of rank r
// has finished iteration k before any starts iteration k + 1, as the kernel
// boundary between two calls on one GPU guarantees.  Without it, block 0 of
// a rank (the only emitter of its ARRIVE flag) could run two calls ahead of
// another block of the same rank and overwrite, in the same parity half,
// the flag that block is still waiting for.  The ranks stay free to drift
// against each other: only the collective's own barriers order them.  Block
// b of rank r stores rbase_k + 1 into its slot (values only grow) and waits,
// bounded, until every block of rank r has stored at least that.
__device__ __forceinline__ bool rank_boundary(const SignalArgs &s, int r, int b, int B, int *s_ok)
{
    __syncthreads();
    uint64_t *slots = s.lflags + (size_t)r * s.Bmax;
    const uint64_t target = s.rbase + 1u;
    if (threadIdx.x == 0) st_flag64_release(slots + b, target);
    if (threadIdx.x < 32) {
        // warp 0 polls the B slots of rank r (lane i: slots i, i + 32, ...)
        const uint64_t t0 = global_ns();
        bool ok = true;
        for (uint32_t spins = 0;; ++spins) {
            bool seen = true;
            for (int j = threadIdx.x; j < B; j += 32)
                if ((int64_t)(ld_flag64_acquire(slots + j) - target) < 0) seen = false;
            if (__all_sync(0xffffffffu, seen)) break;
            if ((spins & 31u) == 0u) {
                const bool bad = (threadIdx.x == 0 && ld_relaxed(s.status + kStAbort) != 0u) ||
                                 spins > s.max_spins || (global_ns() - t0) > s.timeout_ns;
                if (__any_sync(0xffffffffu, bad)) {
                    ok = false;
                    break;
                }
            }
            if (spins >= 8) __nanosleep(128);
        }
        if (!ok && threadIdx.x == 0) record_timeout(s, RR_BARRIER_END, r, b);
        if (threadIdx.x == 0) *s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Run body(args of iteration k, signal of iteration k) for k = 0..iters-1,
// with a rank-local boundary between iterations; stop once any wait of the
// call has given up (the pad's abort word, read by one thread and shared
// with the block).
template <class Args, class Body>
__device__ __forceinline__ void run_iterations(const Args &a, const SignalArgs &sig, Body body)
{
    __shared__ int s_stop;
    Args ai = a;
    const int r = blockIdx.x / a.B;
    const int b = blockIdx.x - r * a.B;
    for (int k = 0; k < a.iters; ++k) {
        if (k > 0) {
            if (!rank_boundary(iteration_signal(sig, k - 1), r, b, a.B, &s_stop)) return;
            __syncthreads();
            if (threadIdx.x == 0) s_stop = ld_relaxed(sig.status + kStAbort) != 0u;
            __syncthreads();
            if (s_stop) return;
            advance_args(ai, a, k);
        }
        skew_delay(sig, r, k, a.skew_ns);
        body(ai, iteration_signal(sig, k));
    }
}

// ---------------------------------------------------------------- arithmetic
// A 16-byte vector holds kEPV elements.  combine() adds the W vectors
// x[0..W-1] element-wise: binary32 accumulator starting at rank 0's value,
// ranks added in order, one round-to-nearest-even conversion at the end
// (int32: wrapping adds in the same order).
__device__ __forceinline__ uint32_t word(const uint4 &v, int k)
{
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ void set_word(uint4 &v, int k, uint32_t w)
{
    if (k == 0) v.x = w;
    else if (k == 1) v.y = w;
    else if (k == 2) v.z = w;
    else v.w = w;
}

enum OpKind { kHalfWidth = 0, kF32 = 1, kI32 = 2 };

struct OpBF16 {
    static constexpr int kKind = kHalfWidth;
    static constexpr int kEPV = 8;
    static constexpr int kBytes = 2;
    // bfloat16 is the top half of a binary32: widening is a shift.
    __device__ static float widen(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
    __device__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ static float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
    __device__ static uint32_t pack(float l, float h)
    {
        __nv_bfloat162 p = __floats2bfloat162_rn(l, h);
        return *reinterpret_cast<uint32_t *>(&p);
    }
    __device__ static uint32_t narrow(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
};

struct OpFP16 {
    static constexpr int kKind = kHalfWidth;
    static constexpr int kEPV = 8;
    static constexpr int kBytes = 2;
    __device__ static float widen(uint32_t bits16) { return __half2float(__ushort_as_half((unsigned short)bits16)); }
    __device__ static float lo(uint32_t w) { return widen(w & 0xffffu); }
    __device__ static float hi(uint32_t w) { return widen(w >> 16); }
    __device__ static uint32_t pack(float l, float h)
    {
        __half2 p = __floats2half2_rn(l, h);
        return *reinterpret_cast<uint32_t *>(&p);
    }
    __device__ static uint32_t narrow(float f) { return __half_as_ushort(__float2half_rn(f)); }
};

struct OpFP32 {
    static constexpr int kKind = kF32;
    static constexpr int kEPV = 4;
    static constexpr int kBytes = 4;
};

struct OpI32 {
    static constexpr int kKind = kI32;
    static constexpr int kEPV = 4;
    static constexpr int kBytes = 4;
};

template <class Op, int WMAX>
__device__ __forceinline__ uint4 combine(const uint4 (&x)[WMAX], int W)
{
    uint4 o;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (Op::kKind == kHalfWidth) {
            float l = Op::lo(word(x[0], k));
            float h = Op::hi(word(x[0], k));
#pragma unroll
            for (int r = 1; r < WMAX; ++r) {
                if (r < W) {
                    l = __fadd_rn(l, Op::lo(word(x[r], k)));
                    h = __fadd_rn(h, Op::hi(word(x[r], k)));
                }
            }
            set_word(o, k, Op::pack(l, h));
        } else if constexpr (Op::kKind == kF32) {
            float acc = __uint_as_float(word(x[0], k));
#pragma unroll
            for (int r = 1; r < WMAX; ++r)
                if (r < W) acc = __fadd_rn(acc, __uint_as_float(word(x[r], k)));
            set_word(o, k, __float_as_uint(acc));
        } else {
            uint32_t acc = word(x[0], k);
#pragma unroll
            for (int r = 1; r < WMAX; ++r)
                if (r < W) acc += word(x[r], k);
            set_word(o, k, acc);
        }
    }
    return o;
}

// Element e of the ragged tail (fewer than kEPV elements after the last whole
// vector): the same rule as combine(), one element at a time, stored into
// outputs dst[0..ndst) after all W loads (so an output may be a rank buffer).
template <class Op>
__device__ __forceinline__ void combine_scalar_to(void *const *bufs, int W, void *const *dst, int ndst, int64_t e)
{
    uint32_t res;
    if constexpr (Op::kBytes == 2) {
        float acc = Op::widen(__ldcg(reinterpret_cast<const unsigned short *>(bufs[0]) + e));
        for (int r = 1; r < W; ++r)
            acc = __fadd_rn(acc, Op::widen(__ldcg(reinterpret_cast<const unsigned short *>(bufs[r]) + e)));
        res = Op::narrow(acc);
        for (int q = 0; q < ndst; ++q) reinterpret_cast<unsigned short *>(dst[q])[e] = (unsigned short)res;
    } else {
        auto ld = [&](int r) -> uint32_t { return __ldcg(reinterpret_cast<const unsigned int *>(bufs[r]) + e); };
        if constexpr (Op::kKind == kF32) {
            float acc = __uint_as_float(ld(0));
            for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, __uint_as_float(ld(r)));
            res = __float_as_uint(acc);
        } else {
            uint32_t acc = ld(0);
            for (int r = 1; r < W; ++r) acc += ld(r);
            res = acc;
        }
        for (int q = 0; q < ndst; ++q) reinterpret_cast<unsigned int *>(dst[q])[e] = res;
    }
}

template <class Op>
__device__ __forceinline__ void combine_scalar(void *const *bufs, int W, void *dst, int64_t e)
{
    if constexpr (Op::kBytes == 2) {
        auto ld = [&](int r) -> uint32_t { return __ldcg(reinterpret_cast<const unsigned short *>(bufs[r]) + e); };
        float acc = Op::widen(ld(0));
        for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, Op::widen(ld(r)));
        reinterpret_cast<unsigned short *>(dst)[e] = (unsigned short)Op::narrow(acc);
    } else {
        auto ld = [&](int r) -> uint32_t { return __ldcg(reinterpret_cast<const unsigned int *>(bufs[r]) + e); };
        if constexpr (Op::kKind == kF32) {
            float acc = __uint_as_float(ld(0));
            for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, __uint_as_float(ld(r)));
            reinterpret_cast<unsigned int *>(dst)[e] = __float_as_uint(acc);
        } else {
            uint32_t acc = ld(0);
            for (int r = 1; r < W; ++r) acc += ld(r);
            reinterpret_cast<unsigned int *>(dst)[e] = acc;
        }
    }
}

}  // namespace rr
