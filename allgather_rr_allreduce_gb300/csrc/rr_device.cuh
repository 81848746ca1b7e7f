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

// Publish "block b of rank r reached barrier `bar`" to every listener.  All
// threads of the block call it; the CTA barrier orders every thread's earlier
// writes before the release stores of lanes 0..W-1 of warp 0.
__device__ __forceinline__ void emit(const SignalArgs &s, int bar, int r, int b)
{
    __syncthreads();
    if ((int)threadIdx.x < s.W && s.inject != r * kNumBarriers + bar)
        st_flag_release(flag_slot(s, threadIdx.x, bar, b, r), s.g);
}

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

// Warp 0 waits until every emitter's slot of (listener r, bar, block b) holds
// this call's generation.  Lane p polls emitter p.  Bounded: gives up after
// timeout_ns of %globaltimer, after max_spins polls, or as soon as the pad's
// abort word is set (checked on the first poll and every 32nd after), and
// then records the timeout.  Returns the same verdict to every thread.
__device__ __forceinline__ bool wait(const SignalArgs &s, int bar, int r, int b, int *s_ok)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const bool active = lane < s.W;
        const uint32_t *slot = flag_slot(s, r, bar, b, active ? lane : 0);
        const uint64_t t0 = global_ns();
        bool seen = !active;
        bool ok = true;
        uint32_t ns = 0;
        for (uint32_t spins = 0;; ++spins) {
            uint32_t aborted = 0;
            const bool check = (spins & 31u) == 0u;
            if (check && lane == 0) aborted = ld_relaxed(s.status + kStAbort);
            if (!seen) seen = ld_flag_acquire(slot) == s.g;
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
    __syncthreads();
    return *s_ok != 0;
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
// vector): the same rule as combine(), one element at a time.
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
