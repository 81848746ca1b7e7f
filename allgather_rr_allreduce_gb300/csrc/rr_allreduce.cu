// One-shot and two-shot allreduce over W ranks emulated on one GPU.
//
// One launch runs every rank's per-GPU kernel: block index = rank * B + b,
// where B is the number of blocks each rank would launch on its own GPU.
// Rank r's blocks read the other ranks' buffers exactly where a real rank
// would read its peers' registered (IPC / symmetric) buffers, and they order
// themselves through the pad's generation flags.
//
// Sources: "Question and suggestions about custom allreduce" (sglang
// discussion 2918) -- the trt_reduce_internal.cu block comment quoted in
// yizhang2077's reply (chunk per block; copy, block barrier, pull and sum) and
// leizhao1234's opening post (two-shot: arrival barrier, reduce-scatter, block
// barrier, allgather); "triton_multimem_all_reduce.py" (symm-mem-recipes) --
// owned slice per rank, grid-stride loop over 128-bit units, a barrier at
// both ends.
#include "rr_device.cuh"

namespace rr {

constexpr int kReduceThreads = 256;

// Vectors kept in flight per thread: 16 loads of 16 bytes whatever W is.
template <int WMAX>
struct Unroll {
    static constexpr int U = WMAX >= 16 ? 1 : 16 / WMAX;
};

// dst[v] = combine over r of buf[r][v], for v in [v0, v1).  Thread t takes
// vectors v0 + t, v0 + t + 256, ...: each warp load is 512 contiguous bytes.
template <class Op, int WMAX>
__device__ __forceinline__ void reduce_vectors(const ReduceArgs &a, void *dst_base, int64_t v0,
                                               int64_t v1)
{
    constexpr int U = Unroll<WMAX>::U;
    uint4 *dst = static_cast<uint4 *>(dst_base);
    const int W = a.W;
    for (int64_t base = v0 + threadIdx.x; base < v1; base += (int64_t)kReduceThreads * U) {
        uint4 x[U][WMAX];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = base + (int64_t)u * kReduceThreads;
            if (v < v1) {
#pragma unroll
                for (int r = 0; r < WMAX; ++r)
                    if (r < W) x[u][r] = ld_vec(static_cast<const uint4 *>(a.buf[r]) + v);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = base + (int64_t)u * kReduceThreads;
            if (v < v1) st_vec(dst + v, combine<Op, WMAX>(x[u], W));
        }
    }
}

// dst[0..n) = src[0..n), 16-byte vectors, 8 in flight per thread.
__device__ __forceinline__ void copy_vectors(const void *src_base, void *dst_base, int64_t n)
{
    constexpr int U = 8;
    const uint4 *src = static_cast<const uint4 *>(src_base);
    uint4 *dst = static_cast<uint4 *>(dst_base);
    for (int64_t base = threadIdx.x; base < n; base += (int64_t)kReduceThreads * U) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = base + (int64_t)u * kReduceThreads;
            if (v < n) x[u] = ld_vec(src + v);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = base + (int64_t)u * kReduceThreads;
            if (v < n) st_vec(dst + v, x[u]);
        }
    }
}

// Elements [e0, e0 + n) of the ragged tail, copied one element at a time.
template <int kBytes>
__device__ __forceinline__ void copy_tail(const void *src, void *dst, int64_t e0, int n)
{
    for (int i = threadIdx.x; i < n; i += kReduceThreads) {
        if constexpr (kBytes == 2)
            static_cast<unsigned short *>(dst)[e0 + i] = __ldcg(static_cast<const unsigned short *>(src) + e0 + i);
        else
            static_cast<unsigned int *>(dst)[e0 + i] = __ldcg(static_cast<const unsigned int *>(src) + e0 + i);
    }
}

// ------------------------------------------------------------------ one-shot
// Block b of every rank works on chunk b (vectors part_range(nvec, B, b); the
// ragged tail belongs to the last chunk).
//  copy_mode: stage inputs[r] chunk b into rank_bufs[r], STAGE barrier on
//             block b (block b of every rank has staged chunk b).
//  otherwise: ARRIVE barrier (block 0 of every rank has started).
//  Reduce chunk b for the materialised outputs.  With every output
//  materialised, block (r, b) reduces chunk b of output r, as rank r's own
//  kernel would.  With fewer, the W blocks of chunk b share that chunk's
//  outputs evenly, so the bandwidth of ranks whose output is not kept is not
//  left idle; every one of them has passed the same barrier on chunk b.
//  END barrier on block b: no rank leaves while a peer still reads its chunk.
template <class Op, int WMAX>
__global__ void __launch_bounds__(kReduceThreads)
    oneshot_kernel(const __grid_constant__ ReduceArgs a)
{
    __shared__ int s_ok;
    const int r = blockIdx.x / a.B;
    const int b = blockIdx.x - r * a.B;
    const bool last = b == a.B - 1;
    int64_t v0, v1;
    part_range(a.nvec, a.B, b, v0, v1);
    const int64_t t0 = a.nvec * Op::kEPV;
    const int ntail = (int)(a.numel - t0);

    if (a.copy_mode) {
        copy_vectors(static_cast<const uint4 *>(a.in[r]) + v0, static_cast<uint4 *>(a.buf[r]) + v0, v1 - v0);
        if (last && ntail > 0) copy_tail<Op::kBytes>(a.in[r], a.buf[r], t0, ntail);
        emit(a.sig, RR_BARRIER_STAGE, r, b);
        if (!wait(a.sig, RR_BARRIER_STAGE, r, b, &s_ok)) return;
    } else {
        if (b == 0) emit(a.sig, RR_BARRIER_ARRIVE, r, 0);
        if (!wait(a.sig, RR_BARRIER_ARRIVE, r, 0, &s_ok)) return;
    }

    const int64_t L = v1 - v0;
    if (L > 0) {
        const int64_t total = (int64_t)a.nout * L;
        int64_t pos = split_point(total, a.W, r);
        const int64_t hi = split_point(total, a.W, r + 1);
        while (pos < hi) {
            const int m = (int)(pos / L);
            const int64_t end = min(hi, (int64_t)(m + 1) * L);
            const int64_t off = pos - (int64_t)m * L;
            reduce_vectors<Op, WMAX>(a, a.out[a.qlist[m]], v0 + off, v0 + off + (end - pos));
            pos = end;
        }
    }
    if (last && ntail > 0) {
        for (int m = r; m < a.nout; m += a.W)
            for (int e = threadIdx.x; e < ntail; e += kReduceThreads)
                combine_scalar<Op>(a.buf, a.W, a.out[a.qlist[m]], t0 + e);
    }

    emit(a.sig, RR_BARRIER_END, r, b);
    wait(a.sig, RR_BARRIER_END, r, b, &s_ok);
}

// ------------------------------------------------------------------ two-shot
// Rank c owns segment owned_segment(nvec, W, c); block b handles chunk b of
// every segment (owned_chunk).  The ragged tail is owned by rank W-1.
//  copy_mode: block b of rank r stages, from inputs[r], chunk b of every
//             owner's segment (everything block b of any rank will read),
//             then the STAGE barrier on block b; otherwise ARRIVE.
//  Reduce-scatter: block (r, b) reduces chunk b of rank r's own segment into
//             outputs[r].  MID barrier on block b.
//  Allgather: block (r, b) copies chunk b of every other owner c's reduced
//             segment from outputs[c] into outputs[r], starting at c = r + 1
//             so that the ranks spread over different sources.  END barrier.
template <class Op, int WMAX>
__global__ void __launch_bounds__(kReduceThreads)
    twoshot_kernel(const __grid_constant__ ReduceArgs a)
{
    __shared__ int s_ok;
    const int W = a.W;
    const int r = blockIdx.x / a.B;
    const int b = blockIdx.x - r * a.B;
    const bool last = b == a.B - 1;
    const int64_t t0 = a.nvec * Op::kEPV;
    const int ntail = (int)(a.numel - t0);
    int64_t c0, c1;

    if (a.copy_mode) {
        for (int c = 0; c < W; ++c) {
            owned_chunk(a.nvec, W, a.B, c, b, c0, c1);
            copy_vectors(static_cast<const uint4 *>(a.in[r]) + c0, static_cast<uint4 *>(a.buf[r]) + c0, c1 - c0);
        }
        if (last && ntail > 0) copy_tail<Op::kBytes>(a.in[r], a.buf[r], t0, ntail);
        emit(a.sig, RR_BARRIER_STAGE, r, b);
        if (!wait(a.sig, RR_BARRIER_STAGE, r, b, &s_ok)) return;
    } else {
        if (b == 0) emit(a.sig, RR_BARRIER_ARRIVE, r, 0);
        if (!wait(a.sig, RR_BARRIER_ARRIVE, r, 0, &s_ok)) return;
    }

    owned_chunk(a.nvec, W, a.B, r, b, c0, c1);
    reduce_vectors<Op, WMAX>(a, a.out[r], c0, c1);
    if (last && ntail > 0 && r == W - 1)
        for (int e = threadIdx.x; e < ntail; e += kReduceThreads)
            combine_scalar<Op>(a.buf, W, a.out[r], t0 + e);

    emit(a.sig, RR_BARRIER_MID, r, b);
    if (!wait(a.sig, RR_BARRIER_MID, r, b, &s_ok)) return;

    for (int k = 1; k < W; ++k) {
        const int c = (r + k) % W;
        owned_chunk(a.nvec, W, a.B, c, b, c0, c1);
        copy_vectors(static_cast<const uint4 *>(a.out[c]) + c0, static_cast<uint4 *>(a.out[r]) + c0, c1 - c0);
    }
    if (last && ntail > 0 && r != W - 1) copy_tail<Op::kBytes>(a.out[W - 1], a.out[r], t0, ntail);

    emit(a.sig, RR_BARRIER_END, r, b);
    wait(a.sig, RR_BARRIER_END, r, b, &s_ok);
}

// ------------------------------------------------------------------ dispatch
template <class Op, bool kTwoShot>
static KernelChoice pick(int W)
{
    const void *fn;
    if (W <= 2) fn = kTwoShot ? (const void *)twoshot_kernel<Op, 2> : (const void *)oneshot_kernel<Op, 2>;
    else if (W <= 4) fn = kTwoShot ? (const void *)twoshot_kernel<Op, 4> : (const void *)oneshot_kernel<Op, 4>;
    else if (W <= 8) fn = kTwoShot ? (const void *)twoshot_kernel<Op, 8> : (const void *)oneshot_kernel<Op, 8>;
    else fn = kTwoShot ? (const void *)twoshot_kernel<Op, 16> : (const void *)oneshot_kernel<Op, 16>;
    return KernelChoice{fn, kReduceThreads, 0};
}

template <bool kTwoShot>
static KernelChoice pick_dtype(rr_dtype dtype, int W)
{
    switch (dtype) {
    case RR_BF16: return pick<OpBF16, kTwoShot>(W);
    case RR_FP16: return pick<OpFP16, kTwoShot>(W);
    case RR_FP32: return pick<OpFP32, kTwoShot>(W);
    default: return pick<OpI32, kTwoShot>(W);
    }
}

KernelChoice oneshot_kernel_for(rr_dtype dtype, int W) { return pick_dtype<false>(dtype, W); }
KernelChoice twoshot_kernel_for(rr_dtype dtype, int W) { return pick_dtype<true>(dtype, W); }

}  // namespace rr
